// Tensor-memory (tcgen05) variant of the down kernel, d = 2560, K = 320,
// T <= 8 tokens in one pass (the mma.sync kernels take T = 5..8 in two
// 4-token groups).
//
// The contraction is 20 tcgen05.mma issued by a single thread: A = a 64-row
// weight tile (M = 64), B = the activations as 2T columns (each token's FP32
// value split into hi = bf16(x) and lo = bf16(x - hi), the two-term split of
// hc_kernels_tc.cuh), K = 320, an FP32 accumulator in tensor memory.  The
// weight tile arrives by TMA
// (2-D tensor maps, boxes of 64 columns, 128-byte swizzle), which writes the
// K-major 128-byte-swizzle layout the MMA reads; the activations are written
// by the threads that form them into the K-major layout without swizzle
// (core matrices of 8 rows x 16 bytes, 128 bytes between core matrices
// adjacent along K, K/8 * 128 bytes between 8-row groups).  With
// M = 64 the accumulator row 16 w + l lives in tensor-memory lane 32 w + l
// (l < 16), so warp w reads rows 16 w .. 16 w + 15 from its own lane
// quadrant.
//
// Down kernel: grid (32 column chunks, 5 row groups), clusters of the 8
// chunks of one stream, 128 threads.  A CTA owns rows 64 g .. 64 g + 63 of
// W_down x 320 columns.  It commits the pending write for its columns,
// stages x = R' * w_norm (split), sends its sums of squares to every rank of
// the cluster, runs the MMA, and sends each row's partial sum to the rank
// that finishes that row (rank q: rows 8 q .. 8 q + 7), which adds the 8
// chunks in a fixed order, applies rs and writes part[s][t][k].
//
// It writes the partial-sum scratch exactly as the other down kernels do,
// so the up kernel of the mma.sync family (hc_kernels_tc.cuh) completes the
// read.  Launch protocol, independent mode and error reporting are those of
// the other kernel families (hc_kernels.cuh).
#pragma once

#include <cuda.h>  // CUtensorMap

#include "hc_kernels_tc.cuh"

namespace hc {

// Kernel parameters: the tensor map of W_down (dims {N, K}, boxes of 64
// columns x 64 rows, BF16, 128-byte swizzle) with the arguments of the other
// kernel families.
struct DownUArgs {
  CUtensorMap w;
  DownArgs a;
};

template <int D, int KD>
struct UGeo {
  static constexpr int N = kStreams * D;
  static constexpr int M = 64;                   // MMA rows per CTA (both kernels)
  static constexpr int KC = D / 8;               // down: columns per CTA
  static constexpr int CPS = D / KC;             // column chunks per stream = cluster size
  static constexpr int CHUNKS = N / KC;
  static constexpr int ROW_GROUPS = KD / M;
  static constexpr int RPR = M / CPS;            // rows of the tile each rank finishes
  static constexpr int TMAX = 8;                 // tokens per launch
  static constexpr int NMAX = 2 * TMAX;          // MMA columns
  static constexpr int THREADS = 128;
  static constexpr int TMEM_COLS = 32;           // the accumulator: NMAX columns
  static constexpr int DN_SBO = (KC / 8) * 128;  // between 8-row groups, KC-wide operands
  static constexpr int SLICE = M * 128;          // one 64-column box of the weight tile (8 KB)
  static constexpr int ALIGN = 1024;             // the swizzled tile starts on a 1024-byte boundary
  // down kernel shared memory (bytes, from the 1024-aligned base; BYTES
  // includes the slack for aligning the dynamic base)
  static constexpr int DN_BAR = 0;               // mbarriers: weight tile landed, MMA chain done
  static constexpr int DN_TSLOT = 16;            // tensor-memory address
  static constexpr int DN_A = ALIGN;             // [KC/64 slices][M][64] W_down tile, 128-byte swizzle
  static constexpr int DN_B = DN_A + M * KC * 2;             // [NMAX][KC] x tile
  static constexpr int DN_SSW = DN_B + NMAX * KC * 2;        // [4 warps][TMAX]
  static constexpr int DN_RSS = DN_SSW + 4 * TMAX * 4;       // [CPS][TMAX] sums of squares received
  static constexpr int DN_RP = DN_RSS + CPS * TMAX * 4;      // [CPS][TMAX][RPR] partials received
  static constexpr int DN_RS = DN_RP + CPS * TMAX * RPR * 4; // [TMAX]
  static constexpr int DN_BYTES = DN_RS + TMAX * 4 + ALIGN;

  static_assert(D == 2560 && KD == 320, "tensor-memory kernels: d = 2560, K = 320");
  static_assert(CPS == 8 && RPR == 8, "clusters of 8 chunks, 8 rows per rank");
  static_assert(KC % 16 == 0 && KD % 16 == 0, "K-steps of 16");
  static_assert(KC / 4 <= THREADS, "one float4 of a chunk per thread and token");
  static_assert(M == 4 * 16, "warp w reads tile rows 16 w .. 16 w + 15");
  static_assert(DN_B % 16 == 0, "operands start on 16-byte boundaries");
  static_assert(KC % 64 == 0 && M * KC * 2 == (KC / 64) * SLICE, "whole 64-column boxes");
  static_assert(SLICE % ALIGN == 0, "every box starts on a swizzle atom");
  static_assert(DN_BYTES <= 56 * 1024, "four CTAs per SM");
  static_assert(NMAX <= 16 && TMEM_COLS >= NMAX, "the accumulator is read with one 16-column load");
};

// The dynamic shared memory rounded up to the 1024-byte boundary the
// swizzled weight tiles need (the kernels reserve the slack).
__device__ __forceinline__ unsigned char* aligned_smem(unsigned char* raw) {
  const uint32_t s = ptx::smem_u32(raw);
  return raw + (((s + 1023u) & ~1023u) - s);
}

// Byte offset of element (r, k) of a K-major operand `KW` elements wide in
// the no-swizzle canonical layout.
template <int KW>
__device__ __forceinline__ int ucanon(int r, int k) {
  return (r >> 3) * (KW / 8) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// ------------------------------------------------------------------ kernel 1
// One tile of a swizzled tile order (hc_pack_down_sw_kernel,
// hc_pack_up_sw_kernel): BYTES contiguous bytes, already in the 128-byte
// swizzle layout the TMA boxes would write, copied in four pieces.
template <int BYTES>
__device__ __forceinline__ void copy_sw_tile(unsigned char* dst, const void* tiles, size_t tile, uint64_t* bar,
                                             uint64_t policy) {
  static_assert(BYTES % 64 == 0, "four 16-byte-aligned pieces");
  const unsigned char* src = static_cast<const unsigned char*>(tiles) + tile * BYTES;
#pragma unroll
  for (int q = 0; q < 4; ++q) ptx::bulk_g2s(dst + q * (BYTES / 4), src + q * (BYTES / 4), BYTES / 4, bar, policy);
}

template <int D, int KD>
__global__ void __launch_bounds__(UGeo<D, KD>::THREADS, 4) hc_down_u_kernel(const __grid_constant__ DownUArgs args) {
  using U = UGeo<D, KD>;
  const DownArgs& a = args.a;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = aligned_smem(smem_raw);
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + U::DN_BAR);
  uint64_t* bar_mma = bar_w + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + U::DN_TSLOT);
  unsigned char* sa = smem + U::DN_A;
  unsigned char* sb = smem + U::DN_B;
  float* ssw = reinterpret_cast<float*>(smem + U::DN_SSW);
  float* rss = reinterpret_cast<float*>(smem + U::DN_RSS);
  float* rpr = reinterpret_cast<float*>(smem + U::DN_RP);
  float* rs_s = reinterpret_cast<float*>(smem + U::DN_RS);

  const uint64_t t_entry = ptx::globaltimer_ns();
  const int chunk = blockIdx.x;
  const int stream = chunk / U::CPS;
  const int rg = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = chunk * U::KC;
  const int row0 = rg * U::M;
  const int T = a.T;
  const int nb = T <= 4 ? 8 : 16;  // MMA columns (tokens past T are zero)

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  ptx::cluster_arrive_relaxed();

  // The W_down tile (weights, independent of earlier kernels): one TMA box of
  // 64 columns x 64 rows per slice.
  if (tid == 0) {
    ptx::mbar_init(bar_w, 1);
    ptx::mbar_init(bar_mma, 1);
    ptx::fence_barrier_init();
    ptx::mbar_arrive_expect_tx(bar_w, U::M * U::KC * 2);
    const uint64_t once = ptx::policy_evict_first();
    if (a.W_tiles_sw == nullptr) {
#pragma unroll
      for (int j = 0; j < U::KC / 64; ++j) ptx::tma_load_2d(sa + j * U::SLICE, &args.w, col0 + 64 * j, row0, bar_w, once);
    } else {
      copy_sw_tile<U::M * U::KC * 2>(sa, a.W_tiles_sw, (size_t)rg * U::CHUNKS + chunk, bar_w, once);
    }
  }
  const int c4 = tid;
  const bool has4 = c4 < U::KC / 4;
  const float4 wn = has4 ? __ldg(reinterpret_cast<const float4*>(a.w_norm + col0) + c4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
  if (warp == 1) {
    ptx::tmem_alloc(tslot, U::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  // Independent reads on the batch lanes let the up kernel launch only at
  // the end (see hc_down_kernel); all T of this kernel are one pass.
  const bool late_launch = a.late_launch && a.independent;
  if (!late_launch) ptx::launch_dependents();
  ptx::tc_fence_before();
  __syncthreads();  // tensor-memory address and mbarrier visible to all
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (!a.independent) ptx::wait_prerequisites();
  ptx::cluster_wait();  // every CTA of the cluster runs before anyone writes a peer

  // x = R' * w_norm, split into two MMA columns per token, and the sums of
  // squares of R'.
  float4 rv[U::TMAX], pv[U::TMAX];
#pragma unroll
  for (int t = 0; t < U::TMAX; ++t) {
    rv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    pv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < T && has4) {
      const size_t base = (size_t)t * U::N + col0;
      rv[t] = __ldcg(reinterpret_cast<const float4*>(a.R + base) + c4);
      if (a.P) pv[t] = __ldcg(reinterpret_cast<const float4*>(a.P + base) + c4);
    }
  }
  float ssl[U::TMAX];
#pragma unroll
  for (int t = 0; t < U::TMAX; ++t) {
    ssl[t] = 0.f;
    if (2 * t < nb && has4) {
      float4 r = rv[t];
      r.x = __fadd_rn(r.x, pv[t].x);
      r.y = __fadd_rn(r.y, pv[t].y);
      r.z = __fadd_rn(r.z, pv[t].z);
      r.w = __fadd_rn(r.w, pv[t].w);
      const float4 x = make_float4(__fmul_rn(r.x, wn.x), __fmul_rn(r.y, wn.y), __fmul_rn(r.z, wn.z),
                                   __fmul_rn(r.w, wn.w));
      uint2 hi, lo;
      split4(x, hi, lo);
      *reinterpret_cast<uint2*>(sb + ucanon<U::KC>(2 * t, 4 * c4)) = hi;
      *reinterpret_cast<uint2*>(sb + ucanon<U::KC>(2 * t + 1, 4 * c4)) = lo;
      ssl[t] = __fmaf_rn(r.x, r.x, ssl[t]);
      ssl[t] = __fmaf_rn(r.y, r.y, ssl[t]);
      ssl[t] = __fmaf_rn(r.z, r.z, ssl[t]);
      ssl[t] = __fmaf_rn(r.w, r.w, ssl[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < U::TMAX; ++t) {
    float v = ssl[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) ssw[warp * U::TMAX + t] = v;
  }
  const bool ok = wait_bar_from(bar_w, 0, a.err, kErrDownWeights, t_entry, first_wait_limit(a.wait_ns));
  ptx::fence_proxy_async_smem();  // this thread's x stores, visible to the tensor cores
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  // This chunk's sums of squares to every rank of the cluster.
  if (tid < T) {
    const float v = ((ssw[tid] + ssw[U::TMAX + tid]) + ssw[2 * U::TMAX + tid]) + ssw[3 * U::TMAX + tid];
#pragma unroll
    for (int q = 0; q < U::CPS; ++q) cluster.map_shared_rank(rss, q)[rank * U::TMAX + tid] = v;
  }
  if (tid == 0 && ok) {
    const uint32_t idesc = ptx::umma_idesc_bf16(U::M, nb);
    const uint32_t a0 = ptx::smem_u32(sa), b0 = ptx::smem_u32(sb);
    for (int ks = 0; ks < U::KC / 16; ++ks) {
      ptx::umma_bf16(tmem, ptx::umma_desc_sw128(a0 + (ks >> 2) * U::SLICE + (ks & 3) * 32),
                     ptx::umma_desc(b0 + ks * 256, 128, U::DN_SBO), idesc, ks > 0 ? 1u : 0u);
    }
    ptx::umma_commit(bar_mma);
  }
  // A CTA whose weight tile did not land skips the MMA (its outputs are
  // void, the error word says so) and waits for the copies before it exits.
  if (ok) {
    wait_bar(bar_mma, 0, a.err, kErrDownWeights);
  } else {
    drain(bar_w, 0);
  }
  ptx::tc_fence_after();
  uint32_t d[16];
  ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16), d);
  ptx::tmem_wait_ld();
  // Lanes 0..15 of warp w hold tile rows 16 w + lane: each row's partial per
  // token (hi column + lo column) goes to the rank that finishes the row.
  if (lane < 16) {
    const int row = 16 * warp + lane;
    float* dst = cluster.map_shared_rank(rpr, row / U::RPR);
#pragma unroll
    for (int t = 0; t < U::TMAX; ++t) {
      if (t < T) {
        dst[(rank * U::TMAX + t) * U::RPR + (row % U::RPR)] =
            __fadd_rn(__uint_as_float(d[2 * t]), __uint_as_float(d[2 * t + 1]));
      }
    }
  }
  ptx::tc_fence_before();
  if (late_launch) ptx::launch_dependents();
  ptx::cluster_arrive_release();
  ptx::cluster_wait();  // every chunk's sums of squares and partials are here
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, U::TMEM_COLS);

  if (tid < T) {
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < U::CPS; ++q) ss += rss[q * U::TMAX + tid];
    const float rs = rsqrtf(ss * (1.0f / (float)D) + a.eps);
    rs_s[tid] = rs;
    if (rg == 0 && rank == 0 && a.rs_out != nullptr) a.rs_out[tid * kStreams + stream] = rs;
  }
  __syncthreads();
  float* part = a.part + (size_t)stream * a.T_max * KD;
  for (int idx = tid; idx < T * U::RPR; idx += U::THREADS) {
    const int t = idx / U::RPR, r8 = idx - t * U::RPR;
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < U::CPS; ++q) p += rpr[(q * U::TMAX + t) * U::RPR + r8];
    __stcg(part + (size_t)t * KD + row0 + (int)rank * U::RPR + r8, __fmul_rn(rs_s[t], p));
  }
  if (a.independent) ptx::wait_prerequisites();  // complete only after the previous read
}

}  // namespace hc
