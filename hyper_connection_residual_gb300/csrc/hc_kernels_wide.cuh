// Tensor-memory (tcgen05) kernels of the read for many tokens: d = 2560,
// K = 320, 9 <= T <= 64.  The read is then a skinny dense contraction,
// [T x N] x [N x K] and [T x K] x [K x N], and both projections run on the
// 5th-generation tensor cores with every weight byte read from HBM once for
// all T tokens ("read the weights once for all tokens": Strata pull request
// #2070, first paragraph; #2812, section "What changed", for the kernels'
// roles).
//
// Both kernels hold a 64-row weight tile (M = 64) in shared memory, brought
// by 2-D TMA boxes of 64 columns in the 128-byte swizzle layout, and run the
// tokens in passes of 16 (the up kernel; the down kernel of T > 16 runs
// all tokens in one pass, below): the FP32 activations of a pass are split
// into two BF16 terms (hi = bf16(x), lo = bf16(x - hi), the split of
// hc_kernels_tc.cuh) as 2 x 16 rows of the B operand, also in the 128-byte
// swizzle layout (threads running along the columns of one token then store
// with at most two-way bank conflicts), and 20 tcgen05.mma (K = 16 each) of
// one thread accumulate the pass into 32 columns of a 128-column FP32
// accumulator in tensor memory.  One B buffer serves the passes in turn; the
// next pass's loads go out as soon as a pass is staged, so they are in
// flight while its MMAs run.  Shared memory is sized by T, and three CTAs
// fit an SM (the up kernel: up to T = 48).  For T <= 16 the up kernel has a
// single-pass instantiation (MULTI = false: fewer registers, no pass loop)
// and the down kernel a single-pass kernel of its own, measured 4-10 %
// faster there than the general forms.
//
// Down kernels: grid (32 column chunks, 5 row groups), clusters of the 8
// chunks of one stream, 256 threads.  A CTA owns rows 64 g .. 64 g + 63 of
// W_down x 320 columns and stages x = R' * w_norm (the sums of squares by
// shuffles); after its MMAs each accumulator row's partial sum per token
// (hi + lo column) goes through distributed shared memory to the rank that
// finishes it (rank q: rows 8 q .. 8 q + 7), which adds the 8 chunks in a
// fixed order, applies rs and writes part[s][t][k] exactly as the other down
// kernels do.  hc_down_w1_kernel (T <= 16) stages every token at once, warp w
// taking tokens w and w + 8.  hc_down_w_kernel (T > 16) stages B one K slice
// at a time, for every token, into a ring of slices, so a single chain of 20
// MMAs with N = 2 T covers all tokens: a tcgen05.mma of M = 64 costs about
// the same ~56 cycles at N = 16, 32 or 64 (measured), so 16-token passes
// would pay for the chain once per pass.
//
// hc_up_w_kernel: 160 CTAs of 16 columns x 4 streams = 64 rows of W_up (the
// stream mean of a column stays inside the CTA), clusters of UCL.  lo is the
// sum of the four streams' partials: rank r of a cluster forms it for its
// TP / UCL tokens of the pass over all K, writes their B rows into its own
// buffer and pushes those rows (whole 128-byte rows of each K slice, so the
// swizzle is kept) into the same place of every peer with shared-to-shared
// bulk copies on the TMA engine, counted on the peer's per-pass mbarrier.
// The cluster thereby loads the partials once instead of every CTA loading
// all of them, and no thread stores into a peer.  The epilogue (pending
// write, gate, stream mean) reads u straight from the accumulator: row
// 16 s + l of the tile (stream s, column c0 + l) is tensor-memory lane
// 32 s + l.
//
// Launch protocol, independent mode and error reporting are those of the
// other kernel families (hc_kernels.cuh).
#pragma once

#include "hc_kernels_umma.cuh"

namespace hc {

// Up-kernel parameters: the tensor map of W_up (dims {K, N}, boxes of 64
// columns x 16 rows, BF16, 128-byte swizzle) with the up kernels' arguments.
struct UpWArgs {
  CUtensorMap w;
  UpArgs a;
};

template <int D, int KD>
struct WGeo {
  static constexpr int N = kStreams * D;
  static constexpr int M = 64;                    // MMA rows per CTA (both kernels)
  static constexpr int THREADS = 256;
  static constexpr int WARPS = THREADS / 32;
  static constexpr int TP = 16;                   // tokens per pass: 2 TP MMA columns
  static constexpr int TW = 64;                   // most tokens of a launch
  static constexpr int NPASS = TW / TP;
  static constexpr int BROWS = 2 * TP;            // B rows of a pass (hi, lo per token)
  static constexpr int SLICE_A = M * 128;         // a 64-wide K slice of A, 8 KB
  static constexpr int SLICE_B = BROWS * 128;     // ... of B, 4 KB
  static constexpr int PCOLS = 2 * TP;            // accumulator columns of a pass
  static constexpr int TMEM_COLS = NPASS * PCOLS; // 128
  // ---- down kernel: 64 rows x KC columns per CTA
  static constexpr int KC = D / 8;
  static constexpr int NSL_D = KC / 64;           // K slices
  static constexpr int BBUF_D = NSL_D * SLICE_B;  // one B buffer
  static constexpr int CPS = 8;                   // chunks per stream = cluster size
  static constexpr int CHUNKS = N / KC;
  static constexpr int ROW_GROUPS = KD / M;
  static constexpr int RPR = M / CPS;             // rows each rank finishes
  static constexpr int KC4 = KC / 4;              // float4 of a token's chunk
  static constexpr int C4L = (KC4 + 31) / 32;     // ... per lane
  static constexpr int DN_BAR = 0;                // bar_w, bar_slot[2]
  static constexpr int DN_TSLOT = 64;
  static constexpr int DN_A = 1024;
  static constexpr int DN_B = DN_A + NSL_D * SLICE_A;
  // ---- up kernel: UC columns x 4 streams = 64 rows of W_up per CTA
  static constexpr int UC = M / kStreams;
  static constexpr int UP_CTAS = D / UC;
  static constexpr int UCL = 4;                   // cluster size
  static constexpr int NSL_U = KD / 64;
  static constexpr int KD4 = KD / 4;
  static constexpr int UP_BAR = 0;                // bar_w, bar_mma[NPASS], bar_b[NPASS]
  static constexpr int UP_TSLOT = 96;
  static constexpr int UP_A = 1024;
  static constexpr int UP_B = UP_A + NSL_U * SLICE_A;

  __host__ __device__ static constexpr int npass(int T) { return (T + TP - 1) / TP; }
  __host__ __device__ static constexpr int r16(int b) { return (b + 15) / 16 * 16; }
  // down kernel: B is a ring of K slices, each slice the 64 columns of one
  // TMA box for every token (dn_brows rows: hi, lo per token, padded to a
  // multiple of 8), so one chain of 20 MMAs with N = dn_brows covers all T
  // tokens.  After the ring: this chunk's sums of squares [T], those received
  // [CPS][T], rs [T], and the partials received from the cluster
  // ([CPS][T][RPR]) in their own region, or over the A tile once every CTA of
  // the cluster is past its MMAs (one more cluster barrier).  Two ring slots
  // and the own region are used while three CTAs still fit an SM.
  static constexpr int SMEM3 = 76800;  // at most this per CTA for three CTAs per SM
  __host__ __device__ static constexpr int dn_brows(int T) { return (2 * T + 7) / 8 * 8; }
  __host__ __device__ static constexpr int dn_slot(int T) { return dn_brows(T) * 128; }
  __host__ __device__ static constexpr int dn_layout(int T, int nbuf, bool own) {
    return DN_B + nbuf * dn_slot(T) + r16(4 * T) + r16(4 * CPS * T) + r16(4 * T) + (own ? 4 * CPS * T * RPR : 0) + 1024;
  }
  __host__ __device__ static constexpr int dn_nbuf(int T) {
    return dn_layout(T, 2, false) <= SMEM3 ? 2 : 1;
  }
  __host__ __device__ static constexpr bool dn_rp_own(int T) { return dn_layout(T, dn_nbuf(T), true) <= SMEM3; }
  __host__ __device__ static constexpr int dn_ssv(int T) { return DN_B + dn_nbuf(T) * dn_slot(T); }  // [T]
  __host__ __device__ static constexpr int dn_rss(int T) { return dn_ssv(T) + r16(4 * T); }          // [CPS][T]
  __host__ __device__ static constexpr int dn_rs(int T) { return dn_rss(T) + r16(4 * CPS * T); }     // [T]
  __host__ __device__ static constexpr int dn_rp(int T) { return dn_rp_own(T) ? dn_rs(T) + r16(4 * T) : DN_A; }
  __host__ __device__ static constexpr int dn_bytes(int T) { return dn_layout(T, dn_nbuf(T), dn_rp_own(T)); }
  // single-pass down kernel (T <= TP): one B buffer of TP tokens over all
  // K slices, then [T], [CPS][T], [T] and its own [CPS][T][RPR] region
  __host__ __device__ static constexpr int d1_ssv(int T) { return DN_B + BBUF_D; }
  __host__ __device__ static constexpr int d1_rss(int T) { return d1_ssv(T) + r16(4 * T); }
  __host__ __device__ static constexpr int d1_rs(int T) { return d1_rss(T) + r16(4 * CPS * T); }
  __host__ __device__ static constexpr int d1_rp(int T) { return d1_rs(T) + r16(4 * T); }
  __host__ __device__ static constexpr int d1_bytes(int T) { return d1_rp(T) + 4 * CPS * T * RPR + 1024; }
  __host__ __device__ static constexpr int imax(int x, int y) { return x > y ? x : y; }
  __host__ __device__ static constexpr int dn_bytes_max(int T) { return T == 0 ? 0 : imax(dn_bytes(T), dn_bytes_max(T - 1)); }
  static constexpr int DN_BYTES_MAX = dn_bytes_max(TW);

  static_assert(D == 2560 && KD == 320, "wide tensor-memory kernels: d = 2560, K = 320");
  static_assert(KC % 64 == 0 && KD % 64 == 0, "whole 64-wide K slices");
  static_assert(CHUNKS == kStreams * CPS && RPR == 8, "clusters of one stream's 8 chunks");
  static_assert(TP == 2 * WARPS, "warp w stages tokens w and w + 8 of a pass");
  static_assert(UP_CTAS % UCL == 0, "up clusters");
  static_assert(SLICE_A % 1024 == 0 && SLICE_B % 1024 == 0 && DN_B % 1024 == 0 && UP_B % 1024 == 0,
                "swizzled operands start on 1024-byte atoms");
  static_assert(4 * CPS * TW * RPR <= NSL_D * SLICE_A, "the received partials fit over the A tile");
  static_assert(DN_BYTES_MAX <= SMEM3 && d1_bytes(TP) <= SMEM3, "three down CTAs per SM");
  static_assert(dn_brows(TW) <= TMEM_COLS && dn_brows(TW) <= 256, "one MMA chain covers every token");
  static_assert(3 * TMEM_COLS <= 512, "three CTAs' accumulators fit the tensor memory");
};

// The up kernel's pass geometry: passes of TP tokens (2 TP B rows, 2 TP
// accumulator columns), each rank of a cluster combining TP / UCL tokens of
// a pass.  TP = 16 keeps three CTAs per SM up to T = 48; above, where the R'
// of 64 tokens already limits the kernel to two CTAs per SM, TP = 32 halves
// the passes (and their MMA chains, buffer-reuse barriers and exchanges).
template <int D, int KD, int TP_>
struct UpPass {
  using W = WGeo<D, KD>;
  static constexpr int TP = TP_;
  static constexpr int BROWS = 2 * TP;                 // B rows of a pass
  static constexpr int SLICE_B = BROWS * 128;          // a 64-wide K slice of B
  static constexpr int PCOLS = 2 * TP;                 // accumulator columns of a pass
  static constexpr int NPASS = W::TW / TP;
  static constexpr int TPR = TP / W::UCL;              // tokens of a pass each rank combines
  static constexpr int RROWS = 2 * TPR;                // ... B rows
  static constexpr int BBUF_U = W::NSL_U * SLICE_B;    // the B buffer
  static constexpr int UP_RECV = (W::UCL - 1) * W::NSL_U * RROWS * 128;  // bytes from the peers per pass
  __host__ __device__ static constexpr int npass(int T) { return (T + TP - 1) / TP; }
  __host__ __device__ static constexpr int up_sig(int T) { return W::UP_B + BBUF_U; }     // [M]
  __host__ __device__ static constexpr int up_rp(int T) { return up_sig(T) + 4 * W::M; }  // [T][M]
  __host__ __device__ static constexpr int up_bytes(int T) { return up_rp(T) + 4 * W::M * T + 1024; }
  static_assert(TP % W::UCL == 0 && (RROWS * 128) % 16 == 0, "clusters split a pass by tokens");
  static_assert(NPASS * PCOLS == W::TMEM_COLS, "the passes' accumulators fill the tensor memory");
  static_assert(8 * (1 + 2 * NPASS) <= W::UP_TSLOT, "the barriers fit before the tensor-memory slot");
  static_assert(SLICE_B % 1024 == 0 && W::UP_B % 1024 == 0, "swizzled operands start on 1024-byte atoms");
  static_assert(up_bytes(W::TW) <= 113 * 1024, "two CTAs per SM at any T");
};

static_assert(UpPass<2560, 320, 16>::up_bytes(48) <= WGeo<2560, 320>::SMEM3,
              "three up CTAs per SM with 16-token passes up to T = 48");

// Byte offset of element (n, k) of a K-major BF16 operand of ROWS rows in the
// 128-byte swizzle layout: 64-wide K slices of ROWS * 128 bytes, rows of 128
// bytes, the 16-byte chunk index XOR the row within its 8-row atom (the
// layout a TMA load with 128-byte swizzle writes and umma_desc_sw128 reads).
template <int ROWS>
__device__ __forceinline__ int sw128_off(int n, int k) {
  return (k >> 6) * (ROWS * 128) + n * 128 + ((((k >> 3) & 7) ^ (n & 7)) << 4) + (k & 7) * 2;
}

__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}

// 20 (K / 16) MMAs of one pass, D (tensor memory) = A (M x K, swizzled
// slices of SLICE_A bytes) * B (npad rows of a SLICE_B-byte-slice operand).
template <int KK, int SLICE_A, int SLICE_B>
__device__ __forceinline__ void umma_pass(uint32_t tmem_d, uint32_t a0, uint32_t b0, int m, int npad) {
  const uint32_t idesc = ptx::umma_idesc_bf16(m, npad);
#pragma unroll
  for (int ks = 0; ks < KK / 16; ++ks) {
    ptx::umma_bf16(tmem_d, ptx::umma_desc_sw128(a0 + (ks >> 2) * SLICE_A + (ks & 3) * 32),
                   ptx::umma_desc_sw128(b0 + (ks >> 2) * SLICE_B + (ks & 3) * 32), idesc, ks > 0 ? 1u : 0u);
  }
}

// ------------------------------------------------------------------ kernel 1, T <= 16
// One pass of at most 16 tokens: every token staged at once (the loads of
// all of them in flight together), one chain of 20 MMAs.
template <int D, int KD>
__global__ void __launch_bounds__(WGeo<D, KD>::THREADS, 3) hc_down_w1_kernel(const __grid_constant__ DownUArgs args) {
  using W = WGeo<D, KD>;
  const DownArgs& a = args.a;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = aligned_smem(smem_raw);
  const int T = a.T;
  const int npass = 1;  // T <= TP
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + W::DN_BAR);
  uint64_t* bar_mma = bar_w + 1;  // [NPASS]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + W::DN_TSLOT);
  unsigned char* sa = smem + W::DN_A;
  unsigned char* sb = smem + W::DN_B;
  float* ssv = reinterpret_cast<float*>(smem + W::d1_ssv(T));
  float* rss = reinterpret_cast<float*>(smem + W::d1_rss(T));
  float* rpr = reinterpret_cast<float*>(smem + W::d1_rp(T));  // own region, or over the A tile
  float* rs_s = reinterpret_cast<float*>(smem + W::d1_rs(T));

  const uint64_t t_entry = ptx::globaltimer_ns();
  const int chunk = blockIdx.x;
  const int stream = chunk / W::CPS;
  const int rg = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = chunk * W::KC;
  const int row0 = rg * W::M;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  ptx::cluster_arrive_relaxed();

  // The W_down tile (weights, independent of earlier kernels).
  if (tid == 0) {
    ptx::mbar_init(bar_w, 1);
#pragma unroll
    for (int p = 0; p < W::NPASS; ++p) ptx::mbar_init(&bar_mma[p], 1);
    ptx::fence_barrier_init();
    ptx::mbar_arrive_expect_tx(bar_w, W::M * W::KC * 2);
    const uint64_t once = ptx::policy_evict_first();
    if (a.W_tiles_sw == nullptr) {
#pragma unroll
      for (int j = 0; j < W::NSL_D; ++j) ptx::tma_load_2d(sa + j * W::SLICE_A, &args.w, col0 + 64 * j, row0, bar_w, once);
    } else {
      copy_sw_tile<W::M * W::KC * 2>(sa, a.W_tiles_sw, (size_t)rg * W::CHUNKS + chunk, bar_w, once);
    }
  }
  // w_norm of this lane's float4 columns lane, lane + 32, ...
  float4 wn[W::C4L];
#pragma unroll
  for (int c = 0; c < W::C4L; ++c) {
    const int c4 = lane + 32 * c;
    wn[c] = c4 < W::KC4 ? __ldg(reinterpret_cast<const float4*>(a.w_norm + col0) + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (warp == 1) {
    __syncwarp();  // tcgen05.alloc is .aligned
    ptx::tmem_alloc(tslot, W::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  // Independent reads on the batch lanes let the up kernel launch only at
  // the end (see hc_down_kernel).
  const bool late_launch = a.late_launch && a.independent;
  if (!late_launch) ptx::launch_dependents();
  ptx::tc_fence_before();
  __syncthreads();  // tensor-memory address and mbarriers visible to all
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (!a.independent) ptx::wait_prerequisites();
  ptx::cluster_wait();  // every CTA of the cluster runs before anyone writes a peer

  bool ok = true;
  const uint32_t a0 = ptx::smem_u32(sa);
  // Warp w stages tokens t0 + w and t0 + w + 8 of pass p: R' = R + P,
  // x = R' * w_norm split into B rows 2 tl (hi) and 2 tl + 1 (lo), and the
  // token's sum of squares over this chunk.
  using Reg = float4[2][W::C4L];
  auto load_pass = [&](int p, Reg& rv, Reg& pv) {
    const int t0 = p * W::TP;
    const int tp = min(W::TP, T - t0);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int tl = warp + W::WARPS * m;
#pragma unroll
      for (int c = 0; c < W::C4L; ++c) {
        const int c4 = lane + 32 * c;
        rv[m][c] = make_float4(0.f, 0.f, 0.f, 0.f);
        pv[m][c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tl < tp && c4 < W::KC4) {
          const size_t base = (size_t)(t0 + tl) * W::N + col0;
          rv[m][c] = __ldcg(reinterpret_cast<const float4*>(a.R + base) + c4);
          if (a.P) pv[m][c] = __ldcg(reinterpret_cast<const float4*>(a.P + base) + c4);
        }
      }
    }
  };
  Reg rv, pv;
  load_pass(0, rv, pv);
  for (int p = 0; p < npass; ++p) {
    const int t0 = p * W::TP;
    const int tp = min(W::TP, T - t0);
    unsigned char* bp = sb;
    // The buffer was last read by the MMAs of pass p - 1.
    if (p >= 1) {
      if (ok) ok = wait_bar(&bar_mma[p - 1], 0, a.err, kErrDownWeights);
      ptx::tc_fence_after();
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int tl = warp + W::WARPS * m;
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < W::C4L; ++c) {
        const int c4 = lane + 32 * c;
        if (tl < tp && c4 < W::KC4) {
          float4 r = rv[m][c];
          r.x = __fadd_rn(r.x, pv[m][c].x);
          r.y = __fadd_rn(r.y, pv[m][c].y);
          r.z = __fadd_rn(r.z, pv[m][c].z);
          r.w = __fadd_rn(r.w, pv[m][c].w);
          const float4 x = make_float4(__fmul_rn(r.x, wn[c].x), __fmul_rn(r.y, wn[c].y), __fmul_rn(r.z, wn[c].z),
                                       __fmul_rn(r.w, wn[c].w));
          uint2 hi, lo;
          split4(x, hi, lo);
          *reinterpret_cast<uint2*>(bp + sw128_off<W::BROWS>(2 * tl, 4 * c4)) = hi;
          *reinterpret_cast<uint2*>(bp + sw128_off<W::BROWS>(2 * tl + 1, 4 * c4)) = lo;
          ss = __fmaf_rn(r.x, r.x, ss);
          ss = __fmaf_rn(r.y, r.y, ss);
          ss = __fmaf_rn(r.z, r.z, ss);
          ss = __fmaf_rn(r.w, r.w, ss);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0 && tl < tp) ssv[t0 + tl] = ss;
    }
    // The registers are free: the next pass's loads go out now, in flight
    // while this pass's MMAs run.
    if (p + 1 < npass) load_pass(p + 1, rv, pv);
    if (p == 0) ok = wait_bar_from(bar_w, 0, a.err, kErrDownWeights, t_entry, first_wait_limit(a.wait_ns)) && ok;
    ptx::fence_proxy_async_smem();  // this thread's B stores, visible to the tensor cores
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (tid == 0) {
      if (ok) {
        umma_pass<W::KC, W::SLICE_A, W::SLICE_B>(tmem + (uint32_t)(p * W::PCOLS), a0, ptx::smem_u32(bp), W::M,
                                                 (2 * tp + 7) & ~7);
        ptx::umma_commit(&bar_mma[p]);
      } else {
        mbar_arrive_local(&bar_mma[p]);  // nothing issued: release the waiters
      }
    }
  }
  // The last commit tracks every MMA of the CTA.
  if (ok) ok = wait_bar(&bar_mma[npass - 1], 0, a.err, kErrDownWeights);
  if (!ok) drain(bar_w, 0);
  // This chunk's sums of squares to every rank of the cluster.
  if (tid < T) {
    const float v = ssv[tid];
#pragma unroll
    for (int q = 0; q < W::CPS; ++q) cluster.map_shared_rank(rss, q)[rank * T + tid] = v;
  }
  __syncwarp();
  ptx::tc_fence_after();

  // Accumulators: warp w reads lane quadrant w % 4 (tile rows 16 (w % 4) ..
  // + 15 in its lanes 0..15) over half w / 4 of the columns in use; each
  // row's partial per token goes to the rank that finishes the row.
  {
    const int qd = warp & 3, h = warp >> 2;
    const int ncols = npass * W::PCOLS;
    const int row = 16 * qd + (lane & 15);
    float* dst = cluster.map_shared_rank(rpr, row / W::RPR);
    for (int c = h * (ncols / 2); c < (h + 1) * (ncols / 2); c += 16) {
      uint32_t d[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)c, d);
      ptx::tmem_wait_ld();
      if (lane < 16) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int col = c + 2 * e;
          const int t = (col / W::PCOLS) * W::TP + (col % W::PCOLS) / 2;
          if (t < T) {
            dst[((int)rank * T + t) * W::RPR + row % W::RPR] =
                __fadd_rn(__uint_as_float(d[2 * e]), __uint_as_float(d[2 * e + 1]));
          }
        }
      }
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  if (late_launch) ptx::launch_dependents();
  ptx::cluster_arrive_release();
  ptx::cluster_wait();  // every chunk's sums of squares and partials are here
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, W::TMEM_COLS);

  for (int t = tid; t < T; t += W::THREADS) {
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < W::CPS; ++q) ss += rss[q * T + t];
    const float rs = rsqrtf(ss * (1.0f / (float)D) + a.eps);
    rs_s[t] = rs;
    if (rg == 0 && rank == 0 && a.rs_out != nullptr) a.rs_out[t * kStreams + stream] = rs;
  }
  __syncthreads();
  float* part = a.part + (size_t)stream * a.T_max * KD;
  for (int idx = tid; idx < T * W::RPR; idx += W::THREADS) {
    const int t = idx / W::RPR, r8 = idx - t * W::RPR;
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < W::CPS; ++q) p += rpr[(q * T + t) * W::RPR + r8];
    __stcg(part + (size_t)t * KD + row0 + (int)rank * W::RPR + r8, __fmul_rn(rs_s[t], p));
  }
  if (a.independent) ptx::wait_prerequisites();  // complete only after the previous read
}

// ------------------------------------------------------------------ kernel 1, T > 16
// TT: tokens per staging thread (T <= 16 TT); HASP: the read has a pending
// write (without it the P loads and their registers go away, and more K
// slices of R loads fit in flight).
template <int D, int KD, int TT, bool HASP>
__global__ void __launch_bounds__(WGeo<D, KD>::THREADS, 3) hc_down_w_kernel(const __grid_constant__ DownUArgs args) {
  using W = WGeo<D, KD>;
  const DownArgs& a = args.a;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = aligned_smem(smem_raw);
  const int T = a.T;
  const int nbuf = W::dn_nbuf(T);        // ring slots (1 or 2)
  const int brows = W::dn_brows(T);      // B rows = MMA N (hi, lo per token, padded to 8)
  const int slot_bytes = W::dn_slot(T);
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + W::DN_BAR);
  uint64_t* bar_slot = bar_w + 1;  // [2] the MMAs of the slice in a ring slot are done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + W::DN_TSLOT);
  unsigned char* sa = smem + W::DN_A;
  unsigned char* sb = smem + W::DN_B;
  float* ssv = reinterpret_cast<float*>(smem + W::dn_ssv(T));
  float* rss = reinterpret_cast<float*>(smem + W::dn_rss(T));
  float* rpr = reinterpret_cast<float*>(smem + W::dn_rp(T));  // own region, or over the A tile
  float* rs_s = reinterpret_cast<float*>(smem + W::dn_rs(T));

  const uint64_t t_entry = ptx::globaltimer_ns();
  const int chunk = blockIdx.x;
  const int stream = chunk / W::CPS;
  const int rg = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = chunk * W::KC;
  const int row0 = rg * W::M;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  ptx::cluster_arrive_relaxed();

  // The W_down tile (weights, independent of earlier kernels).
  if (tid == 0) {
    ptx::mbar_init(bar_w, 1);
    ptx::mbar_init(&bar_slot[0], 1);
    ptx::mbar_init(&bar_slot[1], 1);
    ptx::fence_barrier_init();
    ptx::mbar_arrive_expect_tx(bar_w, W::M * W::KC * 2);
    const uint64_t once = ptx::policy_evict_first();
    if (a.W_tiles_sw == nullptr) {
#pragma unroll
      for (int j = 0; j < W::NSL_D; ++j) ptx::tma_load_2d(sa + j * W::SLICE_A, &args.w, col0 + 64 * j, row0, bar_w, once);
    } else {
      copy_sw_tile<W::M * W::KC * 2>(sa, a.W_tiles_sw, (size_t)rg * W::CHUNKS + chunk, bar_w, once);
    }
  }
  if (warp == 1) {
    __syncwarp();  // tcgen05.alloc is .aligned
    ptx::tmem_alloc(tslot, W::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  // Independent reads on the batch lanes let the up kernel launch only at
  // the end (see hc_down_kernel).
  const bool late_launch = a.late_launch && a.independent;
  if (!late_launch) ptx::launch_dependents();
  ptx::tc_fence_before();
  __syncthreads();  // tensor-memory address and mbarriers visible to all
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (!a.independent) ptx::wait_prerequisites();
  ptx::cluster_wait();  // every CTA of the cluster runs before anyone writes a peer

  // Thread (tg = tid / 16, c4 = tid % 16) stages tokens tg + 16 m (m < TT)
  // at columns 4 c4 .. 4 c4 + 3 of every K slice: R' = R + P, x = R' * w_norm
  // split into B rows 2 t (hi) and 2 t + 1 (lo), and its share of each
  // token's sum of squares.  The loads of NPF slices are in flight at once,
  // as many as the 85 registers of three CTAs per SM hold without spilling
  // (at TT = 4 two without P, one with it; three at TT = 4 or five at TT = 2
  // fit too but measured slower); a slice's registers are refilled with the
  // loads of slice j + NPF as soon as it is staged.
  constexpr int NPF = TT == 1 ? W::NSL_D : TT == 2 ? (HASP ? 2 : 3) : (HASP ? 1 : 2);
  const int tg = tid >> 4, c4 = tid & 15;
  float4 rv[NPF][TT], pv[NPF][TT], wn[NPF];
  float ssr[TT];
#pragma unroll
  for (int m = 0; m < TT; ++m) ssr[m] = 0.f;
  auto load_slice = [&](int j, float4 (&r)[TT], float4 (&q)[TT], float4& w) {
    const int col = col0 + 64 * j + 4 * c4;
    w = __ldg(reinterpret_cast<const float4*>(a.w_norm + col));
#pragma unroll
    for (int m = 0; m < TT; ++m) {
      const int t = tg + 16 * m;
      r[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      q[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < T) {
        r[m] = __ldcg(reinterpret_cast<const float4*>(a.R + (size_t)t * W::N + col));
        if (HASP) q[m] = __ldcg(reinterpret_cast<const float4*>(a.P + (size_t)t * W::N + col));
      }
    }
  };
  bool ok = true;
  const uint32_t a0 = ptx::smem_u32(sa);
  const uint32_t idesc = ptx::umma_idesc_bf16(W::M, brows);
#pragma unroll
  for (int j = 0; j < NPF; ++j) load_slice(j, rv[j], pv[j], wn[j]);
#pragma unroll
  for (int j = 0; j < W::NSL_D; ++j) {
    const int slot = j % nbuf;
    const int f = j % NPF;  // register set of the slice (compile-time: the loop is unrolled)
    unsigned char* bp = sb + slot * slot_bytes;
    // The slot was last read by the MMAs of slice j - nbuf.
    if (j >= nbuf) {
      if (ok) ok = wait_bar(&bar_slot[slot], (uint32_t)((j / nbuf - 1) & 1), a.err, kErrDownWeights);
      ptx::tc_fence_after();
    }
#pragma unroll
    for (int m = 0; m < TT; ++m) {
      const int t = tg + 16 * m;
      if (t < T) {
        float4 r = rv[f][m];
        if (HASP) {
          r.x = __fadd_rn(r.x, pv[f][m].x);
          r.y = __fadd_rn(r.y, pv[f][m].y);
          r.z = __fadd_rn(r.z, pv[f][m].z);
          r.w = __fadd_rn(r.w, pv[f][m].w);
        }
        const float4 w = wn[f];
        const float4 x = make_float4(__fmul_rn(r.x, w.x), __fmul_rn(r.y, w.y), __fmul_rn(r.z, w.z), __fmul_rn(r.w, w.w));
        uint2 hi, lo;
        split4(x, hi, lo);
        *reinterpret_cast<uint2*>(bp + sw128_off<1>(2 * t, 4 * c4)) = hi;  // within one 64-column slice
        *reinterpret_cast<uint2*>(bp + sw128_off<1>(2 * t + 1, 4 * c4)) = lo;
        ssr[m] = __fmaf_rn(r.x, r.x, ssr[m]);
        ssr[m] = __fmaf_rn(r.y, r.y, ssr[m]);
        ssr[m] = __fmaf_rn(r.z, r.z, ssr[m]);
        ssr[m] = __fmaf_rn(r.w, r.w, ssr[m]);
      }
    }
    if (j + NPF < W::NSL_D) load_slice(j + NPF, rv[f], pv[f], wn[f]);
    if (j == 0) ok = wait_bar_from(bar_w, 0, a.err, kErrDownWeights, t_entry, first_wait_limit(a.wait_ns)) && ok;
    ptx::fence_proxy_async_smem();  // this thread's B stores, visible to the tensor cores
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (tid == 0) {
      if (ok) {
        // K-steps 4 j .. 4 j + 3 of the chain, N = brows (every token).
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ptx::umma_bf16(tmem, ptx::umma_desc_sw128(a0 + j * W::SLICE_A + k * 32),
                         ptx::umma_desc_sw128(ptx::smem_u32(bp) + k * 32), idesc, (j | k) ? 1u : 0u);
        }
        ptx::umma_commit(&bar_slot[slot]);
      } else {
        mbar_arrive_local(&bar_slot[slot]);  // nothing issued: release the waiters
      }
    }
  }
  // The last slice's commit tracks every MMA of the CTA.
  {
    const int jl = W::NSL_D - 1;
    if (ok) ok = wait_bar(&bar_slot[jl % nbuf], (uint32_t)((jl / nbuf) & 1), a.err, kErrDownWeights);
  }
  if (!ok) drain(bar_w, 0);
  // Each token's sum of squares over the chunk: the 16 threads of a token,
  // in a fixed order.
#pragma unroll
  for (int m = 0; m < TT; ++m) {
    float v = ssr[m];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (c4 == 0 && tg + 16 * m < T) ssv[tg + 16 * m] = v;
  }
  __syncthreads();
  // This chunk's sums of squares to every rank of the cluster.
  if (tid < T) {
    const float v = ssv[tid];
#pragma unroll
    for (int q = 0; q < W::CPS; ++q) cluster.map_shared_rank(rss, q)[rank * T + tid] = v;
  }
  if (!W::dn_rp_own(T)) {
    // The received partials go over the A tile: every CTA of the cluster is
    // past its MMAs before anyone writes into a peer.
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
  }
  __syncwarp();
  ptx::tc_fence_after();

  // Accumulators: warp w reads lane quadrant w % 4 (tile rows 16 (w % 4) ..
  // + 15 in its lanes 0..15) over half w / 4 of the columns in use (token t
  // in columns 2 t, 2 t + 1); each row's partial per token goes to the rank
  // that finishes the row.
  {
    const int qd = warp & 3, h = warp >> 2;
    const int ncols = (2 * T + 31) / 32 * 32;
    const int row = 16 * qd + (lane & 15);
    float* dst = cluster.map_shared_rank(rpr, row / W::RPR);
    for (int c = h * (ncols / 2); c < (h + 1) * (ncols / 2); c += 16) {
      uint32_t d[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)c, d);
      ptx::tmem_wait_ld();
      if (lane < 16) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = c / 2 + e;
          if (t < T) {
            dst[((int)rank * T + t) * W::RPR + row % W::RPR] =
                __fadd_rn(__uint_as_float(d[2 * e]), __uint_as_float(d[2 * e + 1]));
          }
        }
      }
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  if (late_launch) ptx::launch_dependents();
  ptx::cluster_arrive_release();
  ptx::cluster_wait();  // every chunk's sums of squares and partials are here
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, W::TMEM_COLS);

  for (int t = tid; t < T; t += W::THREADS) {
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < W::CPS; ++q) ss += rss[q * T + t];
    const float rs = rsqrtf(ss * (1.0f / (float)D) + a.eps);
    rs_s[t] = rs;
    if (rg == 0 && rank == 0 && a.rs_out != nullptr) a.rs_out[t * kStreams + stream] = rs;
  }
  __syncthreads();
  float* part = a.part + (size_t)stream * a.T_max * KD;
  for (int idx = tid; idx < T * W::RPR; idx += W::THREADS) {
    const int t = idx / W::RPR, r8 = idx - t * W::RPR;
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < W::CPS; ++q) p += rpr[(q * T + t) * W::RPR + r8];
    __stcg(part + (size_t)t * KD + row0 + (int)rank * W::RPR + r8, __fmul_rn(rs_s[t], p));
  }
  if (a.independent) ptx::wait_prerequisites();  // complete only after the previous read
}

// ------------------------------------------------------------------ kernel 2
template <int D, int KD, bool MULTI, int TPU>
__global__ void __launch_bounds__(WGeo<D, KD>::THREADS, TPU == 16 ? 3 : 2)
    hc_up_w_kernel(const __grid_constant__ UpWArgs args) {
  using W = WGeo<D, KD>;
  using P = UpPass<D, KD, TPU>;
  const UpArgs& a = args.a;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = aligned_smem(smem_raw);
  const int T = a.T;
  const int npass = MULTI ? P::npass(T) : 1;  // MULTI = false: T <= TP
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + W::UP_BAR);
  uint64_t* bar_mma = bar_w + 1;            // [NPASS]
  uint64_t* bar_b = bar_w + 1 + P::NPASS;   // [NPASS] the peers' B rows of a pass have landed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + W::UP_TSLOT);
  unsigned char* sa = smem + W::UP_A;
  unsigned char* sb = smem + W::UP_B;
  float* sig = reinterpret_cast<float*>(smem + P::up_sig(T));
  float* rp = reinterpret_cast<float*>(smem + P::up_rp(T));

  const int c0 = blockIdx.x * W::UC;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const int cq = blockIdx.x / W::UCL;  // cluster
  ptx::cluster_arrive_relaxed();

  // The W_up tile: per stream s, rows s d + c0 .. + 15 in five 64-column
  // boxes, at rows 16 s .. 16 s + 15 of each K slice.  Every pass's B
  // barrier is armed for the bytes the peers will send.
  if (tid == 0) {
    ptx::mbar_init(bar_w, 1);
#pragma unroll
    for (int p = 0; p < P::NPASS; ++p) {
      ptx::mbar_init(&bar_mma[p], 1);
      ptx::mbar_init(&bar_b[p], 1);
    }
    ptx::fence_barrier_init();
    ptx::mbar_arrive_expect_tx(bar_w, W::M * KD * 2);
    for (int p = 0; p < npass; ++p) ptx::mbar_arrive_expect_tx(&bar_b[p], P::UP_RECV);
    const uint64_t once = ptx::policy_evict_first();
    if (a.W_up_tiles == nullptr) {
#pragma unroll
      for (int s = 0; s < kStreams; ++s) {
#pragma unroll
        for (int j = 0; j < W::NSL_U; ++j) {
          ptx::tma_load_2d(sa + j * W::SLICE_A + s * (W::UC * 128), &args.w, 64 * j, s * D + c0, bar_w, once);
        }
      }
    } else {
      copy_sw_tile<W::M * KD * 2>(sa, a.W_up_tiles, blockIdx.x, bar_w, once);
    }
  }
  // Gates of the 64 rows (weights: before the dependency wait).
  if (tid < W::M) {
    const float g = __ldg(a.gate + (tid / W::UC) * D + c0 + (tid % W::UC));
    sig[tid] = 1.0f / (1.0f + expf(-g));
  }
  if (warp == 1) {
    __syncwarp();  // tcgen05.alloc is .aligned
    ptx::tmem_alloc(tslot, W::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;

  // R' = R + P of the tile's rows for every token, into rp[t][row]: 16
  // float4 per token (four streams x 16 columns).
  constexpr int RP4 = ((MULTI ? W::TW : P::TP) * 16 + W::THREADS - 1) / W::THREADS;
  float4 rr[RP4], pp[RP4];
  auto load_rp = [&]() {
#pragma unroll
    for (int m = 0; m < RP4; ++m) {
      const int idx = tid + m * W::THREADS;
      rr[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      pp[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < T * 16) {
        const int t = idx >> 4, s = (idx >> 2) & 3, f = idx & 3;
        const size_t off = (size_t)t * W::N + s * D + c0 + 4 * f;
        rr[m] = __ldcg(reinterpret_cast<const float4*>(a.R + off));
        if (a.P) pp[m] = __ldcg(reinterpret_cast<const float4*>(a.P + off));
      }
    }
  };
  // Independent mode: R and P do not depend on the previous read.
  if (a.independent) load_rp();
  ptx::wait_prerequisites();  // the partials, R and P are ready from here on
  ptx::launch_dependents();
  if (!a.independent) load_rp();
  // R' of every token into shared memory (read by the epilogue only).
#pragma unroll
  for (int m = 0; m < RP4; ++m) {
    const int idx = tid + m * W::THREADS;
    if (idx < T * 16) {
      const int t = idx >> 4, s = (idx >> 2) & 3, f = idx & 3;
      *reinterpret_cast<float4*>(rp + t * W::M + s * W::UC + 4 * f) =
          make_float4(__fadd_rn(rr[m].x, pp[m].x), __fadd_rn(rr[m].y, pp[m].y), __fadd_rn(rr[m].z, pp[m].z),
                      __fadd_rn(rr[m].w, pp[m].w));
    }
  }
  ptx::cluster_wait();  // every CTA of the cluster runs, its barriers armed, before anyone sends

  const uint32_t a0 = ptx::smem_u32(sa);
  bool ok = true;  // thread 0: the weight tile and the peers' rows landed
  constexpr int CI = (P::TPR * W::KD4 + W::THREADS - 1) / W::THREADS;  // combine items per thread
  using Part = float4[CI][kStreams];
  // This rank's tokens of pass p: the four streams' partials over all K.
  auto load_pass = [&](int p, Part& pv) {
    const int t0 = p * P::TP;
#pragma unroll
    for (int i = 0; i < CI; ++i) {
      const int idx = tid + i * W::THREADS;
      const int t = t0 + (int)rank * P::TPR + idx / W::KD4;
#pragma unroll
      for (int s = 0; s < kStreams; ++s) {
        pv[i][s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < P::TPR * W::KD4 && t < T) {
          pv[i][s] = __ldcg(reinterpret_cast<const float4*>(a.part + ((size_t)s * a.T_max + t) * KD) + idx % W::KD4);
        }
      }
    }
  };
  Part pv;
  load_pass(0, pv);
  for (int p = 0; p < npass; ++p) {
    const int t0 = p * P::TP;
    unsigned char* bp = sb;
    if (p >= 1) {
      // The buffer of every CTA of the cluster was last read by the MMAs of
      // pass p - 1: all of them are done before anyone writes it again.
      if (tid == 0 && ok) ok = wait_bar(&bar_mma[p - 1], 0, a.err, kErrUpWeights);
      __syncwarp();
      ptx::tc_fence_before();
      ptx::cluster_arrive_release();
      ptx::cluster_wait();
      ptx::tc_fence_after();
    }
    // lo in stream order, its B rows into this CTA's buffer.
#pragma unroll
    for (int i = 0; i < CI; ++i) {
      const int idx = tid + i * W::THREADS;
      const int tl = (int)rank * P::TPR + idx / W::KD4;  // token within the pass
      if (idx < P::TPR * W::KD4 && t0 + tl < T) {
        const int k = 4 * (idx % W::KD4);
        float4 l;
        l.x = ((pv[i][0].x + pv[i][1].x) + pv[i][2].x) + pv[i][3].x;
        l.y = ((pv[i][0].y + pv[i][1].y) + pv[i][2].y) + pv[i][3].y;
        l.z = ((pv[i][0].z + pv[i][1].z) + pv[i][2].z) + pv[i][3].z;
        l.w = ((pv[i][0].w + pv[i][1].w) + pv[i][2].w) + pv[i][3].w;
        if (cq == 0) *reinterpret_cast<float4*>(a.lo + (size_t)(t0 + tl) * KD + k) = l;
        uint2 hi, lo;
        split4(l, hi, lo);
        *reinterpret_cast<uint2*>(bp + sw128_off<P::BROWS>(2 * tl, k)) = hi;
        *reinterpret_cast<uint2*>(bp + sw128_off<P::BROWS>(2 * tl + 1, k)) = lo;
      }
    }
    // The registers are free: the next pass's partial loads go out now.
    if (p + 1 < npass) load_pass(p + 1, pv);
    ptx::fence_proxy_async_smem();  // these stores, visible to the bulk copies and the tensor cores
    __syncthreads();
    if (tid == 0) {
      // This rank's B rows (whole 128-byte rows of every K slice) into the
      // same place of every peer.
      const uint32_t rows = ptx::smem_u32(bp) + rank * (uint32_t)(P::RROWS * 128);
      const uint32_t bar = ptx::smem_u32(&bar_b[p]);
#pragma unroll
      for (int j = 0; j < W::NSL_U; ++j) {
#pragma unroll
        for (int q = 1; q < W::UCL; ++q) {
          const uint32_t peer = (rank + (uint32_t)q) % W::UCL;
          ptx::bulk_s2peer(rows + j * P::SLICE_B, rows + j * P::SLICE_B, P::RROWS * 128, bar, peer);
        }
      }
      // The peers' rows of the pass, then the MMAs.
      ok = wait_bar(&bar_b[p], 0, a.err, kErrUpWeights) && ok;
      if (p == 0) ok = wait_bar(bar_w, 0, a.err, kErrUpWeights) && ok;
      ptx::tc_fence_after();
      if (ok) {
        umma_pass<KD, W::SLICE_A, P::SLICE_B>(tmem + (uint32_t)(p * P::PCOLS), a0, ptx::smem_u32(bp), W::M,
                                              (2 * min(P::TP, T - t0) + 7) & ~7);
        ptx::umma_commit(&bar_mma[p]);
      } else {
        mbar_arrive_local(&bar_mma[p]);
      }
    }
  }
  // Every bulk copy out of this CTA has landed once every peer has passed its
  // waits above: only then may a CTA leave (a copy reads its source rows).
  __syncwarp();
  ptx::cluster_arrive_release();
  ptx::cluster_wait();
  bool done = wait_bar(&bar_mma[npass - 1], 0, a.err, kErrUpWeights);
  (void)done;
  __syncwarp();
  ptx::tc_fence_after();

  // Epilogue: u from the accumulator, out = R' + sigmoid(g) u, R' replaced
  // by out in rp for the stream mean.
  {
    const int s = warp & 3, h = warp >> 2;
    const int ncols = npass * P::PCOLS;
    const int row = 16 * s + (lane & 15);
    for (int c = h * (ncols / 2); c < (h + 1) * (ncols / 2); c += 16) {
      uint32_t d[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(32 * s) << 16) + (uint32_t)c, d);
      ptx::tmem_wait_ld();
      if (lane < 16) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int col = c + 2 * e;
          const int t = (col / P::PCOLS) * P::TP + (col % P::PCOLS) / 2;
          if (t < T) {
            const float u = __fadd_rn(__uint_as_float(d[2 * e]), __uint_as_float(d[2 * e + 1]));
            const float r = rp[t * W::M + row];
            const float o = __fmaf_rn(sig[row], u, r);
            const size_t off = (size_t)t * W::N + s * D + c0 + lane;
            a.out[off] = o;
            if (a.r_out != nullptr) a.r_out[off] = r;
            rp[t * W::M + row] = o;
          }
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, W::TMEM_COLS);
  for (int idx = tid; idx < T * W::UC; idx += W::THREADS) {
    const int t = idx / W::UC, j = idx % W::UC;
    const float* o = rp + t * W::M + j;
    a.mean[(size_t)t * D + c0 + j] = (((o[0] + o[W::UC]) + o[2 * W::UC]) + o[3 * W::UC]) * 0.25f;
  }
  if (tid == 0 && !ok) drain(bar_w, 0);
}

// ---- Weights in swizzled tile order: each CTA's tile of the tensor-memory
// kernels (64 rows x 320 columns of W_down for a down CTA, 64 rows x K of
// W_up for a wide up CTA) as one contiguous block of five 64-column slices,
// each 64 rows of 128 bytes whose 16-byte chunk p holds the row's chunk
// p ^ (row mod 8): the layout the TMA boxes write into shared memory, so a
// CTA copies its tile in four contiguous pieces and computes on the same
// bytes.  One thread per 16-byte chunk.
template <int D, int KD>
__global__ void __launch_bounds__(256) hc_pack_down_sw_kernel(const uint16_t* __restrict__ W,
                                                              uint16_t* __restrict__ tiles) {
  using G = WGeo<D, KD>;
  constexpr int CHUNKS16 = G::M * G::KC / 8;  // 16-byte chunks of a tile
  const size_t tile = (size_t)blockIdx.y * G::CHUNKS + blockIdx.x;  // (row group, column chunk)
  uint4* dst = reinterpret_cast<uint4*>(tiles) + tile * CHUNKS16;
  for (int i = threadIdx.x; i < CHUNKS16; i += blockDim.x) {
    const int j = i / (G::M * 8), r = (i / 8) % G::M, p = i % 8;  // slice, row, chunk position
    const int k = 64 * j + 8 * (p ^ (r & 7));
    dst[i] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)(blockIdx.y * G::M + r) * G::N + blockIdx.x * G::KC + k));
  }
}

template <int D, int KD>
__global__ void __launch_bounds__(256) hc_pack_up_sw_kernel(const uint16_t* __restrict__ W,
                                                            uint16_t* __restrict__ tiles) {
  using G = WGeo<D, KD>;
  constexpr int CHUNKS16 = G::M * KD / 8;
  uint4* dst = reinterpret_cast<uint4*>(tiles) + (size_t)blockIdx.x * CHUNKS16;
  for (int i = threadIdx.x; i < CHUNKS16; i += blockDim.x) {
    const int j = i / (G::M * 8), r = (i / 8) % G::M, p = i % 8;  // slice, row 16 s + c, chunk position
    const int k = 64 * j + 8 * (p ^ (r & 7));
    const size_t row = (size_t)(r / G::UC) * D + blockIdx.x * G::UC + (r % G::UC);
    dst[i] = __ldg(reinterpret_cast<const uint4*>(W + row * KD + k));
  }
}

}  // namespace hc
