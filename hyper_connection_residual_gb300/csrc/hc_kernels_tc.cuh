// Tensor-core (warp-level mma.sync, BF16 in, FP32 accumulate) variants of the
// two read kernels.
//
// The read is a skinny contraction: [T x N] x [N x K] for the down projection
// and [T x K] x [K x N] for the up projection, with BF16 weights.  The FP32
// activations (x = R' * w_norm for the down projection, lo for the up
// projection) are split into two BF16 terms, hi = bf16(x) and
// lo = bf16(x - hi) (x - hi is exact in FP32), so that hi + lo carries 16
// significant bits and the products keep a relative error near 2^-17 instead
// of the 2^-9 of a single BF16 term; both terms go through the MMA as separate
// columns of the B operand (column 2t holds token t's hi, column 2t+1 its lo)
// and are added in FP32 afterwards.  Accumulation is FP32 inside the MMA.
//
// Tiling, data movement, the cluster combine and the programmatic-launch
// protocol are the ones of the CUDA-core kernels (hc_kernels.cuh): the down
// kernel's CTA owns 32 rows of W_down x one d/4-column slab (two m16 tiles x
// four K-parts over 8 warps), the up kernel's CTA owns 64 rows of W_up (four
// m16 tiles x two K-halves).  Tokens are processed in groups of TG = 4 * NT
// (N = 8 * NT MMA columns).
#pragma once

#include <cuda_bf16.h>

#include "hc_kernels.cuh"

namespace hc {

// hi = bf16(x) and lo = bf16(x - hi) for four values, packed two per word.
// Each pair is converted by one packed round-to-nearest instruction; the hi
// values are widened back exactly by a shift or a mask.
__device__ __forceinline__ void split4(const float4 x, uint2& hi, uint2& lo) {
  const __nv_bfloat162 h01 = __floats2bfloat162_rn(x.x, x.y);
  const __nv_bfloat162 h23 = __floats2bfloat162_rn(x.z, x.w);
  const uint32_t u01 = *reinterpret_cast<const uint32_t*>(&h01);
  const uint32_t u23 = *reinterpret_cast<const uint32_t*>(&h23);
  const __nv_bfloat162 l01 = __floats2bfloat162_rn(__fsub_rn(x.x, __uint_as_float(u01 << 16)),
                                                   __fsub_rn(x.y, __uint_as_float(u01 & 0xffff0000u)));
  const __nv_bfloat162 l23 = __floats2bfloat162_rn(__fsub_rn(x.z, __uint_as_float(u23 << 16)),
                                                   __fsub_rn(x.w, __uint_as_float(u23 & 0xffff0000u)));
  hi = make_uint2(u01, u23);
  lo = make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
}

template <int D, int KD, int NT>
struct DownTcSmem {
  using G = Geo<D, KD>;
  static constexpr int TG = 4 * NT;
  static constexpr int NCOL = 8 * NT;
  static constexpr int XS_PITCH = G::SLAB * 2 + 16;   // bytes; = 16 (mod 128)
  static constexpr int BAR = 0;
  static constexpr int W = 128;
  static constexpr int XS = W + G::DN_ROWS * G::DN_PITCH;  // [NCOL][SLAB] bf16: hi, lo rows
  // [4 K-parts][TG][32] partials, over the x rows: written only once every
  // warp is past its MMAs (a CTA barrier), read before the next group's x.
  static constexpr int RED = XS;
  // [kMaxT] rs of the cluster leader, over the partials: used only after the
  // cluster barrier, when this CTA's own sums are done.
  static constexpr int RS = RED;
  static constexpr int SSW = XS + NCOL * XS_PITCH;    // [8 warps][TG]
  static constexpr int RECV = SSW + kWarps * TG * 4;  // [4][T] ss, then [4][T][32] partials
  static constexpr int bytes(int T) { return RECV + 4 * T * 4 + 4 * T * 32 * 4; }
  static constexpr int BYTES_MAX = RECV + 4 * kMaxT * 4 + 4 * kMaxT * 32 * 4;
  static_assert(XS_PITCH % 128 == 16, "x rows must be conflict-free for ldmatrix");
  static_assert(4 * TG * 32 * 4 <= NCOL * XS_PITCH && kMaxT <= 4 * TG * 32, "aliased regions fit");
};

template <int D, int KD, int NT>
struct UpTcSmem {
  using G = Geo<D, KD>;
  static constexpr int TG = 4 * NT;
  static constexpr int NCOL = 8 * NT;
  static constexpr int LS_PITCH = KD * 2 + 16;        // bytes; = 16 (mod 128)
  static constexpr int BAR = 0;
  static constexpr int W = 128;
  static constexpr int GATE = W + G::UP_ROWS * G::UP_PITCH;
  static constexpr int SIG = GATE + G::UP_ROWS * 4;
  static constexpr int LS = SIG + G::UP_ROWS * 4;     // [NCOL][KD] bf16: hi, lo rows
  static constexpr int RED = LS + NCOL * LS_PITCH;    // [2 K-halves][TG][64]
  static constexpr int OUT = RED + 2 * TG * G::UP_ROWS * 4;
  static constexpr int RP = OUT + TG * G::UP_ROWS * 4;
  static constexpr int BYTES = RP + TG * G::UP_ROWS * 4;
  static constexpr int bytes(int) { return BYTES; }
  static constexpr int BYTES_MAX = BYTES;
  static_assert(LS_PITCH % 128 == 16, "lo rows must be conflict-free for ldmatrix");
};

// CTAs per SM the register budget is cut for: at d = 2560 four for one token
// group (no spills at 64 registers; reads of a batch overlap better, measured
// 3.06 -> 2.71 us per read at T = 2 and 3.15 -> 2.82 at T = 4 on six
// streams), three for two groups (64 registers would spill: 3.67 -> 4.78 us
// at T = 6).
template <int D, int NT>
constexpr int tc_min_blocks() {
  return D == 2560 ? (NT == 1 ? 4 : 3) : 2;
}

// ------------------------------------------------------------------ kernel 1
// Grid (16 slabs, K/32 row groups), clusters of 4 along x (one stream).
template <int D, int KD, int NT>
__global__ void __launch_bounds__(kThreads, tc_min_blocks<D, NT>()) hc_down_tc_kernel(const DownArgs a) {
  using G = Geo<D, KD>;
  using S = DownTcSmem<D, KD, NT>;
  constexpr int TG = S::TG;
  constexpr int KPART = G::SLAB / 4;   // columns per K-part
  constexpr int KS = KPART / 16;       // k-steps per warp
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + S::BAR);
  unsigned char* w_s = smem + S::W;
  unsigned char* xs = smem + S::XS;
  float* red_s = reinterpret_cast<float*>(smem + S::RED);
  float* ssw_s = reinterpret_cast<float*>(smem + S::SSW);
  float* rs_s = reinterpret_cast<float*>(smem + S::RS);

  const int slab = blockIdx.x;
  const int stream = slab / G::SLABS_PER_STREAM;
  const int rg = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = slab * G::SLAB;
  const int row0 = rg * G::DN_ROWS;
  const int T = a.T;
  const int mt = warp & 1;    // m16 tile: rows 16 mt .. 16 mt + 15
  const int kp = warp >> 1;   // K-part: columns kp * KPART .. + KPART

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  float* recv_ss = cluster.map_shared_rank(reinterpret_cast<float*>(smem + S::RECV), 0);
  float* recv_p = recv_ss + 4 * T;

  ptx::cluster_arrive_relaxed();
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_w, G::DN_ROWS * G::SLAB * 2);
    }
    __syncwarp();
    const uint64_t once = ptx::policy_evict_first();
    ptx::bulk_g2s(w_s + lane * G::DN_PITCH, a.W_down + (size_t)(row0 + lane) * G::N + col0,
                  G::SLAB * 2, bar_w, once);
  }
  // This thread's float4 of the w_norm slab goes straight to registers (it is
  // not written by the previous kernel): no shared copy, no barrier.
  const int c4 = tid;  // one float4 of the slab per thread and token
  static_assert(G::DN_F4 <= kThreads, "one float4 per thread and token");
  const float4 wn = c4 < G::DN_F4 ? __ldg(reinterpret_cast<const float4*>(a.w_norm + col0) + c4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
  ptx::launch_dependents();
  __syncthreads();  // the mbarriers are initialised before any thread waits on them
  bool ok = true;
  // R, P and the scratch slot belong to the previous kernel until its end
  // (in independent mode only the previous read's outputs do, and the down
  // kernel waits at its end instead).
  if (!a.independent) ptx::wait_prerequisites();
  ptx::cluster_wait();

  // Lane address pattern of an ldmatrix.x4 on a 16x16 A tile.
  const int a_row = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
  const int a_col = kp * KPART + 8 * (lane >> 4);
  const uint32_t a_base = ptx::smem_u32(w_s + a_row * G::DN_PITCH + a_col * 2);
  // ... and of the B operand (rows = MMA columns).
  const int b_row = (lane & 7) + 8 * (lane >> 4);
  const int b_col = kp * KPART + 8 * ((lane >> 3) & 1);

  // R and P of one token group, this thread's float4 of the slab.
  float4 rv[TG], pv[TG];
  auto load_group = [&](int g0) {
    const int gn = min(TG, T - g0);
#pragma unroll
    for (int t = 0; t < TG; ++t) {
      rv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      pv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < gn && c4 < G::DN_F4) {
        const size_t base = (size_t)(g0 + t) * G::N + col0;
        rv[t] = __ldcg(reinterpret_cast<const float4*>(a.R + base) + c4);
        if (a.P) pv[t] = __ldcg(reinterpret_cast<const float4*>(a.P + base) + c4);
      }
    }
  };
  // The next group's loads go out while this group's MMAs run, in the
  // 4-token kernels (the 8-token ones would spill them at d = 2560 and
  // measured slower with them at d = 4096).
  constexpr bool kEarly = NT == 1;
  if (kEarly) load_group(0);
  for (int t0 = 0; t0 < T; t0 += TG) {
    const int tg = min(TG, T - t0);
    if (!kEarly) load_group(t0);
    float ssl[TG];
#pragma unroll
    for (int t = 0; t < TG; ++t) {
      ssl[t] = 0.f;
      if (c4 < G::DN_F4) {
        float4 r = rv[t];
        r.x = __fadd_rn(r.x, pv[t].x);
        r.y = __fadd_rn(r.y, pv[t].y);
        r.z = __fadd_rn(r.z, pv[t].z);
        r.w = __fadd_rn(r.w, pv[t].w);
        const float4 x = make_float4(__fmul_rn(r.x, wn.x), __fmul_rn(r.y, wn.y), __fmul_rn(r.z, wn.z),
                                     __fmul_rn(r.w, wn.w));
        uint2 hi, lo;
        split4(x, hi, lo);  // tokens past tg carry zeros
        *reinterpret_cast<uint2*>(xs + (2 * t) * S::XS_PITCH + c4 * 8) = hi;
        *reinterpret_cast<uint2*>(xs + (2 * t + 1) * S::XS_PITCH + c4 * 8) = lo;
        ssl[t] = __fmaf_rn(r.x, r.x, ssl[t]);
        ssl[t] = __fmaf_rn(r.y, r.y, ssl[t]);
        ssl[t] = __fmaf_rn(r.z, r.z, ssl[t]);
        ssl[t] = __fmaf_rn(r.w, r.w, ssl[t]);
      }
    }
    if (kEarly && t0 + TG < T) load_group(t0 + TG);
#pragma unroll
    for (int t = 0; t < TG; ++t) {
      float v = ssl[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) ssw_s[warp * TG + t] = v;
    }
    if (t0 == 0) ok = wait_bar(bar_w, 0, a.err, kErrDownWeights) && ok;
    __syncthreads();  // x (hi, lo) and the per-warp sums of squares are complete
    if (tid < tg) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += ssw_s[w * TG + tid];
      recv_ss[rank * T + t0 + tid] = v;
    }

    // Two accumulator sets (even and odd k-steps), added at the end: half the
    // dependent-MMA chain, a fixed order.
    float acc[NT][4], acc2[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
      acc2[n][0] = acc2[n][1] = acc2[n][2] = acc2[n][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t afrag[4];
      ptx::ldsm_x4(a_base + ks * 32, afrag[0], afrag[1], afrag[2], afrag[3]);
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3;
        float (&c0)[4] = (ks & 1) ? acc2[n] : acc[n];
        if (n + 1 < NT) {
          float (&c1)[4] = (ks & 1) ? acc2[n + 1] : acc[n + 1];
          ptx::ldsm_x4(ptx::smem_u32(xs + (n * 8 + b_row) * S::XS_PITCH + (b_col + ks * 16) * 2), b0, b1,
                       b2, b3);
          ptx::mma_bf16_16816(c0, afrag, b0, b1);
          ptx::mma_bf16_16816(c1, afrag, b2, b3);
        } else {
          ptx::ldsm_x2(ptx::smem_u32(xs + (n * 8 + (lane & 7)) * S::XS_PITCH + (b_col + ks * 16) * 2), b0,
                       b1);
          ptx::mma_bf16_16816(c0, afrag, b0, b1);
        }
      }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = __fadd_rn(acc[n][e], acc2[n][e]);
    }
    __syncthreads();  // every warp is done with the x rows the partials overwrite
    // Column 2t holds token t's hi part, 2t + 1 its lo part.
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int t = n * 4 + (lane & 3);
      const int r = mt * 16 + (lane >> 2);
      red_s[(kp * TG + t) * 32 + r] = __fadd_rn(acc[n][0], acc[n][1]);
      red_s[(kp * TG + t) * 32 + r + 8] = __fadd_rn(acc[n][2], acc[n][3]);
    }
    __syncthreads();
    for (int idx = tid; idx < tg * 32; idx += kThreads) {
      const int t = idx >> 5, r = idx & 31;
      const float v = ((red_s[(0 * TG + t) * 32 + r] + red_s[(1 * TG + t) * 32 + r]) +
                       red_s[(2 * TG + t) * 32 + r]) +
                      red_s[(3 * TG + t) * 32 + r];
      recv_p[(rank * T + t0 + t) * 32 + r] = v;
    }
    __syncthreads();
  }
  if (!ok) drain(bar_w, 0);
  ptx::cluster_arrive_release();
  ptx::cluster_wait();
  if (rank != 0) {
    if (a.independent) ptx::wait_prerequisites();
    return;
  }

  for (int t = tid; t < T; t += kThreads) {
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < G::SLABS_PER_STREAM; ++q) ss += recv_ss[q * T + t];
    const float rs = rsqrtf(ss * (1.0f / (float)D) + a.eps);
    rs_s[t] = rs;
    if (rg == 0 && a.rs_out != nullptr) a.rs_out[t * kStreams + stream] = rs;
  }
  __syncthreads();
  float* part = a.part + (size_t)stream * a.T_max * KD;
  for (int idx = tid; idx < T * G::DN_ROWS; idx += kThreads) {
    const int t = idx >> 5, r = idx & 31;
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < G::SLABS_PER_STREAM; ++q) p += recv_p[(q * T + t) * 32 + r];
    __stcg(part + (size_t)t * KD + row0 + r, __fmul_rn(rs_s[t], p));
  }
  if (a.independent) ptx::wait_prerequisites();  // complete only after the previous read
}

// ------------------------------------------------------------------ kernel 2
template <int D, int KD, int NT>
__global__ void __launch_bounds__(kThreads, tc_min_blocks<D, NT>()) hc_up_tc_kernel(const UpArgs a) {
  using G = Geo<D, KD>;
  using S = UpTcSmem<D, KD, NT>;
  constexpr int TG = S::TG;
  constexpr int KHALF = KD / 2;
  constexpr int KS = KHALF / 16;
  constexpr int EPI = (TG * G::UP_ROWS + kThreads - 1) / kThreads;
  constexpr int LO4 = (TG * KD / 4 + kThreads - 1) / kThreads;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + S::BAR);
  uint64_t* bar_g = bar_w + 1;
  unsigned char* w_s = smem + S::W;
  const float* g_s = reinterpret_cast<const float*>(smem + S::GATE);
  float* sig_s = reinterpret_cast<float*>(smem + S::SIG);
  unsigned char* ls = smem + S::LS;
  float* red_s = reinterpret_cast<float*>(smem + S::RED);
  float* out_s = reinterpret_cast<float*>(smem + S::OUT);
  float* rp_s = reinterpret_cast<float*>(smem + S::RP);

  const int c0 = blockIdx.x * G::UP_COLS;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int mt = warp & 3;   // m16 tile of the 64 rows
  const int kh = warp >> 2;  // K half

  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::mbar_init(bar_g, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_w, G::UP_ROWS * KD * 2);
      ptx::mbar_arrive_expect_tx(bar_g, G::UP_ROWS * 4);
    }
    __syncwarp();
    const uint64_t once = ptx::policy_evict_first();
    if (lane < kStreams) {
      ptx::bulk_g2s(smem + S::GATE + lane * G::UP_COLS * 4, a.gate + lane * D + c0,
                    G::UP_COLS * 4, bar_g, once);
    }
    for (int r = lane; r < G::UP_ROWS; r += 32) {
      const int grow = (r / G::UP_COLS) * D + c0 + (r % G::UP_COLS);
      ptx::bulk_g2s(w_s + r * G::UP_PITCH, a.W_up + (size_t)grow * KD, KD * 2, bar_w, once);
    }
  }
  __syncthreads();  // the mbarriers are initialised before any thread waits on them
  bool ok = true;
  if (tid < G::UP_ROWS) {
    ok = wait_bar(bar_g, 0, a.err, kErrUpGate);
    sig_s[tid] = 1.0f / (1.0f + expf(-g_s[tid]));
  }
  // Independent mode: R and P of the first token group do not depend on the
  // previous read; fetch them before waiting.
  float rr0[EPI], pp0[EPI];
  if (a.independent) load_rp<D, EPI>(a, c0, 0, min(TG, a.T), rr0, pp0);
  ptx::wait_prerequisites();  // the partials, R and P are ready from here on
  ptx::launch_dependents();

  const int a_row = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
  const int a_col = kh * KHALF + 8 * (lane >> 4);
  const uint32_t a_base = ptx::smem_u32(w_s + a_row * G::UP_PITCH + a_col * 2);
  const int b_row = (lane & 7) + 8 * (lane >> 4);
  const int b_col = kh * KHALF + 8 * ((lane >> 3) & 1);

  const int T = a.T;
  // All global loads of a token group: the four per-stream partials of lo,
  // then R and P of this CTA's rows.
  float4 pv[LO4][kStreams];
  float rr[EPI], pp[EPI];
  auto load_group = [&](int g0) {
    const int gn = min(TG, T - g0);
#pragma unroll
    for (int m = 0; m < LO4; ++m) {
      const int idx = tid + m * kThreads;
#pragma unroll
      for (int s = 0; s < kStreams; ++s) {
        pv[m][s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < gn * KD / 4) {
          pv[m][s] = __ldcg(reinterpret_cast<const float4*>(
                                a.part + ((size_t)s * a.T_max + g0) * KD) + idx);
        }
      }
    }
    if (g0 == 0 && a.independent) {
#pragma unroll
      for (int m = 0; m < EPI; ++m) {
        rr[m] = rr0[m];
        pp[m] = pp0[m];
      }
    } else {
      load_rp<D, EPI>(a, c0, g0, gn, rr, pp);
    }
  };
  // The next group's loads go out while this group's MMAs run, in the
  // 4-token kernels (the 8-token ones would spill them at d = 2560 and
  // measured slower with them at d = 4096).
  constexpr bool kEarly = NT == 1;
  if (kEarly) load_group(0);
  for (int t0 = 0; t0 < T; t0 += TG) {
    const int tg = min(TG, T - t0);
    if (!kEarly) load_group(t0);
    // lo (four partials in stream order), its hi/lo split, and this CTA's
    // share of the lo output.
#pragma unroll
    for (int m = 0; m < LO4; ++m) {
      const int idx = tid + m * kThreads;
      if (idx < TG * KD / 4) {
        float4 l;
        l.x = ((pv[m][0].x + pv[m][1].x) + pv[m][2].x) + pv[m][3].x;
        l.y = ((pv[m][0].y + pv[m][1].y) + pv[m][2].y) + pv[m][3].y;
        l.z = ((pv[m][0].z + pv[m][1].z) + pv[m][2].z) + pv[m][3].z;
        l.w = ((pv[m][0].w + pv[m][1].w) + pv[m][2].w) + pv[m][3].w;
        const int t = idx / (KD / 4), k4 = idx % (KD / 4);
        uint2 hi, lo;
        split4(l, hi, lo);  // tokens past tg carry zeros
        *reinterpret_cast<uint2*>(ls + (2 * t) * S::LS_PITCH + k4 * 8) = hi;
        *reinterpret_cast<uint2*>(ls + (2 * t + 1) * S::LS_PITCH + k4 * 8) = lo;
        const int k = k4 * 4;
        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = k + e;
          if (t < tg && kk / G::LO_PER_CTA == (int)blockIdx.x) a.lo[(size_t)(t0 + t) * KD + kk] = lv[e];
        }
      }
    }
#pragma unroll
    for (int m = 0; m < EPI; ++m) {
      const int idx = tid + m * kThreads;
      if (idx < tg * G::UP_ROWS) rp_s[idx] = __fadd_rn(rr[m], pp[m]);
    }
    if (kEarly && t0 + TG < T) load_group(t0 + TG);
    if (t0 == 0) ok = wait_bar(bar_w, 0, a.err, kErrUpWeights) && ok;
    __syncthreads();  // lo (hi, lo), R' and the gates are in shared memory

    // Two accumulator sets (even and odd k-steps), added at the end: half the
    // dependent-MMA chain, a fixed order.
    float acc[NT][4], acc2[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
      acc2[n][0] = acc2[n][1] = acc2[n][2] = acc2[n][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t afrag[4];
      ptx::ldsm_x4(a_base + ks * 32, afrag[0], afrag[1], afrag[2], afrag[3]);
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3;
        float (&c0)[4] = (ks & 1) ? acc2[n] : acc[n];
        if (n + 1 < NT) {
          float (&c1)[4] = (ks & 1) ? acc2[n + 1] : acc[n + 1];
          ptx::ldsm_x4(ptx::smem_u32(ls + (n * 8 + b_row) * S::LS_PITCH + (b_col + ks * 16) * 2), b0, b1,
                       b2, b3);
          ptx::mma_bf16_16816(c0, afrag, b0, b1);
          ptx::mma_bf16_16816(c1, afrag, b2, b3);
        } else {
          ptx::ldsm_x2(ptx::smem_u32(ls + (n * 8 + (lane & 7)) * S::LS_PITCH + (b_col + ks * 16) * 2), b0,
                       b1);
          ptx::mma_bf16_16816(c0, afrag, b0, b1);
        }
      }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = __fadd_rn(acc[n][e], acc2[n][e]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int t = n * 4 + (lane & 3);
      const int r = mt * 16 + (lane >> 2);
      red_s[(kh * TG + t) * G::UP_ROWS + r] = __fadd_rn(acc[n][0], acc[n][1]);
      red_s[(kh * TG + t) * G::UP_ROWS + r + 8] = __fadd_rn(acc[n][2], acc[n][3]);
    }
    __syncthreads();

    // Epilogue: pending write, gate, stream mean.
    for (int idx = tid; idx < tg * G::UP_ROWS; idx += kThreads) {
      const int t = idx / G::UP_ROWS, r = idx % G::UP_ROWS;
      const float u = red_s[(0 * TG + t) * G::UP_ROWS + r] + red_s[(1 * TG + t) * G::UP_ROWS + r];
      const int i = (r / G::UP_COLS) * D + c0 + (r % G::UP_COLS);
      const size_t off = (size_t)(t0 + t) * G::N + i;
      const float rp = rp_s[idx];
      const float o = __fmaf_rn(sig_s[r], u, rp);
      a.out[off] = o;
      if (a.r_out != nullptr) a.r_out[off] = rp;
      out_s[idx] = o;
    }
    __syncthreads();
    for (int idx = tid; idx < tg * G::UP_COLS; idx += kThreads) {
      const int t = idx / G::UP_COLS, j = idx % G::UP_COLS;
      const float* o = out_s + t * G::UP_ROWS + j;
      const float m = (((o[0] + o[G::UP_COLS]) + o[2 * G::UP_COLS]) + o[3 * G::UP_COLS]) * 0.25f;
      a.mean[(size_t)(t0 + t) * D + c0 + j] = m;
    }
    __syncthreads();
  }
  if (!ok) {
    drain(bar_g, 0);
    drain(bar_w, 0);
  }
}

}  // namespace hc
