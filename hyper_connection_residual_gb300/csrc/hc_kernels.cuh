// CUDA-core kernels of the hyper-connection read for sm_103a.
//
// The read (defined in include/hc_read.h) is two dependent weight streams:
// W_down (K x N BF16) and W_up (N x K BF16), 13.1 MB per read at d = 2560,
// K = 320.  At T <= 8 tokens it is bound by HBM bandwidth, so both kernels are
// built around one idea: every CTA issues bulk async copies (TMA engine) of its
// whole weight tile into shared memory at entry, before it waits for the
// previous kernel (programmatic dependent launch), so the weights of this
// kernel and of the kernels queued behind it stream continuously.
//
// Kernel 1, hc_down_kernel (design ancestor: gr_fused_down_kernel in "#2812
// sycl: STRATA_GR_FUSED=1, the two-kernel BF16 hyper-connection read
// (opt-in)", section "What changed"): a CTA owns 32 rows of W_down x one slab
// of d/4 columns (a quarter of a stream).  It commits the pending write for
// its slab, stages x = R' * w_norm unscaled in shared memory with the slab's
// sums of squares, and forms 32 partial dot products per token over the slab.
// The last CTA of a row group to arrive (atomic ticket) combines the 16
// slabs' partials in a fixed order, applies rs per stream, writes lo and
// resets the ticket.
//
// Kernel 2, hc_up_kernel (design ancestor: gr_fused_up_kernel, same section):
// a CTA owns 16 columns x 4 streams = 64 rows of W_up, so the stream mean of
// its columns stays inside the CTA.  Four quarters of K are summed in a fixed
// order, then the epilogue writes out = R' + sigmoid(g) * u and the mean.
//
// Both kernels process tokens in groups of TT (TT = T for T <= 8) with the
// weight tile held in shared memory across groups.  Every reduction has a
// fixed order, so results do not depend on scheduling: direct calls and graph
// replays give the same bits.
#pragma once

#include <cstdint>

#include "hc_ptx.cuh"

namespace hc {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStreams = 4;
constexpr int kMaxT = 64;
// A bounded wait gives up after this long (the copies it waits for take a few
// microseconds) and records an error bit instead of hanging.
constexpr uint64_t kWaitNs = 1000000000ull;

// Error bits of the handle's device error word.
constexpr unsigned kErrDownNorm = 1u;
constexpr unsigned kErrDownWeights = 2u;
constexpr unsigned kErrUpGate = 4u;
constexpr unsigned kErrUpWeights = 8u;

template <int D, int KD>
struct Geo {
  static constexpr int N = kStreams * D;
  // ---- down kernel: 32 rows x SLAB columns per CTA
  static constexpr int SLAB = D / 4;
  static constexpr int SLABS = N / SLAB;             // 16
  static constexpr int SLABS_PER_STREAM = D / SLAB;  // 4
  static constexpr int DN_ROWS = 32;
  static constexpr int ROW_GROUPS = KD / DN_ROWS;
  static constexpr int DN_PITCH = SLAB * 2 + 16;     // bytes; = 16 (mod 128): conflict-free rows
  static constexpr int DN_CPW = SLAB / kWarps;       // columns per warp
  static constexpr int DN_CHUNKS = DN_CPW / 8;       // 16-byte chunks per warp row
  // ---- up kernel: 16 columns x 4 streams = 64 rows per CTA
  static constexpr int UP_COLS = 16;
  static constexpr int UP_ROWS = UP_COLS * kStreams;
  static constexpr int UP_CTAS = D / UP_COLS;
  static constexpr int UP_PITCH = KD * 2 + 16;       // bytes; = 16 (mod 128)
  static constexpr int UP_KQ = KD / 4;               // K per quarter
  static constexpr int UP_CHUNKS = UP_KQ / 8;

  static_assert(SLAB % (8 * kWarps) == 0, "slab must split into 16-byte chunks per warp");
  static_assert(KD % DN_ROWS == 0 && KD % 32 == 0, "K must be a multiple of 32");
  static_assert(DN_PITCH % 128 == 16 && UP_PITCH % 128 == 16, "pitch must be 16 mod 128");
  static_assert(D % UP_COLS == 0, "d must be a multiple of 16");
};

template <int D, int KD, int TT>
struct DownSmem {
  using G = Geo<D, KD>;
  static constexpr int BAR = 0;  // two mbarriers
  static constexpr int FLAG = 16;
  static constexpr int W = 128;
  static constexpr int WN = W + G::DN_ROWS * G::DN_PITCH;
  static constexpr int X = WN + G::SLAB * 4;
  static constexpr int RED = X + TT * G::SLAB * 4;
  static constexpr int SSW = RED + kWarps * TT * 32 * 4;
  static constexpr int RS = SSW + kWarps * TT * 4;
  static constexpr int BYTES = RS + kMaxT * kStreams * 4;
};

template <int D, int KD, int TT>
struct UpSmem {
  using G = Geo<D, KD>;
  static constexpr int BAR = 0;
  static constexpr int FLAG = 16;
  static constexpr int W = 128;
  static constexpr int GATE = W + G::UP_ROWS * G::UP_PITCH;
  static constexpr int SIG = GATE + G::UP_ROWS * 4;
  static constexpr int LO = SIG + G::UP_ROWS * 4;
  static constexpr int RED = LO + TT * KD * 4;
  static constexpr int OUT = RED + 4 * TT * G::UP_ROWS * 4;
  static constexpr int BYTES = OUT + TT * G::UP_ROWS * 4;
};

struct DownArgs {
  const float* R;          // [T][N]
  const float* P;          // [T][N] or null
  const float* w_norm;     // [N]
  const uint16_t* W_down;  // [K][N] BF16
  float* part;             // scratch [SLABS][T_max][K]
  float* ss_part;          // scratch [ROW_GROUPS][SLABS][T_max]
  unsigned* counters;      // scratch [ROW_GROUPS], zero between reads
  unsigned* err;           // scratch error word
  float* lo;               // [T][K]
  float* rs_out;           // [T][4] or null
  int T;
  int T_max;
  float eps;
};

struct UpArgs {
  const float* R;        // [T][N]
  const float* P;        // [T][N] or null
  const float* gate;     // [N]
  const uint16_t* W_up;  // [N][K] BF16
  const float* lo;       // [T][K]
  float* out;            // [T][N]
  float* mean;           // [T][d]
  float* r_out;          // [T][N] or null
  unsigned* err;
  int T;
};

// Eight BF16 values (one 16-byte chunk) widened to fp32: a BF16 is the upper
// half of a binary32, so widening is a shift or a mask.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&w)[8]) {
  w[0] = __uint_as_float(v.x << 16);
  w[1] = __uint_as_float(v.x & 0xffff0000u);
  w[2] = __uint_as_float(v.y << 16);
  w[3] = __uint_as_float(v.y & 0xffff0000u);
  w[4] = __uint_as_float(v.z << 16);
  w[5] = __uint_as_float(v.z & 0xffff0000u);
  w[6] = __uint_as_float(v.w << 16);
  w[7] = __uint_as_float(v.w & 0xffff0000u);
}

// Thread 0 waits (bounded) for the barrier's phase `parity`; the outcome is
// shared through `flag`.  On success every thread then observes the completed
// phase itself (which returns at once), so the bulk-copied data is visible to
// all.  Returns false after recording `code` in *err on a timeout.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                         unsigned code, volatile int* flag) {
  if (threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    bool ok = true;
    while (!ptx::mbar_try_wait(bar, parity)) {
      if (ptx::globaltimer_ns() - t0 > kWaitNs) {
        ok = false;
        break;
      }
    }
    if (!ok) atomicOr(err, code);
    *flag = ok ? 1 : 0;
  }
  __syncthreads();
  const bool ok = *flag != 0;
  if (ok) {
    for (uint32_t i = 0; !ptx::mbar_try_wait(bar, parity) && i < (1u << 20); ++i) {
    }
  }
  __syncthreads();
  return ok;
}

// After a timeout: wait (bounded again) for copies still in flight into this
// CTA's shared memory before the CTA exits.
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  if (threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < kWaitNs) {
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ kernel 1
template <int D, int KD, int TT>
__global__ void __launch_bounds__(kThreads, 2) hc_down_kernel(const DownArgs a) {
  using G = Geo<D, KD>;
  using S = DownSmem<D, KD, TT>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + S::BAR);
  uint64_t* bar_n = bar_w + 1;
  volatile int* flag = reinterpret_cast<volatile int*>(smem + S::FLAG);
  unsigned char* w_s = smem + S::W;
  const float* wn_s = reinterpret_cast<const float*>(smem + S::WN);
  float* x_s = reinterpret_cast<float*>(smem + S::X);
  float* red_s = reinterpret_cast<float*>(smem + S::RED);
  float* ssw_s = reinterpret_cast<float*>(smem + S::SSW);
  float* rs_s = reinterpret_cast<float*>(smem + S::RS);

  const int slab = blockIdx.x;
  const int rg = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = slab * G::SLAB;
  const int row0 = rg * G::DN_ROWS;

  // Parameters first: they do not depend on the previous kernel.
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::mbar_init(bar_n, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_w, G::DN_ROWS * G::SLAB * 2);
      ptx::mbar_arrive_expect_tx(bar_n, G::SLAB * 4);
    }
    __syncwarp();
    const uint64_t once = ptx::policy_evict_first();  // each weight byte is read once
    ptx::bulk_g2s(w_s + lane * G::DN_PITCH, a.W_down + (size_t)(row0 + lane) * G::N + col0,
                  G::SLAB * 2, bar_w, once);
    if (lane == 0) {
      // w_norm's slab is read by every row group: keep it in L2.
      ptx::bulk_g2s(smem + S::WN, a.w_norm + col0, G::SLAB * 4, bar_n, ptx::policy_evict_last());
    }
  }
  ptx::launch_dependents();
  ptx::wait_prerequisites();
  __syncthreads();

  if (!cta_wait(bar_n, 0, a.err, kErrDownNorm, flag)) {
    drain(bar_w, 0);
    return;
  }

  const int T = a.T;
  bool weights_ready = false;
  for (int t0 = 0; t0 < T; t0 += TT) {
    const int tg = min(TT, T - t0);

    // Commit the pending write, stage x = R' * w_norm, sum R'^2 (this slab).
    float ssl[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      ssl[t] = 0.f;
      if (t < tg) {
        const size_t base = (size_t)(t0 + t) * G::N + col0;
        const float4* Rt = reinterpret_cast<const float4*>(a.R + base);
        const float4* Pt = a.P ? reinterpret_cast<const float4*>(a.P + base) : nullptr;
        for (int c4 = tid; c4 < G::SLAB / 4; c4 += kThreads) {
          float4 r = __ldcg(Rt + c4);
          const float4 p = Pt ? __ldcg(Pt + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
          r.x = __fadd_rn(r.x, p.x);
          r.y = __fadd_rn(r.y, p.y);
          r.z = __fadd_rn(r.z, p.z);
          r.w = __fadd_rn(r.w, p.w);
          const float4 w = reinterpret_cast<const float4*>(wn_s)[c4];
          reinterpret_cast<float4*>(x_s + t * G::SLAB)[c4] =
              make_float4(__fmul_rn(r.x, w.x), __fmul_rn(r.y, w.y), __fmul_rn(r.z, w.z),
                          __fmul_rn(r.w, w.w));
          ssl[t] = __fmaf_rn(r.x, r.x, ssl[t]);
          ssl[t] = __fmaf_rn(r.y, r.y, ssl[t]);
          ssl[t] = __fmaf_rn(r.z, r.z, ssl[t]);
          ssl[t] = __fmaf_rn(r.w, r.w, ssl[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float v = ssl[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) ssw_s[warp * TT + t] = v;
    }
    if (!weights_ready) {
      if (!cta_wait(bar_w, 0, a.err, kErrDownWeights, flag)) return;
      weights_ready = true;
    } else {
      __syncthreads();
    }
    if (tid < tg) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += ssw_s[w * TT + tid];
      __stcg(a.ss_part + (size_t)(rg * G::SLABS + slab) * a.T_max + t0 + tid, s);
    }

    // Partial dot products: lane = row, warp = column range of the slab.
    const unsigned char* wrow = w_s + lane * G::DN_PITCH + warp * G::DN_CPW * 2;
    const float* xw = x_s + warp * G::DN_CPW;
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
#pragma unroll 2
    for (int j = 0; j < G::DN_CHUNKS; ++j) {
      float w[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(wrow + j * 16), w);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float4 xa = *reinterpret_cast<const float4*>(xw + t * G::SLAB + j * 8);
        const float4 xb = *reinterpret_cast<const float4*>(xw + t * G::SLAB + j * 8 + 4);
        float s = acc[t];
        s = __fmaf_rn(w[0], xa.x, s);
        s = __fmaf_rn(w[1], xa.y, s);
        s = __fmaf_rn(w[2], xa.z, s);
        s = __fmaf_rn(w[3], xa.w, s);
        s = __fmaf_rn(w[4], xb.x, s);
        s = __fmaf_rn(w[5], xb.y, s);
        s = __fmaf_rn(w[6], xb.z, s);
        s = __fmaf_rn(w[7], xb.w, s);
        acc[t] = s;
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) red_s[(warp * TT + t) * 32 + lane] = acc[t];
    __syncthreads();
    for (int idx = tid; idx < tg * 32; idx += kThreads) {
      const int t = idx >> 5, r = idx & 31;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red_s[(w * TT + t) * 32 + r];
      __stcg(a.part + ((size_t)slab * a.T_max + t0 + t) * KD + row0 + r, s);
    }
    __syncthreads();
  }

  // Arrival: the last CTA of this row group combines the slabs.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned ticket = atomicAdd(a.counters + rg, 1u);
    *flag = (ticket == (unsigned)(G::SLABS - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (*flag == 0) return;
  __threadfence();

  for (int idx = tid; idx < T * kStreams; idx += kThreads) {
    const int t = idx >> 2, s = idx & 3;
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < G::SLABS_PER_STREAM; ++q) {
      ss += __ldcg(a.ss_part + (size_t)(rg * G::SLABS + s * G::SLABS_PER_STREAM + q) * a.T_max + t);
    }
    const float rs = 1.0f / sqrtf(ss / (float)D + a.eps);
    rs_s[idx] = rs;
    if (a.rs_out != nullptr && rg == 0) a.rs_out[idx] = rs;
  }
  __syncthreads();
  for (int idx = tid; idx < T * G::DN_ROWS; idx += kThreads) {
    const int t = idx >> 5, r = idx & 31;
    float l = 0.f;
#pragma unroll
    for (int s = 0; s < kStreams; ++s) {
      float ps = 0.f;
#pragma unroll
      for (int q = 0; q < G::SLABS_PER_STREAM; ++q) {
        ps += __ldcg(a.part + ((size_t)(s * G::SLABS_PER_STREAM + q) * a.T_max + t) * KD + row0 + r);
      }
      l = __fmaf_rn(rs_s[t * kStreams + s], ps, l);
    }
    a.lo[(size_t)t * KD + row0 + r] = l;
  }
  if (tid == 0) atomicExch(a.counters + rg, 0u);
}

// ------------------------------------------------------------------ kernel 2
template <int D, int KD, int TT>
__global__ void __launch_bounds__(kThreads, 2) hc_up_kernel(const UpArgs a) {
  using G = Geo<D, KD>;
  using S = UpSmem<D, KD, TT>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + S::BAR);
  uint64_t* bar_g = bar_w + 1;
  volatile int* flag = reinterpret_cast<volatile int*>(smem + S::FLAG);
  unsigned char* w_s = smem + S::W;
  const float* g_s = reinterpret_cast<const float*>(smem + S::GATE);
  float* sig_s = reinterpret_cast<float*>(smem + S::SIG);
  float* lo_s = reinterpret_cast<float*>(smem + S::LO);
  float* red_s = reinterpret_cast<float*>(smem + S::RED);
  float* out_s = reinterpret_cast<float*>(smem + S::OUT);

  const int c0 = blockIdx.x * G::UP_COLS;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

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
    // Local row r = s * 16 + j holds global row s * d + c0 + j.
    for (int r = lane; r < G::UP_ROWS; r += 32) {
      const int grow = (r / G::UP_COLS) * D + c0 + (r % G::UP_COLS);
      ptx::bulk_g2s(w_s + r * G::UP_PITCH, a.W_up + (size_t)grow * KD, KD * 2, bar_w, once);
    }
    if (lane < kStreams) {
      ptx::bulk_g2s(smem + S::GATE + lane * G::UP_COLS * 4, a.gate + lane * D + c0,
                    G::UP_COLS * 4, bar_g, once);
    }
  }
  ptx::launch_dependents();
  ptx::wait_prerequisites();
  __syncthreads();

  if (!cta_wait(bar_g, 0, a.err, kErrUpGate, flag)) {
    drain(bar_w, 0);
    return;
  }
  if (tid < G::UP_ROWS) sig_s[tid] = 1.0f / (1.0f + expf(-g_s[tid]));

  const int T = a.T;
  bool weights_ready = false;
  for (int t0 = 0; t0 < T; t0 += TT) {
    const int tg = min(TT, T - t0);
    const float4* lo_g = reinterpret_cast<const float4*>(a.lo + (size_t)t0 * KD);
    for (int idx = tid; idx < tg * KD / 4; idx += kThreads) {
      reinterpret_cast<float4*>(lo_s)[idx] = __ldcg(lo_g + idx);
    }
    if (!weights_ready) {
      if (!cta_wait(bar_w, 0, a.err, kErrUpWeights, flag)) return;
      weights_ready = true;
    } else {
      __syncthreads();
    }

    // u for 64 rows: lane = row within a half, warp = (half, K quarter).
    const int half = warp & 1;
    const int kq = warp >> 1;
    const int row = half * 32 + lane;
    const unsigned char* wrow = w_s + row * G::UP_PITCH + kq * G::UP_KQ * 2;
    const float* lw = lo_s + kq * G::UP_KQ;
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
#pragma unroll 2
    for (int j = 0; j < G::UP_CHUNKS; ++j) {
      float w[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(wrow + j * 16), w);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float4 la = *reinterpret_cast<const float4*>(lw + t * KD + j * 8);
        const float4 lb = *reinterpret_cast<const float4*>(lw + t * KD + j * 8 + 4);
        float s = acc[t];
        s = __fmaf_rn(w[0], la.x, s);
        s = __fmaf_rn(w[1], la.y, s);
        s = __fmaf_rn(w[2], la.z, s);
        s = __fmaf_rn(w[3], la.w, s);
        s = __fmaf_rn(w[4], lb.x, s);
        s = __fmaf_rn(w[5], lb.y, s);
        s = __fmaf_rn(w[6], lb.z, s);
        s = __fmaf_rn(w[7], lb.w, s);
        acc[t] = s;
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) red_s[(kq * TT + t) * G::UP_ROWS + row] = acc[t];
    __syncthreads();

    // Epilogue: pending write, gate, stream mean.
    for (int idx = tid; idx < tg * G::UP_ROWS; idx += kThreads) {
      const int t = idx / G::UP_ROWS, r = idx % G::UP_ROWS;
      const float u = ((red_s[(0 * TT + t) * G::UP_ROWS + r] + red_s[(1 * TT + t) * G::UP_ROWS + r]) +
                       red_s[(2 * TT + t) * G::UP_ROWS + r]) +
                      red_s[(3 * TT + t) * G::UP_ROWS + r];
      const int i = (r / G::UP_COLS) * D + c0 + (r % G::UP_COLS);
      const size_t off = (size_t)(t0 + t) * G::N + i;
      const float rp = __fadd_rn(__ldcg(a.R + off), a.P ? __ldcg(a.P + off) : 0.0f);
      const float o = __fmaf_rn(sig_s[r], u, rp);
      a.out[off] = o;
      if (a.r_out != nullptr) a.r_out[off] = rp;
      out_s[t * G::UP_ROWS + r] = o;
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
}

}  // namespace hc
