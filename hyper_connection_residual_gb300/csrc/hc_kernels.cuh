// CUDA-core kernels of the hyper-connection read for sm_103a.
//
// The read (defined in include/hc_read.h) streams two BF16 weight matrices,
// W_down (K x N) and W_up (N x K): 13.1 MB per read at d = 2560, K = 320.
// On GB300 that is under 2 us of HBM time, so what limits a stream of reads is
// the chain of dependent latencies per read, not bandwidth.  The kernels are
// shaped to keep that chain short:
//
//  * every CTA issues bulk async copies (TMA engine) of its whole weight tile
//    into shared memory at entry, before it waits for the previous kernel
//    (programmatic dependent launch).  Weight prefetch is the only work done
//    before that wait, so nothing can race.  The down kernel lets the up
//    kernel launch at once (the up kernel's W_up streams while the down
//    kernel runs); the up kernel lets the next read launch once its own wait
//    has returned, which keeps waiting CTAs of later reads off the SMs while
//    this read computes;
//  * the down kernel's cross-CTA reduction stays on chip: the four CTAs that
//    cover one stream's four column slabs form a thread-block cluster; each
//    pushes its partial sums and sums of squares into the leader CTA's shared
//    memory (distributed shared memory), one cluster barrier later the leader
//    applies rs and writes the stream's partial; no global atomics, no last
//    arriver;
//  * after its dependency wait, each kernel issues all of its global loads
//    (R and P, or the partials and R and P) before using any of them;
//  * independent mode: when the host has established that the read takes
//    nothing the previous read on the stream writes (it compares address
//    ranges), the down kernel reads R and P and computes before it waits and
//    waits only at its end (so its read still completes after the previous
//    one), and the up kernel fetches R and P before its wait.  Because every
//    up kernel lets the next read launch only after its own wait has returned,
//    a read's down kernel starts after the read before the previous one has
//    completed: the previous read is the only one that can still be running.
//    Its partial sums go to the other of two scratch slots.
//
// Kernel 1, hc_down_kernel (design ancestor: gr_fused_down_kernel in "#2812
// sycl: STRATA_GR_FUSED=1, the two-kernel BF16 hyper-connection read
// (opt-in)", section "What changed"): a CTA owns 32 rows of W_down x one slab
// of d/4 columns.  It commits the pending write for its slab, stages
// x = R' * w_norm (rs not yet applied), accumulates the squares over its
// slab and forms 32 partial dot products per token (lane = row, so the x reads are shared-memory
// broadcasts).  The cluster of the stream's four slabs then sums the slabs in
// a fixed order, applies rs and writes part[s][t][k] = rs[t][s] * (slab sum).
// Partials live in one scratch slot per handle: a read's down kernel writes
// it only after the previous read has completed.
//
// Kernel 2, hc_up_kernel (design ancestor: gr_fused_up_kernel, same section):
// a CTA owns 16 columns x 4 streams = 64 rows of W_up, so the stream mean of
// its columns stays inside the CTA.  lo[t][k] = sum over the 4 streams of
// part (fixed order); four quarters of K are summed in a fixed order; the
// epilogue writes out = R' + sigmoid(g) * u and the mean.
//
// Kernel 1s, hc_down_s_kernel (T = 1, 2 at d = 2560): a CTA owns 8 rows of
// W_down over one stream's whole width, so the stream's sum of squares and
// the rows' dot products finish inside the CTA: no cluster, no exchange.
//
// In a batch of independent reads the kernels of many reads share the SMs,
// and the weight tiles an SM holds in flight set the bandwidth: the T = 1
// kernels are held to at most 48 registers so that registers do not cap the
// CTAs per SM below what their shared memory allows.
//
// Every reduction has a fixed order, so results do not depend on scheduling:
// direct calls and graph replays give the same bits.
#pragma once

#include <cuda_fp16.h>
#include <cooperative_groups.h>

#include <cstdint>

#include "hc_ptx.cuh"

namespace hc {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStreams = 4;
constexpr int kMaxT = 64;
// A bounded wait gives up after this long (the copies it waits for take a few
// microseconds) and records an error bit instead of hanging.
constexpr uint64_t kWaitNs = 1000000000ull;

// Error bits of the device error word.
constexpr unsigned kErrDownNorm = 1u;
constexpr unsigned kErrDownWeights = 2u;
constexpr unsigned kErrUpGate = 4u;
constexpr unsigned kErrUpWeights = 8u;

template <int D, int KD>
struct Geo {
  static constexpr int N = kStreams * D;
  // ---- down kernel: 32 rows x SLAB columns per CTA, 4 slabs per stream
  static constexpr int SLAB = D / 4;
  static constexpr int SLABS = N / SLAB;             // 16
  static constexpr int SLABS_PER_STREAM = D / SLAB;  // 4 = cluster size
  static constexpr int DN_ROWS = 32;
  static constexpr int ROW_GROUPS = KD / DN_ROWS;
  static constexpr int DN_PITCH = SLAB * 2 + 16;     // bytes; = 16 (mod 128): conflict-free rows
  static constexpr int DN_CPW = SLAB / kWarps;       // columns per warp
  static constexpr int DN_CHUNKS = DN_CPW / 8;       // 16-byte chunks per warp row
  static constexpr int DN_F4 = SLAB / 4;             // float4 per token of a slab
  static constexpr int DN_F4_PER_THREAD = (DN_F4 + kThreads - 1) / kThreads;
  // ---- up kernel: 16 columns x 4 streams = 64 rows per CTA
  static constexpr int UP_COLS = 16;
  static constexpr int UP_ROWS = UP_COLS * kStreams;
  static constexpr int UP_CTAS = D / UP_COLS;
  static constexpr int UP_PITCH = KD * 2 + 16;       // bytes; = 16 (mod 128)
  static constexpr int UP_KQ = KD / 4;               // K per quarter
  static constexpr int UP_CHUNKS = UP_KQ / 8;
  static constexpr int LO_PER_CTA = KD / UP_CTAS;    // lo entries each up CTA writes

  static_assert(SLAB % (8 * kWarps) == 0, "slab must split into 16-byte chunks per warp");
  static_assert(SLABS_PER_STREAM == 4, "cluster of four slabs per stream");
  static_assert(KD % DN_ROWS == 0, "K must be a multiple of 32");
  static_assert(DN_PITCH % 128 == 16 && UP_PITCH % 128 == 16, "pitch must be 16 mod 128");
  static_assert(D % UP_COLS == 0, "d must be a multiple of 16");
  static_assert(KD % UP_CTAS == 0, "lo must split evenly over the up CTAs");
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
  static constexpr int RS = SSW + kWarps * TT * 4;       // [kMaxT] rs (cluster leader)
  // Pushed by the cluster's four CTAs into the leader: [4][T] sums of squares,
  // then [4][T][32] partials.  Sized by the launch's T.
  static constexpr int RECV = RS + kMaxT * 4;
  static constexpr int bytes(int T) { return RECV + 4 * T * 4 + 4 * T * 32 * 4; }
  static constexpr int BYTES_MAX = RECV + 4 * kMaxT * 4 + 4 * kMaxT * 32 * 4;
};

template <int D, int KD, int TT, bool Q8 = false>
struct UpSmem {
  using G = Geo<D, KD>;
  static constexpr int BAR = 0;
  static constexpr int FLAG = 16;
  static constexpr int W = 128;
  // Q8_0: quant rows at a pitch of 16 (mod 32) bytes, so that eight lanes
  // reading 16-byte chunks of eight consecutive rows meet no bank twice;
  // then the rows' binary16 block scales, [64][K/32].
  static constexpr int WPITCH = Q8 ? KD + 16 : G::UP_PITCH;
  static constexpr int SCALE = W + G::UP_ROWS * WPITCH;
  static constexpr int GATE = SCALE + (Q8 ? G::UP_ROWS * (KD / 32) * 2 : 0);
  static constexpr int SIG = GATE + G::UP_ROWS * 4;
  static constexpr int LO = SIG + G::UP_ROWS * 4;
  static constexpr int RED = LO + TT * KD * 4;
  static constexpr int OUT = RED + 4 * TT * G::UP_ROWS * 4;
  static constexpr int RP = OUT + TT * G::UP_ROWS * 4;    // [TT][64] committed residual
  static constexpr int BYTES = RP + TT * G::UP_ROWS * 4;
  static constexpr int bytes(int) { return BYTES; }
  static constexpr int BYTES_MAX = BYTES;
};

struct DownArgs {
  const float* R;          // [T][N]
  const float* P;          // [T][N] or null
  const float* w_norm;     // [N]
  const uint16_t* W_down;  // [K][N] BF16 (BF16 kernels)
  const int8_t* Wq;        // [K][N] int8 quants (Q8_0 kernels)
  const uint16_t* Wscale;  // [K][N/32] binary16 block scales (Q8_0 kernels)
  float* part;             // scratch [4][T_max][K]: rs-scaled per-stream partials
  unsigned* err;           // scratch error word
  float* rs_out;           // [T][4] or null
  int T;
  int T_max;
  float eps;
  int independent;         // 1: no read in flight writes R or P (see below)
  int late_launch;         // 1: the read runs among others on the batch lanes (see hc_down_kernel)
  unsigned long long wait_ns;  // limit of the first bulk-copy wait from the kernel's start (0: kWaitNs)
  const void* W_tiles;         // W_down in tile order (hc_pack_down_tiles_kernel) or null: the BF16
                               // kernels of 32-row tiles then copy each tile as one contiguous block
  const void* W_tiles_sw;      // W_down in 64-row swizzled tile order (hc_pack_down_sw_kernel) or
                               // null: the tensor-memory kernels then copy each tile as one block
};

struct UpArgs {
  const float* R;        // [T][N]
  const float* P;        // [T][N] or null
  const float* gate;     // [N]
  const uint16_t* W_up;  // [N][K] BF16 (BF16 kernels)
  const int8_t* Wq;      // [N][K] int8 quants (Q8_0 kernels)
  const uint16_t* Wscale;  // [N][K/32] binary16 block scales (Q8_0 kernels)
  const float* part;     // scratch [4][T_max][K]
  float* out;            // [T][N]
  float* mean;           // [T][d]
  float* lo;             // [T][K]
  float* r_out;          // [T][N] or null
  unsigned* err;
  int T;
  int T_max;
  int independent;       // 1: no read in flight writes R or P (see below)
  const void* W_up_tiles;  // W_up in swizzled up-tile order (hc_pack_up_sw_kernel) or null (the
                           // wide tensor-memory up kernel then copies each tile as one block)
};

// R and P of one token group of this up CTA's rows (64 rows = 16 columns x
// 4 streams), `EPI` entries per thread.
template <int D, int EPI>
__device__ __forceinline__ void load_rp(const UpArgs& a, int c0, int t0, int tg, float (&rr)[EPI],
                                        float (&pp)[EPI]) {
  constexpr int ROWS = 4 * 16;
#pragma unroll
  for (int m = 0; m < EPI; ++m) {
    const int idx = threadIdx.x + m * 256;
    const int t = idx / ROWS, r = idx % ROWS;
    rr[m] = 0.f;
    pp[m] = 0.f;
    if (t < tg) {
      const size_t off = (size_t)(t0 + t) * (4 * D) + (r / 16) * D + c0 + (r % 16);
      rr[m] = __ldcg(a.R + off);
      if (a.P) pp[m] = __ldcg(a.P + off);
    }
  }
}

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

// Sixteen int8 quants (one 16-byte chunk) as fp32.  Each byte b, biased to
// b + 128 by flipping its top bit, is placed in the mantissa of 2^23, which
// makes the float 2^23 + 128 + b; taking away 2^23 + 128 leaves b exactly.
__device__ __forceinline__ void q8x16_to_f32(const uint4 v, float* w) {
  const unsigned words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned u = words[k] ^ 0x80808080u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float f = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u + i));
      w[4 * k + i] = __fsub_rn(f, 8388736.0f);
    }
  }
}

// Every thread waits for the barrier's phase `parity` itself (observing the
// completed phase makes the bulk-copied bytes visible to that thread).  The
// wait is bounded: after kWaitNs the thread records `code` in *err and
// returns false; the kernel then carries on with whatever is in shared
// memory (its results are void and the error word says so) and drains the
// copies before it exits, so no CTA leaves with copies still in flight.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, unsigned* err,
                                         unsigned code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitNs) {
      atomicOr(err, code);
      return false;
    }
  }
  return true;
}

// The first bulk-copy wait of a down kernel: gives up once `limit` ns have
// passed since `t0` (the kernel's start), checked before every probe, so a
// limit shorter than the kernel's start-up gives up whether or not the copy
// has landed (the timeout path of a read can be exercised on purpose: see
// hc_read_set_wait_limit).  The copy itself still lands and is drained.
__device__ __forceinline__ bool wait_bar_from(uint64_t* bar, uint32_t parity, unsigned* err, unsigned code,
                                              uint64_t t0, uint64_t limit) {
  for (;;) {
    if (ptx::globaltimer_ns() - t0 >= limit) {
      atomicOr(err, code);
      return false;
    }
    if (ptx::mbar_try_wait(bar, parity)) return true;
  }
}
__device__ __forceinline__ uint64_t first_wait_limit(unsigned long long wait_ns) {
  return wait_ns != 0ull && wait_ns < kWaitNs ? wait_ns : kWaitNs;
}

// Before a CTA whose wait timed out exits: wait (bounded again) for copies
// still in flight into its shared memory.
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < kWaitNs) {
  }
}

// ---- W_down in tile order.  A down CTA's tile (rows 32 rg .. 32 rg + 31,
// columns SLAB slab .. + SLAB - 1) held as one contiguous block of DN_ROWS
// rows at the shared-memory pitch DN_PITCH (the last 16 bytes of a row are
// padding), tiles in the order (rg, slab).  A CTA then copies its 40 KB as
// kTileCopies pieces of contiguous memory instead of 32 row segments 2N bytes
// apart, which HBM serves faster (measured at d = 2560 in a cold batch: about
// 8 % less time per read at T = 2..4).  The values are the same, and so is
// every bit of every result.
constexpr int kTileCopies = 4;

template <class G>
__device__ __forceinline__ void copy_down_tile(unsigned char* w_s, const void* tiles, int rg, int slab, int piece,
                                               uint64_t* bar, uint64_t policy) {
  constexpr int PIECE = G::DN_ROWS / kTileCopies * G::DN_PITCH;
  static_assert(G::DN_ROWS % kTileCopies == 0 && PIECE % 16 == 0, "whole 16-byte pieces of whole rows");
  const unsigned char* tile =
      static_cast<const unsigned char*>(tiles) + ((size_t)rg * G::SLABS + slab) * (G::DN_ROWS * G::DN_PITCH);
  ptx::bulk_g2s(w_s + piece * PIECE, tile + piece * PIECE, PIECE, bar, policy);
}

// Writes W_down [K][N] in tile order: one CTA per tile, 16-byte words, the
// padding of each row zero.
template <int D, int KD>
__global__ void __launch_bounds__(kThreads) hc_pack_down_tiles_kernel(const uint16_t* __restrict__ W,
                                                                     uint16_t* __restrict__ tiles) {
  using G = Geo<D, KD>;
  constexpr int W16 = G::DN_PITCH / 16;  // 16-byte words of a tile row
  constexpr int DATA16 = G::SLAB * 2 / 16;
  const int slab = blockIdx.x, rg = blockIdx.y;
  uint4* dst = reinterpret_cast<uint4*>(tiles) + ((size_t)rg * G::SLABS + slab) * G::DN_ROWS * W16;
  for (int i = threadIdx.x; i < G::DN_ROWS * W16; i += kThreads) {
    const int r = i / W16, w = i - r * W16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (w < DATA16) {
      v = __ldg(reinterpret_cast<const uint4*>(W + (size_t)(rg * G::DN_ROWS + r) * G::N + slab * G::SLAB) + w);
    }
    dst[i] = v;
  }
}

// Sums V values over the 32 lanes of a warp (V a power of two, at most 32)
// in V - 1 + 5 - log2(V) shuffles rather than 5 V: at each butterfly step
// a lane keeps half of its values, sends the other half to its partner and
// adds what the partner sent.  Afterwards v[0] of lane l holds the warp's sum
// of value l >> (5 - log2 V) (lanes that share it hold the same sum).
template <int V>
__device__ __forceinline__ void warp_sum_transposed(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two up to 32");
  int n = V;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (n > 1) {
      const int half = n / 2;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < V / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
}

// ------------------------------------------------------------------ kernel 1, T = 1 (d = 2560; Q8_0 also T = 2)
// One CTA per 8 rows of W_down and one stream, over all the stream's D
// columns: the stream's sum of squares, its rs and the rows' partial sums
// are complete in the CTA, so there is no cluster and no exchange, and the
// weight tile is 8 row segments of 2D bytes (Q8: D bytes of quants and D/16
// of block scales).  CUDA cores, fp32 (80 multiply-adds a thread and token;
// a Q8_0 weight is scale * q, exact in fp32).  TT: tokens held in registers
// (T <= TT).  Writes the same rs-scaled per-stream partials as the other down
// kernels.
template <int D, int KD, bool Q8 = false, int TT = 1>
struct StreamGeo {
  static constexpr int ROWS = 8;                   // rows of W_down per CTA
  static constexpr int ROW_GROUPS = KD / ROWS;
  static constexpr int N = kStreams * D;
  static constexpr int PAIRS = D / (2 * kThreads);  // column pairs per thread
  static constexpr int ROW_BYTES = Q8 ? D : D * 2;  // a weight row (quants for Q8)
  static constexpr int SC_BYTES = Q8 ? D / 32 * 2 : 0;  // a row's binary16 block scales
  static constexpr int W_BYTES = ROWS * ROW_BYTES;
  static constexpr int BAR = 0;                    // bar_w, bar_n
  static constexpr int WN = 128;                   // w_norm of the stream [D]
  static constexpr int W = WN + D * 4;             // [ROWS][D] bf16 (int8 for Q8)
  static constexpr int SC = W + W_BYTES;           // [ROWS][D/32] binary16 (Q8)
  static constexpr int RED = SC + ROWS * SC_BYTES;  // [kWarps][(ROWS + 1) TT]: row sums, then sums of squares
  static constexpr int BYTES = RED + kWarps * (ROWS + 1) * TT * 4;
  static_assert(D % (2 * kThreads) == 0 && KD % ROWS == 0 && ROWS * TT <= 32, "whole column pairs and row groups");
  static_assert((TT & (TT - 1)) == 0, "tokens a pass: a power of two");
  static_assert(ROW_BYTES % 16 == 0 && SC_BYTES % 16 == 0 && W % 16 == 0 && SC % 16 == 0, "16-byte bulk copies");
};

// Two tokens are held to 48 registers, five CTAs per SM (a 16-byte spill):
// a cold batch of Q8_0 T = 2 reads ran 2.53 us per read at 63 registers
// (four CTAs), 2.42 at 48.  One token needs no bound: 40 (BF16) and 47
// (Q8_0) registers, and the BF16 tile's 51 KB of shared memory allows four.
template <int D, int KD, bool Q8 = false, int TT = 1>
__global__ void __launch_bounds__(kThreads, TT == 1 ? 4 : 5) hc_down_s_kernel(const DownArgs a) {
  using G = StreamGeo<D, KD, Q8, TT>;
  constexpr int V = G::ROWS * TT;  // row sums a thread holds: [ROWS][TT]
  constexpr int RS = V + TT;       // a warp's scratch: V row sums, then TT sums of squares
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + G::BAR);
  uint64_t* bar_n = bar_w + 1;
  const float* wn_s = reinterpret_cast<const float*>(smem + G::WN);
  const unsigned char* w_s = smem + G::W;
  float* red = reinterpret_cast<float*>(smem + G::RED);
  const int rg = blockIdx.x, stream = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = rg * G::ROWS, col0 = stream * D;
  const int T = a.T;
  const uint64_t t_entry = ptx::globaltimer_ns();

  // w_norm of the stream and the 8 weight rows: parameters, issued first.
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::mbar_init(bar_n, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_n, D * 4);
      ptx::mbar_arrive_expect_tx(bar_w, G::W_BYTES + G::ROWS * G::SC_BYTES);
      ptx::bulk_g2s(smem + G::WN, a.w_norm + col0, D * 4, bar_n, ptx::policy_evict_last());
    }
    __syncwarp();
    if (lane < G::ROWS) {
      const uint64_t once = ptx::policy_evict_first();
      if constexpr (Q8) {
        ptx::bulk_g2s(smem + G::W + lane * G::ROW_BYTES, a.Wq + (size_t)(row0 + lane) * G::N + col0, G::ROW_BYTES,
                      bar_w, once);
        ptx::bulk_g2s(smem + G::SC + lane * G::SC_BYTES, a.Wscale + (size_t)(row0 + lane) * (G::N / 32) + col0 / 32,
                      G::SC_BYTES, bar_w, once);
      } else {
        ptx::bulk_g2s(smem + G::W + lane * (D * 2), a.W_down + (size_t)(row0 + lane) * G::N + col0, D * 2, bar_w,
                      once);
      }
    }
  }
  // Late launch of the up kernel on the batch lanes, as in hc_down_kernel.
  const bool late_launch = a.late_launch && a.independent;
  if (!late_launch) ptx::launch_dependents();
  __syncthreads();  // the mbarriers are initialised before any thread waits on them
  if (!a.independent) ptx::wait_prerequisites();

  // This thread's columns: pairs 2 tid + 2 kThreads k (coalesced float2 and
  // BF16 pair loads).  R' = R + P, x = R' * w_norm, and R'^2 summed, per
  // token (tokens past T are zero).
  float2 rv[TT][G::PAIRS], pv[TT][G::PAIRS];
#pragma unroll
  for (int t = 0; t < TT; ++t) {
#pragma unroll
    for (int k = 0; k < G::PAIRS; ++k) {
      const int c = 2 * tid + 2 * kThreads * k;
      rv[t][k] = pv[t][k] = make_float2(0.f, 0.f);
      if (t < T) {
        const size_t off = (size_t)t * G::N + col0 + c;
        rv[t][k] = __ldcg(reinterpret_cast<const float2*>(a.R + off));
        if (a.P) pv[t][k] = __ldcg(reinterpret_cast<const float2*>(a.P + off));
      }
    }
  }
  bool ok = wait_bar_from(bar_n, 0, a.err, kErrDownNorm, t_entry, first_wait_limit(a.wait_ns));
  float x[TT][2 * G::PAIRS];
  float ss[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    ss[t] = 0.f;
#pragma unroll
    for (int k = 0; k < G::PAIRS; ++k) {
      const int c = 2 * tid + 2 * kThreads * k;
      const float r0 = __fadd_rn(rv[t][k].x, pv[t][k].x), r1 = __fadd_rn(rv[t][k].y, pv[t][k].y);
      x[t][2 * k] = __fmul_rn(r0, wn_s[c]);
      x[t][2 * k + 1] = __fmul_rn(r1, wn_s[c + 1]);
      ss[t] = __fmaf_rn(r0, r0, ss[t]);
      ss[t] = __fmaf_rn(r1, r1, ss[t]);
    }
  }
  // Lane l ends with the warp's sum of squares of token l >> (5 - log2 TT).
  warp_sum_transposed<TT>(ss, lane);
  if ((lane & (32 / TT - 1)) == 0) red[warp * RS + V + lane / (32 / TT)] = ss[0];

  ok = wait_bar(bar_w, 0, a.err, kErrDownWeights) && ok;
  if (late_launch) ptx::launch_dependents();
  float acc[V];  // [row][token]
#pragma unroll
  for (int r = 0; r < G::ROWS; ++r) {
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[r * TT + t] = 0.f;
#pragma unroll
    for (int k = 0; k < G::PAIRS; ++k) {
      const int c = 2 * tid + 2 * kThreads * k;
      float w0, w1;
      if constexpr (Q8) {
        // Both columns in the block c / 32: scale * q, exact in fp32, with no
        // integer-to-float conversion: each byte b, biased to b + 128 by
        // flipping its top bit, is placed in the mantissa of 2^23 (the float
        // 2^23 + 128 + b), and subtracting 2^23 + 128 leaves b exactly.  The
        // conversion instruction took more registers (64 against 47 at T = 1,
        // 86 against 63 at T = 2) and fewer CTAs per SM: at T = 2, 3.11 ->
        // 2.90 us per read in a cold batch; at T = 1, with the up kernel at
        // five CTAs per SM, 2.07 -> 2.03 (and 4.9 -> 4.8 read after read).
        const float sc = __half2float(reinterpret_cast<const __half*>(smem + G::SC + r * G::SC_BYTES)[c / 32]);
        const unsigned u = *reinterpret_cast<const unsigned short*>(w_s + r * G::ROW_BYTES + c) ^ 0x8080u;
        w0 = __fmul_rn(sc, __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u)), 8388736.0f));
        w1 = __fmul_rn(sc, __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541u)), 8388736.0f));
      } else {
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(w_s + r * (D * 2) + c * 2);
        w0 = __uint_as_float(w2 << 16);
        w1 = __uint_as_float(w2 & 0xffff0000u);
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        acc[r * TT + t] = __fmaf_rn(w0, x[t][2 * k], acc[r * TT + t]);
        acc[r * TT + t] = __fmaf_rn(w1, x[t][2 * k + 1], acc[r * TT + t]);
      }
    }
  }
  // The warp's [row][token] sums, transposed: lane l ends with entry
  // l >> (5 - log2 V) (T = 1: 9 shuffles, lane 4 r holds row r).
  warp_sum_transposed<V>(acc, lane);
  if ((lane & (32 / V - 1)) == 0) red[warp * RS + lane / (32 / V)] = acc[0];
  __syncthreads();
  if (tid < V) {
    const int r = tid / TT, t = tid % TT;
    float sq = 0.f, p = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      sq += red[w * RS + V + t];
      p += red[w * RS + tid];
    }
    if (t < T) {
      const float rs = rsqrtf(sq * (1.0f / (float)D) + a.eps);
      __stcg(a.part + ((size_t)stream * a.T_max + t) * KD + row0 + r, __fmul_rn(rs, p));
      if (rg == 0 && r == 0 && a.rs_out != nullptr) a.rs_out[t * kStreams + stream] = rs;
    }
  }
  if (tid == 0 && !ok) {
    drain(bar_n, 0);
    drain(bar_w, 0);
  }
  if (a.independent) ptx::wait_prerequisites();  // complete only after the previous read
}

// ------------------------------------------------------------------ kernel 1
// Grid (16 slabs, K/32 row groups), clusters of 4 along x (one stream).
// TILES: the weight tile comes from a.W_tiles (a compile-time choice, so the
// row-segment copies of the plain layout carry no extra test).
template <int D, int KD, int TT, bool TILES = false>
__global__ void __launch_bounds__(kThreads, D == 2560 ? 3 : 2) hc_down_kernel(const DownArgs a) {
  using G = Geo<D, KD>;
  using S = DownSmem<D, KD, TT>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + S::BAR);
  uint64_t* bar_n = bar_w + 1;
  unsigned char* w_s = smem + S::W;
  const float* wn_s = reinterpret_cast<const float*>(smem + S::WN);
  float* x_s = reinterpret_cast<float*>(smem + S::X);
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

  const uint64_t t_entry = ptx::globaltimer_ns();
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();  // = slab within the stream
  // The leader's receive area: [4][T] sums of squares, then [4][T][32] partials.
  float* recv_ss = cluster.map_shared_rank(reinterpret_cast<float*>(smem + S::RECV), 0);
  float* recv_p = recv_ss + 4 * T;

  // Announce this CTA to its cluster; the matching wait below guarantees that
  // every CTA of the cluster runs before anyone writes the leader's memory.
  ptx::cluster_arrive_relaxed();

  // Weights first (w_norm, needed earliest, before the W_down rows); they do
  // not depend on the previous kernel.  Then let the next kernel launch.
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::mbar_init(bar_n, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_n, G::SLAB * 4);
      ptx::mbar_arrive_expect_tx(bar_w, TILES ? G::DN_ROWS * G::DN_PITCH : G::DN_ROWS * G::SLAB * 2);
      // w_norm's slab is read by every row group: keep it in L2.
      ptx::bulk_g2s(smem + S::WN, a.w_norm + col0, G::SLAB * 4, bar_n, ptx::policy_evict_last());
    }
    __syncwarp();
    const uint64_t once = ptx::policy_evict_first();  // each weight byte is read once
    if constexpr (!TILES) {
      ptx::bulk_g2s(w_s + lane * G::DN_PITCH, a.W_down + (size_t)(row0 + lane) * G::N + col0,
                    G::SLAB * 2, bar_w, once);
    } else if (lane < kTileCopies) {
      copy_down_tile<G>(w_s, a.W_tiles, rg, slab, lane, bar_w, once);
    }
  }
  // An independent read of one token group that runs among others on the
  // batch lanes lets its up kernel launch only at the end of this kernel:
  // the up CTAs then hold SM slots for less time and more reads of the batch
  // overlap (six streams: 2.58 -> 2.53-2.56 us per read at T = 1, 2.70 ->
  // 2.64-2.67 at T = 4).  A read on its own keeps the early launch, which
  // streams the up kernel's weights while this kernel runs (one read after
  // another on one stream: 5.16 us per read at T = 1, 6.10 with a late
  // launch; 96 chained calls: 5.9 against 7.3).  Reads of two token groups
  // measured slower with it.
  const bool late_launch = a.late_launch && a.independent && a.T <= TT;
  if (!late_launch) ptx::launch_dependents();
  __syncthreads();  // the mbarriers are initialised before any thread waits on them
  // w_norm is a parameter: wait for it before the previous kernel finishes.
  bool ok = true;
  // R, P and the scratch slot belong to the previous kernel until its end
  // (in independent mode only the previous read's outputs do, and the down
  // kernel waits at its end instead).
  if (!a.independent) ptx::wait_prerequisites();
  ptx::cluster_wait();

  // A timed-out wait leaves garbage in shared memory but the CTA still runs
  // to the end: it must take part in the cluster barrier below.
  for (int t0 = 0; t0 < T; t0 += TT) {
    const int tg = min(TT, T - t0);

    // Issue every R and P load of the group, then commit the pending write,
    // stage x = R' * w_norm and sum R'^2 over this slab.
    float4 rv[TT][G::DN_F4_PER_THREAD];
    float4 pv[TT][G::DN_F4_PER_THREAD];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
#pragma unroll
      for (int m = 0; m < G::DN_F4_PER_THREAD; ++m) {
        const int c4 = tid + m * kThreads;
        rv[t][m] = make_float4(0.f, 0.f, 0.f, 0.f);
        pv[t][m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < tg && c4 < G::DN_F4) {
          const size_t base = (size_t)(t0 + t) * G::N + col0;
          rv[t][m] = __ldcg(reinterpret_cast<const float4*>(a.R + base) + c4);
          if (a.P) pv[t][m] = __ldcg(reinterpret_cast<const float4*>(a.P + base) + c4);
        }
      }
    }
    // w_norm is waited for only now, with this group's R and P loads in flight.
    if (t0 == 0) ok = wait_bar_from(bar_n, 0, a.err, kErrDownNorm, t_entry, first_wait_limit(a.wait_ns)) && ok;
    float ssl[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      ssl[t] = 0.f;
#pragma unroll
      for (int m = 0; m < G::DN_F4_PER_THREAD; ++m) {
        const int c4 = tid + m * kThreads;
        if (t < tg && c4 < G::DN_F4) {
          float4 r = rv[t][m];
          const float4 p = pv[t][m];
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
    if (t0 == 0) ok = wait_bar(bar_w, 0, a.err, kErrDownWeights) && ok;
    __syncthreads();  // x and the per-warp sums of squares are complete
    if (tid < tg) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += ssw_s[w * TT + tid];
      recv_ss[rank * T + t0 + tid] = v;  // into the leader's shared memory
    }

    // Partial dot products: lane = row, warp = column range of the slab.
    // Two accumulation chains per token (elements 0-3 and 4-7 of each chunk),
    // added at the end: a fixed order with half the dependent-FMA latency.
    const unsigned char* wrow = w_s + lane * G::DN_PITCH + warp * G::DN_CPW * 2;
    const float* xw = x_s + warp * G::DN_CPW;
    float acc0[TT], acc1[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc0[t] = acc1[t] = 0.f;
#pragma unroll 2
    for (int j = 0; j < G::DN_CHUNKS; ++j) {
      float w[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(wrow + j * 16), w);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float4 xa = *reinterpret_cast<const float4*>(xw + t * G::SLAB + j * 8);
        const float4 xb = *reinterpret_cast<const float4*>(xw + t * G::SLAB + j * 8 + 4);
        float v0 = acc0[t], v1 = acc1[t];
        v0 = __fmaf_rn(w[0], xa.x, v0);
        v1 = __fmaf_rn(w[4], xb.x, v1);
        v0 = __fmaf_rn(w[1], xa.y, v0);
        v1 = __fmaf_rn(w[5], xb.y, v1);
        v0 = __fmaf_rn(w[2], xa.z, v0);
        v1 = __fmaf_rn(w[6], xb.z, v1);
        v0 = __fmaf_rn(w[3], xa.w, v0);
        v1 = __fmaf_rn(w[7], xb.w, v1);
        acc0[t] = v0;
        acc1[t] = v1;
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) red_s[(warp * TT + t) * 32 + lane] = __fadd_rn(acc0[t], acc1[t]);
    __syncthreads();
    for (int idx = tid; idx < tg * 32; idx += kThreads) {
      const int t = idx >> 5, r = idx & 31;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += red_s[(w * TT + t) * 32 + r];
      recv_p[(rank * T + t0 + t) * 32 + r] = v;  // into the leader's shared memory
    }
    __syncthreads();
  }

  if (!ok) {
    drain(bar_n, 0);
    drain(bar_w, 0);
  }
  if (late_launch) ptx::launch_dependents();
  // One cluster barrier: every slab's pushes are visible to the leader.
  ptx::cluster_arrive_release();
  ptx::cluster_wait();
  if (rank != 0) {
    if (a.independent) ptx::wait_prerequisites();
    return;
  }

  // Leader: sum the four slabs in slab order, apply rs, write the partial.
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

// One 8-column chunk of the up product: w[0..3] and w[4..7] feed two
// accumulators per token, columns in order.
template <int KD, int TT>
__device__ __forceinline__ void up_chunk(const float* w, const float* lw, float (&acc0)[TT],
                                         float (&acc1)[TT]) {
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const float4 la = *reinterpret_cast<const float4*>(lw + t * KD);
    const float4 lb = *reinterpret_cast<const float4*>(lw + t * KD + 4);
    float v0 = acc0[t], v1 = acc1[t];
    v0 = __fmaf_rn(w[0], la.x, v0);
    v1 = __fmaf_rn(w[4], lb.x, v1);
    v0 = __fmaf_rn(w[1], la.y, v0);
    v1 = __fmaf_rn(w[5], lb.y, v1);
    v0 = __fmaf_rn(w[2], la.z, v0);
    v1 = __fmaf_rn(w[6], lb.z, v1);
    v0 = __fmaf_rn(w[3], la.w, v0);
    v1 = __fmaf_rn(w[7], lb.w, v1);
    acc0[t] = v0;
    acc1[t] = v1;
  }
}

// ------------------------------------------------------------------ kernel 2
//
// Q8 = true (Q8_0 projections): the quant rows and their block scales are
// copied instead; each 16-quant chunk (inside one 32-weight block) is decoded
// to fp32 in the loop, its products with lo are summed as a BF16 chunk's
// would be, and the two sums are added to the accumulators times the block's
// scale.
//
// At d = 2560 held to 48 registers, five CTAs per SM (the BF16 tile's 45 KB
// of shared memory allows five, the Q8_0 tile's 26 KB six): more CTAs per
// SM keep more weight tiles in flight.  Cold batches of T = 1 reads: BF16
// 2.28-2.38 -> 2.01-2.03 us per read (60 -> 48 registers); Q8_0 2.53 us at
// 72 registers, 2.18 at 64, 2.07 at 48.
template <int D, int KD, int TT, bool Q8 = false>
__global__ void __launch_bounds__(kThreads, D == 2560 ? 5 : 2) hc_up_kernel(const UpArgs a) {
  using G = Geo<D, KD>;
  using S = UpSmem<D, KD, TT, Q8>;
  static_assert(!Q8 || G::UP_KQ % 16 == 0, "a K quarter must split into 16-quant chunks");
  constexpr int EPI = (TT * G::UP_ROWS + kThreads - 1) / kThreads;  // epilogue items per thread
  constexpr int LO4 = (TT * KD / 4 + kThreads - 1) / kThreads;       // lo float4 per thread
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(smem + S::BAR);
  uint64_t* bar_g = bar_w + 1;
  unsigned char* w_s = smem + S::W;
  const float* g_s = reinterpret_cast<const float*>(smem + S::GATE);
  float* sig_s = reinterpret_cast<float*>(smem + S::SIG);
  float* lo_s = reinterpret_cast<float*>(smem + S::LO);
  float* red_s = reinterpret_cast<float*>(smem + S::RED);
  float* out_s = reinterpret_cast<float*>(smem + S::OUT);
  float* rp_s = reinterpret_cast<float*>(smem + S::RP);

  const int c0 = blockIdx.x * G::UP_COLS;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::mbar_init(bar_g, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_w, Q8 ? G::UP_ROWS * KD + G::UP_ROWS * (KD / 32) * 2 : G::UP_ROWS * KD * 2);
      ptx::mbar_arrive_expect_tx(bar_g, G::UP_ROWS * 4);
    }
    __syncwarp();
    const uint64_t once = ptx::policy_evict_first();
    if (lane < kStreams) {
      ptx::bulk_g2s(smem + S::GATE + lane * G::UP_COLS * 4, a.gate + lane * D + c0,
                    G::UP_COLS * 4, bar_g, once);
    }
    // Local row r = s * 16 + j holds global row s * d + c0 + j.
    for (int r = lane; r < G::UP_ROWS; r += 32) {
      const int grow = (r / G::UP_COLS) * D + c0 + (r % G::UP_COLS);
      if constexpr (Q8) {
        ptx::bulk_g2s(w_s + r * S::WPITCH, a.Wq + (size_t)grow * KD, KD, bar_w, once);
      } else {
        ptx::bulk_g2s(w_s + r * G::UP_PITCH, a.W_up + (size_t)grow * KD, KD * 2, bar_w, once);
      }
    }
    if constexpr (Q8) {
      // The 16 rows of one stream are consecutive rows of the scales: one run.
      constexpr int RUN = G::UP_COLS * (KD / 32) * 2;
      static_assert(RUN % 16 == 0, "scale runs must be whole 16-byte pieces");
      if (lane < kStreams) {
        ptx::bulk_g2s(smem + S::SCALE + lane * RUN, a.Wscale + (size_t)(lane * D + c0) * (KD / 32), RUN,
                      bar_w, once);
      }
    }
  }
  __syncthreads();  // the mbarriers are initialised before any thread waits on them
  // The gates are parameters: their sigmoids are ready before the previous
  // kernel finishes.
  bool ok = true;
  if (tid < G::UP_ROWS) {
    ok = wait_bar(bar_g, 0, a.err, kErrUpGate);
    sig_s[tid] = 1.0f / (1.0f + expf(-g_s[tid]));
  }
  // Independent mode: R and P of the first token group do not depend on the
  // previous read; fetch them before waiting.
  float rr0[EPI], pp0[EPI];
  if (a.independent) load_rp<D, EPI>(a, c0, 0, min(TT, a.T), rr0, pp0);
  ptx::wait_prerequisites();  // the partials, R and P are ready from here on
  // Only now may the next read's kernels launch: launching them earlier lets
  // a cascade of waiting CTAs crowd the SMs that are computing this read.
  ptx::launch_dependents();

  const int T = a.T;
  for (int t0 = 0; t0 < T; t0 += TT) {
    const int tg = min(TT, T - t0);
    // Issue every global load of the group before using any: the four
    // per-stream partials of lo, and R and P of this CTA's rows.
    float4 pv[LO4][kStreams];
#pragma unroll
    for (int m = 0; m < LO4; ++m) {
      const int idx = tid + m * kThreads;
#pragma unroll
      for (int s = 0; s < kStreams; ++s) {
        pv[m][s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < tg * KD / 4) {
          pv[m][s] = __ldcg(reinterpret_cast<const float4*>(
                                a.part + ((size_t)s * a.T_max + t0) * KD) + idx);
        }
      }
    }
    float rr[EPI], pp[EPI];
    if (t0 == 0 && a.independent) {
#pragma unroll
      for (int m = 0; m < EPI; ++m) {
        rr[m] = rr0[m];
        pp[m] = pp0[m];
      }
    } else {
      load_rp<D, EPI>(a, c0, t0, tg, rr, pp);
    }
    // lo: the four per-stream partials summed in stream order.
#pragma unroll
    for (int m = 0; m < LO4; ++m) {
      const int idx = tid + m * kThreads;
      if (idx < tg * KD / 4) {
        float4 l;
        l.x = ((pv[m][0].x + pv[m][1].x) + pv[m][2].x) + pv[m][3].x;
        l.y = ((pv[m][0].y + pv[m][1].y) + pv[m][2].y) + pv[m][3].y;
        l.z = ((pv[m][0].z + pv[m][1].z) + pv[m][2].z) + pv[m][3].z;
        l.w = ((pv[m][0].w + pv[m][1].w) + pv[m][2].w) + pv[m][3].w;
        reinterpret_cast<float4*>(lo_s)[idx] = l;
      }
    }
#pragma unroll
    for (int m = 0; m < EPI; ++m) {
      const int idx = tid + m * kThreads;
      if (idx < tg * G::UP_ROWS) rp_s[idx] = __fadd_rn(rr[m], pp[m]);
    }
    if (t0 == 0) ok = wait_bar(bar_w, 0, a.err, kErrUpWeights) && ok;
    __syncthreads();  // lo, R' and the gates are in shared memory
    // This CTA's share of the lo output.
    for (int idx = tid; idx < tg * G::LO_PER_CTA; idx += kThreads) {
      const int t = idx / G::LO_PER_CTA, k = blockIdx.x * G::LO_PER_CTA + idx % G::LO_PER_CTA;
      a.lo[(size_t)(t0 + t) * KD + k] = lo_s[t * KD + k];
    }

    // u for 64 rows: lane = row within a half, warp = (half, K quarter).
    const int half = warp & 1;
    const int kq = warp >> 1;
    const int row = half * 32 + lane;
    const float* lw = lo_s + kq * G::UP_KQ;
    float acc0[TT], acc1[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc0[t] = acc1[t] = 0.f;
    if constexpr (Q8) {
      const unsigned char* qrow = w_s + row * S::WPITCH + kq * G::UP_KQ;
      const __half* srow = reinterpret_cast<const __half*>(smem + S::SCALE) + row * (KD / 32);
#pragma unroll
      for (int j = 0; j < G::UP_KQ / 16; ++j) {
        float w[16], b0[TT], b1[TT];
        q8x16_to_f32(*reinterpret_cast<const uint4*>(qrow + j * 16), w);
#pragma unroll
        for (int t = 0; t < TT; ++t) b0[t] = b1[t] = 0.f;
        up_chunk<KD, TT>(w, lw + j * 16, b0, b1);
        up_chunk<KD, TT>(w + 8, lw + j * 16 + 8, b0, b1);
        const float sc = __half2float(srow[(kq * G::UP_KQ + j * 16) / 32]);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          acc0[t] = __fmaf_rn(sc, b0[t], acc0[t]);
          acc1[t] = __fmaf_rn(sc, b1[t], acc1[t]);
        }
      }
    } else {
      const unsigned char* wrow = w_s + row * G::UP_PITCH + kq * G::UP_KQ * 2;
#pragma unroll 2
      for (int j = 0; j < G::UP_CHUNKS; ++j) {
        float w[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(wrow + j * 16), w);
        up_chunk<KD, TT>(w, lw + j * 8, acc0, acc1);
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      red_s[(kq * TT + t) * G::UP_ROWS + row] = __fadd_rn(acc0[t], acc1[t]);
    }
    __syncthreads();

    // Epilogue: pending write, gate, stream mean.
    for (int idx = tid; idx < tg * G::UP_ROWS; idx += kThreads) {
      const int t = idx / G::UP_ROWS, r = idx % G::UP_ROWS;
      const float u = ((red_s[(0 * TT + t) * G::UP_ROWS + r] + red_s[(1 * TT + t) * G::UP_ROWS + r]) +
                       red_s[(2 * TT + t) * G::UP_ROWS + r]) +
                      red_s[(3 * TT + t) * G::UP_ROWS + r];
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
