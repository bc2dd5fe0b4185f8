// Persistent multi-read kernel: a list of reads (a verify window, or a sweep of
// independent reads) in one launch.
//
// Why: the two-kernel read pays, per read, two kernel boundaries and two
// round trips through L2 on its dependent chain (about 5 us at d = 2560 on
// GB300), while its 13.1 MB of weights stream in under 2 us.  Here 128 CTAs
// (one per SM, four-CTA thread-block clusters) stay resident for the whole
// list; each CTA owns one column slab of one stream (W = d/32 columns) for
// both projections, so a chained read's output never leaves the chip before
// the next read's down projection consumes it, and the only cross-CTA step per
// read is the reduction of the down projection's partial sums:
//
//   * producer warps stream the weight tiles of the next reads (16-byte
//     cp.async into XOR-swizzled shared memory, L2 evict-first) into a
//     two-entry ring while the compute warps work on the current read;
//   * down projection (tensor cores, two-term BF16 split of x as in the
//     two-kernel path) -> per-CTA partial sums [T][K];
//   * cluster reduce-scatter over distributed shared memory (st.async with
//     mbarrier transaction counts): rank r of the cluster receives the four
//     CTAs' partials for k in its quarter of K and sums them;
//   * global exchange through L2 with self-tagged words: the three low
//     mantissa bits of every exchanged fp32 value carry the read's epoch
//     modulo 8 (a relative change below 2^-20), so a reader polls the data
//     itself, 16 bytes at a time, and needs no separate flag, fence or second
//     round trip.  Words are written by 8-byte strong stores, which are
//     single-copy atomic, so a word is either old or new, never torn.  Rank r
//     of every cluster reads its quarter of K from all 32 clusters, sums the 8
//     clusters of each stream, forms rs per stream from the exchanged sums of
//     squares and lo = sum_s rs_s * S_s;
//   * cluster all-gather of lo (split into BF16 hi/lo terms) over distributed
//     shared memory, then the up projection (one warp per 16 rows of W_up
//     over the whole K) on tensor cores, with the epilogue taken straight
//     from the accumulators;
//   * the stream mean needs the four streams of a column, which live in four
//     clusters: each CTA publishes its output tile as tagged words and
//     computes the mean of its quarter of the columns one read later; those
//     loads are issued with the next read's exchange loads and are long
//     written by then.
//
// Tag safety: exchange buffers have four slots (epoch mod 4), and every read
// rewrites all 8 token rows of its slot whatever T is (rows of tokens >= T
// carry zeros), so a stale word is from epoch - 4 at the oldest, which carries
// another tag; all CTAs are within one read of each other.  Buffers start
// zeroed and epochs at 1, so the first use of each slot (epochs 1..4) cannot
// match a zero tag.  hc_read_reset zeroes the buffers and the epoch bases
// again.
//
// Every sum runs in a fixed order, so repeated launches and graph replays give
// identical bits.  All waits are bounded.  Two kinds:
//   * waits across clusters (the global exchange, the stream-mean tiles)
//     depend on CTAs that the hardware does not co-schedule with this one;
//     they give up after kWaitNs, or at once when any CTA has raised the
//     launch's abort word, and from then on this CTA skips them (its results
//     are void and the error word says so);
//   * waits inside the CTA or its cluster (the weight ring, the cluster
//     exchanges) depend only on this CTA's own copies and on its cluster
//     peers, which run at the same time and never skip a send.  They ignore
//     the abort word, so every byte a peer sends is waited for by its
//     receiver, every transaction count returns to zero, and no CTA leaves
//     while a copy or a peer's store into it is in flight.  Their limit
//     (kLocalWaitNs) is longer than the global one: a peer stuck in a global
//     wait gives up first.
// The kernel checks its launch shape (grid, block and 4-CTA clusters) before
// it touches a peer, and records kErrWinLaunch instead of running when the
// shape is wrong.  The 128 CTAs must be co-resident (the host launches
// cooperatively); if they are not, the global waits give up and the launch
// reports HC_ERR_TIMEOUT.
//
// Design ancestors: the down and up kernels of "#2812 sycl: STRATA_GR_FUSED=1,
// the two-kernel BF16 hyper-connection read (opt-in)", section "What changed"
// (unscaled R'*w_norm staging with sums of squares, rs applied per stream to
// the partial sums, the epilogue's pending write, gate and stream mean).
#pragma once

#include <cuda_bf16.h>

#include "hc_kernels_tc.cuh"

namespace hc {

constexpr int kWinMaxReads = 224;  // reads per launch (kernel parameter space)
constexpr int kWinCtas = 128;
constexpr int kWinCluster = 4;
constexpr int kWinTmaxAlloc = 8;   // exchange buffers are sized for T <= 8
constexpr int kWinXSlots = 4;      // exchange slots (epoch mod 4)

// Error bits of the window kernel.
constexpr unsigned kErrWinFull = 16u;      // weight tiles did not land
constexpr unsigned kErrWinEmpty = 32u;     // producer: ring entry never released
constexpr unsigned kErrWinCluster = 64u;   // cluster exchange did not complete
constexpr unsigned kErrWinGlobal = 128u;   // global exchange did not complete
constexpr unsigned kErrWinLaunch = 256u;   // launched with a grid, block or cluster shape it was not built for
// Waits inside a CTA or its cluster give up only after this long (longer than
// kWaitNs, the limit of the waits across clusters that they may wait behind).
constexpr uint64_t kLocalWaitNs = 4 * kWaitNs;

struct WinRead {
  const float* R;          // [T][N]
  const float* P;          // [T][N] or null
  const float* w_norm;     // [N]
  const uint16_t* W_down;  // [K][N] BF16
  const uint16_t* W_up;    // [N][K] BF16
  const float* gate;       // [N]
  float* out;              // [T][N]
  float* mean;             // [T][d]
  float* lo;               // [T][K]
};

struct WinArgs {
  unsigned* xbuf;            // [2][4 ranks][32 clusters][8][KQ] tagged words: partial sums
  unsigned* xss;             // [2][8][32 clusters][2] tagged words: sums of squares, 0
  unsigned* mbuf;            // [2][4 streams][8][d] tagged words (output tiles)
  unsigned* gen;             // [128] reads completed by each CTA (epoch base)
  unsigned* abort_flag;
  unsigned* err;
  int count;                 // reads in this launch, 1..kWinMaxReads
  int T;
  float eps;
  int pad_;
  unsigned char chained[kWinMaxReads];  // 1: R of this read is the previous read's out
  WinRead rd[kWinMaxReads];
};

template <int D, int KD, int NT>
struct WinGeo {
  static constexpr int N = kStreams * D;
  static constexpr int PER_STREAM = kWinCtas / kStreams;    // CTAs per stream (32)
  static constexpr int CL = kWinCluster;
  static constexpr int CLUSTERS = kWinCtas / CL;            // 32
  static constexpr int CL_PER_STREAM = PER_STREAM / CL;     // 8
  static constexpr int W = D / PER_STREAM;                  // columns per CTA (80)
  static constexpr int KQ = KD / CL;                        // k per cluster rank (80)
  static constexpr int XW = KQ + 4;                         // row of the sums: partials, ss, 0, 0, 0
  static constexpr int XV = KQ / 4;                         // exchange row (partials) in 16-byte vectors
  static constexpr int TMAX = 4 * NT;
  static constexpr int XT = kWinTmaxAlloc;                  // token stride of the buffers
  static constexpr int NCW = 10;                            // compute warps
  // Producer warps: 128 threads keep each thread's cp.async copies in flight
  // near 100 (two ring entries of ~52).  A variant with 64 producer threads
  // raised an illegal-instruction fault on GB300 (cause not established);
  // 14 warps cap the kernel at 128 registers a thread.
  static constexpr int NPW = 4;
  static constexpr int CT = 32 * NCW;
  static constexpr int PT = 32 * NPW;
  static constexpr int THREADS = CT + PT;
  static constexpr int WD_CH = W / 8;                       // 16-byte chunks per W_down row slice
  static constexpr int WU_CH = KD / 8;                      // 16-byte chunks per W_up row
  static constexpr int WD_ROWB = W * 2;
  static constexpr int WU_ROWB = KD * 2;
  static constexpr int XS_PITCH = W * 2 + 16;               // an odd number of 16-byte chunks
  static constexpr int LS_PITCH = KD * 2 + 16;              // ... ditto
  static constexpr int DN_MT = KD / 16;                     // down m16 tiles (rows of W_down)
  static constexpr int DN_MPW = DN_MT / NCW;                // ... per warp
  static constexpr int DN_KS = W / 16;                      // down k-steps
  static constexpr int MT_PER_Q = KQ / 16;                  // down m16 tiles per rank quarter
  static constexpr int UP_MT = W / 16;                      // up m16 tiles (rows of W_up)
  // One ring entry: everything a read takes from HBM.
  static constexpr int E_WD = 0;
  static constexpr int E_WU = E_WD + KD * WD_ROWB;
  static constexpr int E_WN = E_WU + W * WU_ROWB;
  static constexpr int E_GATE = E_WN + W * 4;
  static constexpr int E_R = E_GATE + W * 4;
  static constexpr int E_P = E_R + TMAX * W * 4;
  static constexpr int ENT_BYTES = E_P + TMAX * W * 4;
  // The CTA's shared memory.
  static constexpr int BAR = 0;                              // 10 mbarriers
  static constexpr int ENT = 128;                            // two ring entries
  static constexpr int XS = ENT + 2 * ENT_BYTES;             // [8 NT][W] bf16: x hi/lo rows
  static constexpr int LS = XS + 8 * NT * XS_PITCH;          // [8 NT][K] bf16: lo hi/lo rows
  static constexpr int RP = LS + 8 * NT * LS_PITCH;          // [TMAX][W] R', then out
  static constexpr int RECV = RP + TMAX * W * 4;             // see RECV_BYTES
  static constexpr int RECV_PART = CL * TMAX * KQ * 4;       // [CL src][TMAX][KQ] partials
  static constexpr int RECV_SS = RECV_PART;                  // then [CL src][TMAX] ss
  static constexpr int SUMS_BYTES = kStreams * TMAX * XW * 4;  // exchange sums [4][TMAX][XW]
  static constexpr int RECV_BYTES =
      (RECV_PART + CL * TMAX * 4) > SUMS_BYTES ? (RECV_PART + CL * TMAX * 4) : SUMS_BYTES;
  static constexpr int BYTES = RECV + RECV_BYTES;
  // Transaction bytes per read at each cluster rank.
  __host__ __device__ static constexpr int rs_bytes(int T) { return CL * (T * KQ * 4 + T * 4); }
  __host__ __device__ static constexpr int lo_bytes(int T) { return CL * T * KQ * 4; }

  static_assert(kWinCtas % (kStreams * CL) == 0, "clusters must not straddle streams");
  static_assert(DN_MT % NCW == 0 && KQ % 16 == 0, "down tiles must split over warps and ranks");
  static_assert(UP_MT <= NCW, "one warp per up m16 tile");
  static_assert(W % 16 == 0 && W / 4 <= 32, "column slab must be whole k-steps, one warp per token");
  static_assert(WD_CH % 4 == 2, "W_down swizzle assumes a row of 2 (mod 4) chunks");
  static_assert(WU_CH % 8 == 0, "W_up swizzle assumes a row of a multiple of 8 chunks");
  static_assert(TMAX <= NCW, "one warp stages one token");
  static_assert(TMAX <= XT && XT <= CT, "exchange rows cover every token");
  static_assert((XS_PITCH / 16) % 2 == 1 && (LS_PITCH / 16) % 2 == 1 && XS_PITCH % 16 == 0 && LS_PITCH % 16 == 0,
                "8 B rows of an odd number of 16-byte chunks are conflict-free for ldmatrix");
  static_assert(KQ % 4 == 0 && (W / kStreams) % 4 == 0, "exchange rows and mean quarters are 16-byte vectors");
  static_assert(BYTES <= 232448, "shared memory per CTA");
};

namespace win {

// Shared-memory byte offset of chunk c of row r of the W_down tile (rows of
// 2 mod 4 chunks): chunks of rows 4..7 of every 8 are paired with their
// neighbour, which makes an ldmatrix of 8 rows conflict-free.
__device__ __forceinline__ int wd_off(int r, int c, int rowb) {
  return r * rowb + ((c ^ ((r >> 2) & 1)) << 4);
}
// ... and of the W_up tile (rows of a multiple of 8 chunks): XOR with r mod 8.
__device__ __forceinline__ int wu_off(int r, int c, int rowb) {
  return r * rowb + ((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst)),
               "l"(src), "l"(pol)
               : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the arrival is one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}
// Phase wait with acquire at cluster scope (data written by other CTAs'
// st.async of the cluster).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(ptx::smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 4-byte store into the shared memory of cluster CTA `rank`, counted as 4
// transaction bytes on that CTA's barrier `bar` (both given as this CTA's
// shared addresses of the same variables).
__device__ __forceinline__ void st_async(uint32_t addr, uint32_t v, uint32_t bar, uint32_t rank) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   mapa(addr, rank)),
               "r"(v), "r"(mapa(bar, rank))
               : "memory");
}

// Self-tagged exchange words: fp32 bits with the three low mantissa bits
// replaced by the epoch modulo 8.
__device__ __forceinline__ uint32_t tag_word(float v, uint32_t epoch) {
  return (__float_as_uint(v) & ~7u) | (epoch & 7u);
}
__device__ __forceinline__ float tag_val(uint32_t w) { return __uint_as_float(w & ~7u); }
__device__ __forceinline__ bool tags_ok(const uint4& w, uint32_t epoch) {
  const uint32_t e = epoch & 7u;
  return ((w.x & 7u) == e) & ((w.y & 7u) == e) & ((w.z & 7u) == e) & ((w.w & 7u) == e);
}
// Stores are 8-byte relaxed (strong) stores, loads 16-byte relaxed loads of
// two 8-byte elements; a word is never torn.
__device__ __forceinline__ void st_tag2(unsigned* p, uint32_t lo, uint32_t hi) {
  const unsigned long long w = ((unsigned long long)hi << 32) | lo;
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ void st_tag4(unsigned* p, uint4 w) {
  st_tag2(p, w.x, w.y);
  st_tag2(p + 2, w.z, w.w);
}
__device__ __forceinline__ uint4 ld_tag4(const unsigned* p) {
  unsigned long long a, b;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
  return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
}

__device__ __forceinline__ unsigned load_abort(const unsigned* f) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ void raise_abort(unsigned* f, unsigned* err, unsigned code) {
  atomicOr(err, code);
  atomicExch(f, 1u);
}

// Exit of a CTA of a CL-CTA cluster whose CTAs store into one another's
// shared memory (st.async), called by every thread, converged, after the
// CTA's last store was issued.  Every byte a peer sent was waited for by its
// receiver (local waits never skip), so nothing is in flight any more; the
// cluster barrier keeps every CTA resident until all have passed their last
// wait on a peer's stores.
__device__ __forceinline__ void leave_cluster() {
  ptx::cluster_arrive_release();
  ptx::cluster_wait();
}

// Bounded wait on a phase of an mbarrier of this CTA that only this CTA's
// copies or its cluster peers complete (see the header: such waits ignore the
// abort word).  After kLocalWaitNs the thread records `code`, raises the
// abort word and marks the CTA broken (*broken, shared memory), which makes
// every later local wait of the CTA return at once: the protocol cannot be
// kept any more, and the kernel only runs to its end.
template <bool kCluster>
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile unsigned* broken,
                                           unsigned* abort_flag, unsigned* err, unsigned code) {
  auto probe = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity); };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (unsigned n = 1;; ++n) {
    if (probe()) return true;
    if ((n & 31u) == 0u) {
      if (*broken != 0u) return false;
      if (ptx::globaltimer_ns() - t0 > kLocalWaitNs) {
        *broken = 1u;
        raise_abort(abort_flag, err, code);
        return false;
      }
    }
  }
}

// Bounded poll of MI x MC 16-byte tagged vectors, vector (m, c) at
// base[m] + c * stride: reloads every vector whose tags are not yet `epoch`,
// all in flight together, until all are.  Items m >= ni are ignored.
template <int MI, int MC>
__device__ __forceinline__ bool poll_all(uint4 (&v)[MI][MC], const unsigned* const (&base)[MI], size_t stride,
                                         int ni, uint32_t epoch, unsigned* abort_flag, unsigned* err) {
  uint64_t t0 = 0;
  for (unsigned it = 0;; ++it) {
    bool done = true;
#pragma unroll
    for (int m = 0; m < MI; ++m)
#pragma unroll
      for (int c = 0; c < MC; ++c) done &= (m >= ni) || tags_ok(v[m][c], epoch);
    if (done) return true;
    if (it == 0) {
      t0 = ptx::globaltimer_ns();
    } else if ((it & 15u) == 0u) {
      if (load_abort(abort_flag) != 0u) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitNs) {
        raise_abort(abort_flag, err, kErrWinGlobal);
        return false;
      }
    }
#pragma unroll
    for (int m = 0; m < MI; ++m)
#pragma unroll
      for (int c = 0; c < MC; ++c) {
        if (m < ni && !tags_ok(v[m][c], epoch)) v[m][c] = ld_tag4(base[m] + c * stride);
      }
  }
}

// Named barrier of the compute warps (the producer warps never take part).
template <int COUNT>
__device__ __forceinline__ void compute_sync() {
  asm volatile("barrier.sync 1, %0;" ::"n"(COUNT) : "memory");
}

// hi = bf16(v), lo = bf16(v - hi) for a pair, packed two per word.
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
  const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(__fsub_rn(v0, __uint_as_float(u << 16)),
                                                 __fsub_rn(v1, __uint_as_float(u & 0xffff0000u)));
  hi = u;
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

}  // namespace win

// The stream mean of one read for this CTA's quarter of its columns, from the
// four streams' published output tiles: thread `tid` < T * W/16 owns four
// columns of one token.  mean_issue loads, mean_finish polls and writes.
template <int D, int KD, int NT>
struct WinMean {
  using G = WinGeo<D, KD, NT>;
  static constexpr int QV = G::W / kStreams / 4;  // 16-byte vectors per token in the quarter
  uint4 v[1][kStreams];
  const unsigned* base[1];
  int n;  // 0: this thread owns no columns
  int t, c;

  __device__ __forceinline__ void issue(const WinArgs& a, uint32_t epoch, int s, int j, int tid) {
    n = tid < a.T * QV ? 1 : 0;
    t = n ? tid / QV : 0;
    c = j * G::W + s * (G::W / kStreams) + (tid % QV) * 4;
    base[0] = a.mbuf + ((size_t)(epoch % kWinXSlots) * kStreams * G::XT + t) * D + c;
    if (n) {
#pragma unroll
      for (int s2 = 0; s2 < kStreams; ++s2) v[0][s2] = win::ld_tag4(base[0] + (size_t)s2 * G::XT * D);
    }
  }
  __device__ __forceinline__ bool finish(const WinArgs& a, int i, uint32_t epoch, bool ok) {
    if (n == 0 || !ok) return ok;
    if (!win::poll_all<1, kStreams>(v, base, (size_t)G::XT * D, 1, epoch, a.abort_flag, a.err)) return false;
    const uint4* w = v[0];
    float4 m;
    m.x = (((win::tag_val(w[0].x) + win::tag_val(w[1].x)) + win::tag_val(w[2].x)) + win::tag_val(w[3].x)) * 0.25f;
    m.y = (((win::tag_val(w[0].y) + win::tag_val(w[1].y)) + win::tag_val(w[2].y)) + win::tag_val(w[3].y)) * 0.25f;
    m.z = (((win::tag_val(w[0].z) + win::tag_val(w[1].z)) + win::tag_val(w[2].z)) + win::tag_val(w[3].z)) * 0.25f;
    m.w = (((win::tag_val(w[0].w) + win::tag_val(w[1].w)) + win::tag_val(w[2].w)) + win::tag_val(w[3].w)) * 0.25f;
    *reinterpret_cast<float4*>(a.rd[i].mean + (size_t)t * D + c) = m;
    return true;
  }
};

template <int D, int KD, int NT>
__global__ void __launch_bounds__(WinGeo<D, KD, NT>::THREADS, 1)
    hc_window_kernel(const __grid_constant__ WinArgs a) {
  using G = WinGeo<D, KD, NT>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::BAR);
  uint64_t* full_d = bars;       // [2] W_down tile, w_norm, R, P of a ring entry have landed
  uint64_t* full_u = bars + 2;   // [2] W_up tile and gate have landed
  uint64_t* empty_d = bars + 4;  // [2] the compute warps are done with the down part
  uint64_t* empty_u = bars + 6;  // [2] ... with the up part
  uint64_t* bar_rs = bars + 8;   // partials of this rank's quarter from the 4 CTAs
  uint64_t* bar_lo = bars + 9;   // lo (hi/lo split) from the 4 ranks
  unsigned char* xs = smem + G::XS;
  unsigned char* ls = smem + G::LS;
  float* rp = reinterpret_cast<float*>(smem + G::RP);
  float* recv = reinterpret_cast<float*>(smem + G::RECV);
  float* recv_ss = reinterpret_cast<float*>(smem + G::RECV + G::RECV_SS);
  float* sums = reinterpret_cast<float*>(smem + G::RECV);  // reuses the receive area

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int b = blockIdx.x;
  const int s = b / G::PER_STREAM;      // stream
  const int j = b % G::PER_STREAM;      // column slab within the stream
  const int q = b / G::CL;              // cluster
  const uint32_t rank = b % G::CL;      // rank in the cluster (1-D clusters along x)
  const int col0 = s * D + j * G::W;    // first column of W_down / row of W_up
  const int T = a.T;
  __shared__ unsigned broken;  // a local wait of this CTA ran out (see wait_phase)

  // The launch shape the CTA numbering above assumes: every CTA of a launch
  // sees the same shape, so either all return here or none does.
  if (ptx::cluster_nctarank() != (uint32_t)G::CL || ptx::cluster_ctarank() != rank ||
      gridDim.x != (unsigned)kWinCtas || gridDim.y != 1u || gridDim.z != 1u || blockDim.x != (unsigned)G::THREADS) {
    if (tid == 0) atomicOr(a.err, kErrWinLaunch);
    return;
  }

  if (tid == 0) {
    broken = 0u;
    for (int e = 0; e < 2; ++e) {
      ptx::mbar_init(&full_d[e], G::PT);
      ptx::mbar_init(&full_u[e], G::PT);
      ptx::mbar_init(&empty_d[e], G::NCW);
      ptx::mbar_init(&empty_u[e], G::NCW);
    }
    ptx::mbar_init(bar_rs, 1);
    ptx::mbar_init(bar_lo, 1);
    ptx::mbar_arrive_expect_tx(bar_rs, G::rs_bytes(T));  // arm read 0
    ptx::mbar_arrive_expect_tx(bar_lo, G::lo_bytes(T));
    ptx::fence_barrier_init();
  }
  // B operand rows of tokens >= T stay zero for the whole launch.
  for (int idx = tid; idx < (8 * NT * (G::XS_PITCH + G::LS_PITCH)) / 16; idx += G::THREADS) {
    reinterpret_cast<uint4*>(xs)[idx] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  // No CTA sends into a peer before the peer's barriers exist and its B rows are zeroed.
  ptx::cluster_arrive_release();
  ptx::cluster_wait();

  if (warp >= G::NCW) {
    // ------------------------------------------------------------ producer warps
    const int pt = tid - G::CT;
    const uint64_t pol = ptx::policy_evict_first();
    for (int i = 0; i < a.count; ++i) {
      const int e = i & 1;
      const WinRead& rd = a.rd[i];
      unsigned char* ent = smem + G::ENT + e * G::ENT_BYTES;
      // Entry e was last used by read i - 2.
      if (i >= 2 && !win::wait_phase<false>(&empty_d[e], ((i >> 1) + 1) & 1, &broken, a.abort_flag, a.err, kErrWinEmpty)) break;
      for (int idx = pt; idx < KD * G::WD_CH; idx += G::PT) {
        const int r = idx / G::WD_CH, c = idx - r * G::WD_CH;
        win::cp_async16(ent + G::E_WD + win::wd_off(r, c, G::WD_ROWB), rd.W_down + (size_t)r * G::N + col0 + c * 8,
                        pol);
      }
      for (int idx = pt; idx < G::W / 4; idx += G::PT) {
        win::cp_async16(ent + G::E_WN + idx * 16, rd.w_norm + col0 + idx * 4, pol);
      }
      // R and P may be written by the preceding kernel: wait for it first.
      if (i == 0) ptx::wait_prerequisites();
      if (!a.chained[i]) {
        for (int idx = pt; idx < T * (G::W / 4); idx += G::PT) {
          const int t = idx / (G::W / 4), c4 = idx % (G::W / 4);
          win::cp_async16(ent + G::E_R + (t * G::W + c4 * 4) * 4, rd.R + (size_t)t * G::N + col0 + c4 * 4, pol);
        }
      }
      if (rd.P != nullptr) {
        for (int idx = pt; idx < T * (G::W / 4); idx += G::PT) {
          const int t = idx / (G::W / 4), c4 = idx % (G::W / 4);
          win::cp_async16(ent + G::E_P + (t * G::W + c4 * 4) * 4, rd.P + (size_t)t * G::N + col0 + c4 * 4, pol);
        }
      }
      win::cp_async_arrive(&full_d[e]);
      if (i >= 2 && !win::wait_phase<false>(&empty_u[e], ((i >> 1) + 1) & 1, &broken, a.abort_flag, a.err, kErrWinEmpty)) break;
      for (int idx = pt; idx < G::W * G::WU_CH; idx += G::PT) {
        const int r = idx / G::WU_CH, c = idx - r * G::WU_CH;
        win::cp_async16(ent + G::E_WU + win::wu_off(r, c, G::WU_ROWB), rd.W_up + (size_t)(col0 + r) * KD + c * 8,
                        pol);
      }
      for (int idx = pt; idx < G::W / 4; idx += G::PT) {
        win::cp_async16(ent + G::E_GATE + idx * 16, rd.gate + col0 + idx * 4, pol);
      }
      win::cp_async_arrive(&full_u[e]);
    }
    win::cp_async_wait_all();  // nothing may land after the CTA has exited
  } else {
    // ------------------------------------------------------------ compute warps
    ptx::wait_prerequisites();  // outputs and the epoch base belong to the preceding kernel until here
    const uint32_t base = a.gen[b];
    bool ok = true;
    const int g = lane >> 2;   // MMA row group
    const int qd = lane & 3;   // MMA column pair = token within an n-tile
    const uint32_t xs_a = ptx::smem_u32(xs);
    const uint32_t ls_a = ptx::smem_u32(ls);
    const uint32_t recv_a = ptx::smem_u32(recv);
    const uint32_t recv_ss_a = ptx::smem_u32(recv_ss);
    const uint32_t bar_rs_a = ptx::smem_u32(bar_rs);
    const uint32_t bar_lo_a = ptx::smem_u32(bar_lo);

    // Every compute thread runs every iteration, whatever its `ok`: the named
    // barriers below need all of them.  Once a wait has failed, the abort word
    // makes every later wait return at once.
    for (int i = 0; i < a.count; ++i) {
      const int e = i & 1;
      const uint32_t ph = (i >> 1) & 1;   // ring entry phase
      const uint32_t xp = i & 1;          // exchange barrier phase
      const WinRead& rd = a.rd[i];
      const uint32_t epoch = base + 1u + (uint32_t)i;
      const int p = epoch % kWinXSlots;  // exchange slot
      unsigned char* ent = smem + G::ENT + e * G::ENT_BYTES;

      // (1) down part of the entry: W_down tile, w_norm, R, P.
      ok = win::wait_phase<false>(&full_d[e], ph, &broken, a.abort_flag, a.err, kErrWinFull) && ok;
      // (2) staging, one warp per token: R' = R + P (or the previous read's
      // out + P), x = R' * w_norm split into hi/lo B rows, sums of squares.
      if (warp < T) {
        const int t = warp;
        float ss = 0.f;
        if (lane < G::W / 4) {
          const float4* rsrc = reinterpret_cast<const float4*>(a.chained[i] ? reinterpret_cast<unsigned char*>(rp)
                                                                             : ent + G::E_R);
          float4 r = rsrc[t * (G::W / 4) + lane];
          if (rd.P != nullptr) {
            const float4 pv = reinterpret_cast<const float4*>(ent + G::E_P)[t * (G::W / 4) + lane];
            r.x = __fadd_rn(r.x, pv.x);
            r.y = __fadd_rn(r.y, pv.y);
            r.z = __fadd_rn(r.z, pv.z);
            r.w = __fadd_rn(r.w, pv.w);
          }
          const float4 w = reinterpret_cast<const float4*>(ent + G::E_WN)[lane];
          const float4 x = make_float4(__fmul_rn(r.x, w.x), __fmul_rn(r.y, w.y), __fmul_rn(r.z, w.z),
                                       __fmul_rn(r.w, w.w));
          uint2 hi, lo;
          split4(x, hi, lo);
          *reinterpret_cast<uint2*>(xs + (2 * t) * G::XS_PITCH + lane * 8) = hi;
          *reinterpret_cast<uint2*>(xs + (2 * t + 1) * G::XS_PITCH + lane * 8) = lo;
          reinterpret_cast<float4*>(rp)[t * (G::W / 4) + lane] = r;
          ss = __fmaf_rn(r.x, r.x, ss);
          ss = __fmaf_rn(r.y, r.y, ss);
          ss = __fmaf_rn(r.z, r.z, ss);
          ss = __fmaf_rn(r.w, r.w, ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane < G::CL) {
          win::st_async(recv_ss_a + (rank * G::TMAX + t) * 4, __float_as_uint(ss), bar_rs_a, lane);
        }
      }
      win::compute_sync<G::CT>();  // x rows complete

      // (3) down projection: warp w owns W_down rows 16 * (DN_MPW w + m) ...
      // The warp's lanes left the waits above one by one and the named
      // barrier does not reconverge them: ldmatrix and mma are .aligned.
      __syncwarp();
      {
        float acc[G::DN_MPW][NT][4];
#pragma unroll
        for (int m = 0; m < G::DN_MPW; ++m)
#pragma unroll
          for (int n = 0; n < NT; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
        const unsigned char* wd = ent + G::E_WD;
#pragma unroll
        for (int ks = 0; ks < G::DN_KS; ++ks) {
          uint32_t b0[NT], b1[NT];
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            ptx::ldsm_x2(xs_a + (n * 8 + (lane & 7)) * G::XS_PITCH + (2 * ks + ((lane >> 3) & 1)) * 16, b0[n], b1[n]);
          }
#pragma unroll
          for (int m = 0; m < G::DN_MPW; ++m) {
            const int row = (warp * G::DN_MPW + m) * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
            uint32_t af[4];
            ptx::ldsm_x4(ptx::smem_u32(wd + win::wd_off(row, 2 * ks + (lane >> 4), G::WD_ROWB)), af[0], af[1], af[2],
                         af[3]);
#pragma unroll
            for (int n = 0; n < NT; ++n) ptx::mma_bf16_16816(acc[m][n], af, b0[n], b1[n]);
          }
        }
        __syncwarp();
        if (lane == 0) win::mbar_arrive(&empty_d[e]);
        // Partials of rows in quarter `dst` go to cluster rank dst.
#pragma unroll
        for (int m = 0; m < G::DN_MPW; ++m) {
          const int mt = warp * G::DN_MPW + m;
          const uint32_t dst = mt / G::MT_PER_Q;
          const int kl = mt * 16 - (int)dst * G::KQ + g;
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const int t = n * 4 + qd;
            if (t < T) {
              const float v0 = __fadd_rn(acc[m][n][0], acc[m][n][1]);
              const float v1 = __fadd_rn(acc[m][n][2], acc[m][n][3]);
              const uint32_t at = recv_a + ((rank * G::TMAX + t) * G::KQ + kl) * 4;
              win::st_async(at, __float_as_uint(v0), bar_rs_a, dst);
              win::st_async(at + 32, __float_as_uint(v1), bar_rs_a, dst);
            }
          }
        }
      }

      // (4) this rank's quarter: sum the 4 CTAs, publish as LL packets.
      {
        // Arm the next read only once this phase has completed: arming an
        // incomplete phase would take its arrival count below zero.
        const bool got = win::wait_phase<true>(bar_rs, xp, &broken, a.abort_flag, a.err, kErrWinCluster);
        ok = got && ok;
        if (tid == 0 && got) ptx::mbar_arrive_expect_tx(bar_rs, G::rs_bytes(T));
      }
      {
        unsigned* xrow = a.xbuf + (((size_t)p * G::CL + rank) * G::CLUSTERS + q) * G::XT * G::KQ;
        for (int idx = tid; idx < G::XT * G::XV; idx += G::CT) {
          const int t = idx / G::XV, k = (idx % G::XV) * 4;
          float vx = 0.f, vy = 0.f, vz = 0.f, vw = 0.f;
          if (t < T) {
            const float4* r0 = reinterpret_cast<const float4*>(recv + t * G::KQ + k);
            constexpr int SRC = G::TMAX * G::KQ / 4;  // float4 stride between sources
            const float4 a0 = r0[0], a1 = r0[SRC], a2 = r0[2 * SRC], a3 = r0[3 * SRC];
            vx = ((a0.x + a1.x) + a2.x) + a3.x;
            vy = ((a0.y + a1.y) + a2.y) + a3.y;
            vz = ((a0.z + a1.z) + a2.z) + a3.z;
            vw = ((a0.w + a1.w) + a2.w) + a3.w;
          }
          win::st_tag2(xrow + t * G::KQ + k, win::tag_word(vx, epoch), win::tag_word(vy, epoch));
          win::st_tag2(xrow + t * G::KQ + k + 2, win::tag_word(vz, epoch), win::tag_word(vw, epoch));
        }
        if (rank == 0 && tid < G::XT) {
          const int t = tid;
          const float ss = t >= T ? 0.f
                                  : ((recv_ss[t] + recv_ss[G::TMAX + t]) + recv_ss[2 * G::TMAX + t]) +
                                        recv_ss[3 * G::TMAX + t];
          win::st_tag2(a.xss + (((size_t)p * G::XT + t) * G::CLUSTERS + q) * 2, win::tag_word(ss, epoch),
                       win::tag_word(0.f, epoch));
        }
      }
      win::compute_sync<G::CT>();  // the receive area is read before it is reused for the sums

      // (5) global exchange: this rank's quarter from all 32 clusters, summed
      // per stream over its 8 clusters (fixed order).  Column KQ carries the
      // sums of squares.  Every load of the thread is in flight at once, the
      // previous read's stream-mean loads included.
      {
        constexpr int ITEMS = kStreams * G::TMAX * G::XV;
        constexpr int XI = (ITEMS + G::CT - 1) / G::CT;      // items per thread
        constexpr int CP = G::CL_PER_STREAM;
        constexpr size_t CSTRIDE = (size_t)G::XT * G::KQ;   // words between clusters
        static_assert(kStreams * G::TMAX <= G::CT, "one sum-of-squares item per thread");
        WinMean<D, KD, NT> mean;
        mean.n = 0;
        if (i > 0) mean.issue(a, epoch - 1u, s, j, tid);
        uint4 v[XI][CP];
        const unsigned* base[XI];
        int ni = 0;
#pragma unroll
        for (int m = 0; m < XI; ++m) {
          const int it = tid + m * G::CT;
          base[m] = a.xbuf;
          if (it < kStreams * T * G::XV) {
            const int s2 = it / (T * G::XV);
            const int rem = it - s2 * (T * G::XV);
            const int t = rem / G::XV, k = (rem % G::XV) * 4;
            base[m] = a.xbuf + ((((size_t)p * G::CL + rank) * G::CLUSTERS + s2 * CP) * G::XT + t) * G::KQ + k;
#pragma unroll
            for (int c8 = 0; c8 < CP; ++c8) v[m][c8] = win::ld_tag4(base[m] + c8 * CSTRIDE);
            ni = m + 1;
          }
        }
        // Sums of squares: thread (stream s2, token t) reads its stream's 8
        // clusters, two words each.
        uint4 vs[1][CP / 2];
        const unsigned* bss[1] = {a.xss};
        const int nss = tid < kStreams * T ? 1 : 0;
        if (nss) {
          bss[0] = a.xss + (((size_t)p * G::XT + tid % T) * G::CLUSTERS + (tid / T) * CP) * 2;
#pragma unroll
          for (int c = 0; c < CP / 2; ++c) vs[0][c] = win::ld_tag4(bss[0] + c * 4);
        }
        if (ok && ni > 0) ok = win::poll_all<XI, CP>(v, base, CSTRIDE, ni, epoch, a.abort_flag, a.err);
        if (ok && nss) ok = win::poll_all<1, CP / 2>(vs, bss, 4, 1, epoch, a.abort_flag, a.err);
#pragma unroll
        for (int m = 0; m < XI; ++m) {
          const int it = tid + m * G::CT;
          if (m < ni) {
            const int s2 = it / (T * G::XV);
            const int rem = it - s2 * (T * G::XV);
            const int t = rem / G::XV, k = (rem % G::XV) * 4;
            float4 acc = make_float4(win::tag_val(v[m][0].x), win::tag_val(v[m][0].y), win::tag_val(v[m][0].z),
                                     win::tag_val(v[m][0].w));
#pragma unroll
            for (int c8 = 1; c8 < CP; ++c8) {
              const uint4& w = v[m][c8];
              acc.x = __fadd_rn(acc.x, win::tag_val(w.x));
              acc.y = __fadd_rn(acc.y, win::tag_val(w.y));
              acc.z = __fadd_rn(acc.z, win::tag_val(w.z));
              acc.w = __fadd_rn(acc.w, win::tag_val(w.w));
            }
            *reinterpret_cast<float4*>(sums + (s2 * G::TMAX + t) * G::XW + k) = acc;
          }
        }
        if (nss) {
          // Clusters in order: words 0 and 2 of each 16-byte vector.
          float ss = win::tag_val(vs[0][0].x);
          ss = __fadd_rn(ss, win::tag_val(vs[0][0].z));
#pragma unroll
          for (int c = 1; c < CP / 2; ++c) {
            ss = __fadd_rn(ss, win::tag_val(vs[0][c].x));
            ss = __fadd_rn(ss, win::tag_val(vs[0][c].z));
          }
          sums[((tid / T) * G::TMAX + tid % T) * G::XW + G::KQ] = ss;
        }
        // The previous read's stream mean (its loads were issued above).
        if (i > 0) ok = mean.finish(a, i - 1, epoch - 1u, ok);
      }
      win::compute_sync<G::CT>();

      // (6) lo for this quarter: rs per stream, fixed-order sum over the
      // streams, split into hi/lo, sent to all four ranks.
      for (int it = tid; it < T * (G::KQ / 2); it += G::CT) {
        const int t = it / (G::KQ / 2), k2 = it % (G::KQ / 2);
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kStreams; ++s2) {
          const float* sr = sums + (s2 * G::TMAX + t) * G::XW;
          const float rs = rsqrtf(sr[G::KQ] * (1.0f / (float)D) + a.eps);
          const float p0 = __fmul_rn(rs, sr[2 * k2]);
          const float p1 = __fmul_rn(rs, sr[2 * k2 + 1]);
          l0 = s2 == 0 ? p0 : __fadd_rn(l0, p0);
          l1 = s2 == 0 ? p1 : __fadd_rn(l1, p1);
        }
        uint32_t hi, lo;
        win::split2(l0, l1, hi, lo);
        const int k = (int)rank * G::KQ + 2 * k2;
        const uint32_t ahi = ls_a + (2 * t) * G::LS_PITCH + k * 2;
#pragma unroll
        for (uint32_t dst = 0; dst < (uint32_t)G::CL; ++dst) {
          win::st_async(ahi, hi, bar_lo_a, dst);
          win::st_async(ahi + G::LS_PITCH, lo, bar_lo_a, dst);
        }
        if (q == 0) *reinterpret_cast<float2*>(rd.lo + (size_t)t * KD + k) = make_float2(l0, l1);
      }

      // (7) up part of the entry.
      ok = win::wait_phase<false>(&full_u[e], ph, &broken, a.abort_flag, a.err, kErrWinFull) && ok;
      {
        const bool got = win::wait_phase<true>(bar_lo, xp, &broken, a.abort_flag, a.err, kErrWinCluster);
        ok = got && ok;
        if (tid == 0 && got) ptx::mbar_arrive_expect_tx(bar_lo, G::lo_bytes(T));  // arm the next read
      }

      // (8) up projection, one warp per m16 tile of W_up rows over the whole
      // K, and the epilogue from the accumulators.
      {
        __syncwarp();
        unsigned* mrow = a.mbuf + (((size_t)p * kStreams + s) * G::XT) * D + j * G::W;
        constexpr int UPW = G::UP_MT;
        if (warp < UPW) {
          const int mt = warp;
          const unsigned char* wu = ent + G::E_WU;
          const int row = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          float acc[NT][4], acc2[NT][4];
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
            acc2[n][0] = acc2[n][1] = acc2[n][2] = acc2[n][3] = 0.f;
          }
#pragma unroll
          for (int ks = 0; ks < KD / 16; ++ks) {
            uint32_t af[4];
            ptx::ldsm_x4(ptx::smem_u32(wu + win::wu_off(row, 2 * ks + (lane >> 4), G::WU_ROWB)), af[0], af[1], af[2],
                         af[3]);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              uint32_t b0, b1;
              ptx::ldsm_x2(ls_a + (n * 8 + (lane & 7)) * G::LS_PITCH + (2 * ks + ((lane >> 3) & 1)) * 16, b0, b1);
              ptx::mma_bf16_16816((ks & 1) ? acc2[n] : acc[n], af, b0, b1);
            }
          }
          const float* gate = reinterpret_cast<const float*>(ent + G::E_GATE);
          const int r0 = mt * 16 + g;
          const float sg0 = 1.0f / (1.0f + expf(-gate[r0]));
          const float sg1 = 1.0f / (1.0f + expf(-gate[r0 + 8]));
          __syncwarp();
          if (lane == 0) win::mbar_arrive(&empty_u[e]);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const int t = n * 4 + qd;
            const float u0 = __fadd_rn(__fadd_rn(acc[n][0], acc2[n][0]), __fadd_rn(acc[n][1], acc2[n][1]));
            const float u1 = __fadd_rn(__fadd_rn(acc[n][2], acc2[n][2]), __fadd_rn(acc[n][3], acc2[n][3]));
            float o0 = 0.f, o1 = 0.f;
            if (t < T) {
              o0 = __fmaf_rn(sg0, u0, rp[t * G::W + r0]);
              o1 = __fmaf_rn(sg1, u1, rp[t * G::W + r0 + 8]);
              rd.out[(size_t)t * G::N + col0 + r0] = o0;
              rd.out[(size_t)t * G::N + col0 + r0 + 8] = o1;
              rp[t * G::W + r0] = o0;
              rp[t * G::W + r0 + 8] = o1;
            }
            const float n0 = __shfl_down_sync(0xffffffffu, o0, 4);
            const float n1 = __shfl_down_sync(0xffffffffu, o1, 4);
            if ((g & 1) == 0) {
              win::st_tag2(mrow + (size_t)t * D + r0, win::tag_word(o0, epoch), win::tag_word(n0, epoch));
              win::st_tag2(mrow + (size_t)t * D + r0 + 8, win::tag_word(o1, epoch), win::tag_word(n1, epoch));
            }
          }
        } else {
          __syncwarp();
          if (lane == 0) win::mbar_arrive(&empty_u[e]);
          for (int idx = tid - 32 * UPW; idx < (G::XT - G::TMAX) * (G::W / 2); idx += G::CT - 32 * UPW) {
            const int t = G::TMAX + idx / (G::W / 2), c = (idx % (G::W / 2)) * 2;
            win::st_tag2(mrow + (size_t)t * D + c, win::tag_word(0.f, epoch), win::tag_word(0.f, epoch));
          }
        }
      }
      win::compute_sync<G::CT>();  // the out tile is complete before the next read
    }
    // The last read's stream mean.
    {
      WinMean<D, KD, NT> mean;
      mean.issue(a, base + (uint32_t)a.count, s, j, tid);
      ok = mean.finish(a, a.count - 1, base + (uint32_t)a.count, ok);
    }
    win::compute_sync<G::CT>();
    if (tid == 0) a.gen[b] = base + (uint32_t)a.count;
  }
  __syncwarp();
  __syncthreads();
  win::leave_cluster();
}

}  // namespace hc
