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
#include <cuda_fp16.h>

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

template <int D, int KD, int NT, int Q8 = 0>
struct DownTcSmem {
  using G = Geo<D, KD>;
  static constexpr int TG = 4 * NT;
  static constexpr int NCOL = 8 * NT;
  static constexpr int XS_PITCH = G::SLAB * 2 + 16;   // bytes; = 16 (mod 128)
  // W_down rows: BF16, or Q8_0 int8 quants with their block scales apart
  // (mode 1: pitch an odd multiple of 32 bytes, so the 64-bit loads of four
  // rows x four lanes cover the 32 banks once; mode 2: BF16 rows, the quants
  // landing at byte Q8_OFF of each).
  static constexpr int WPITCH = Q8 == 1 ? G::SLAB + 32 : G::DN_PITCH;
  static constexpr int Q8_OFF = Q8 == 2 ? WPITCH - G::SLAB : 0;
  static constexpr int NB = G::SLAB / 32;              // Q8_0 blocks per row
  static constexpr int BAR = 0;
  static constexpr int W = 128;
  static constexpr int XS = W + G::DN_ROWS * WPITCH;  // [NCOL][SLAB] bf16: hi, lo rows
  // [4 K-parts][TG][32] partials, over the x rows: written only once every
  // warp is past its MMAs (a CTA barrier), read before the next group's x.
  static constexpr int RED = XS;
  // [kMaxT] rs of the cluster leader, over the partials: used only after the
  // cluster barrier, when this CTA's own sums are done.
  static constexpr int RS = RED;
  static constexpr int SSW = XS + NCOL * XS_PITCH;    // [8 warps][TG]
  // [32 rows][NB] binary16 block scales (Q8_0), copied in 8-byte pieces.
  static constexpr int SC = (SSW + kWarps * TG * 4 + 15) / 16 * 16;
  static constexpr int RECV = SC + (Q8 ? (G::DN_ROWS * NB * 2 + 15) / 16 * 16 : 0);  // [4][T] ss, then [4][T][32] partials
  static constexpr int bytes(int T) { return RECV + 4 * T * 4 + 4 * T * 32 * 4; }
  static constexpr int BYTES_MAX = RECV + 4 * kMaxT * 4 + 4 * kMaxT * 32 * 4;
  static_assert(XS_PITCH % 128 == 16, "x rows must be conflict-free for ldmatrix");
  static_assert(4 * TG * 32 * 4 <= NCOL * XS_PITCH && kMaxT <= 4 * TG * 32, "aliased regions fit");
  static_assert(!Q8 || (NB % 4 == 0 && (G::N / 32 * 2) % 8 == 0 && (NB * 2) % 8 == 0),
                "a row's scales are whole 8-byte pieces at 8-byte aligned addresses");
  static_assert(Q8 != 1 || WPITCH % 64 == 32, "Q8_0 rows: 64-bit fragment loads conflict-free");
  static_assert(Q8 != 2 || (Q8_OFF % 16 == 0 && Q8_OFF >= G::SLAB), "int8 rows on 16 bytes, past the BF16 half");
};

template <int D, int KD, int NT, int Q8 = 0>
struct UpTcSmem {
  using G = Geo<D, KD>;
  static constexpr int TG = 4 * NT;
  static constexpr int NCOL = 8 * NT;
  static constexpr int LS_PITCH = KD * 2 + 16;        // bytes; = 16 (mod 128)
  static constexpr int WPITCH = Q8 == 1 ? KD + 32 : G::UP_PITCH;  // W_up rows, as the down kernel's
  static constexpr int Q8_OFF = Q8 == 2 ? WPITCH - KD : 0;
  static constexpr int NB = KD / 32;                  // Q8_0 blocks per row
  static constexpr int BAR = 0;
  static constexpr int W = 128;
  static constexpr int GATE = W + G::UP_ROWS * WPITCH;
  static constexpr int SIG = GATE + G::UP_ROWS * 4;
  static constexpr int LS = SIG + G::UP_ROWS * 4;     // [NCOL][KD] bf16: hi, lo rows
  static constexpr int RED = LS + NCOL * LS_PITCH;    // [2 K-halves][TG][64]
  static constexpr int OUT = RED + 2 * TG * G::UP_ROWS * 4;
  static constexpr int RP = OUT + TG * G::UP_ROWS * 4;
  // [64 rows][NB] binary16 block scales (Q8_0): each stream's 16 rows are
  // one contiguous run of 16 NB scales in global memory, copied in 16-byte
  // pieces.
  static constexpr int SC = (RP + TG * G::UP_ROWS * 4 + 15) / 16 * 16;
  static constexpr int BYTES = SC + (Q8 ? G::UP_ROWS * NB * 2 : 0);
  static_assert(!Q8 || (G::UP_COLS * NB * 2) % 16 == 0, "a stream's scale run is whole 16-byte pieces");
  static_assert(Q8 != 1 || WPITCH % 64 == 32, "Q8_0 rows: 64-bit fragment loads conflict-free");
  static_assert(Q8 != 2 || (Q8_OFF % 16 == 0 && Q8_OFF >= KD), "int8 rows on 16 bytes, past the BF16 half");
  static constexpr int bytes(int) { return BYTES; }
  static constexpr int BYTES_MAX = BYTES;
  static_assert(LS_PITCH % 128 == 16, "lo rows must be conflict-free for ldmatrix");
};

// ---- Q8_0 weights on the BF16 MMA.
//
// Inside each 32-column block the MMA's k index is a permutation of the
// memory column, chosen so that the eight quants a thread needs of one row
// (both k-steps of the block) are eight consecutive bytes: lane (g, q) loads
// bytes 8q .. 8q + 7 of rows g and g + 8 with one 64-bit load each.  Column
// p = 8q + j of a block is MMA k
//   kperm(p) = 16 (j >> 2) + 8 (j & 1) + 2q + ((j >> 1) & 1),
// a bijection of 0..31; the activations are staged at kperm of their column,
// so every product pairs a weight with its own activation.
__device__ __forceinline__ int q8_kperm(int p) {
  const int q = (p >> 3) & 3, j = p & 7;
  return 16 * (j >> 2) + 8 * (j & 1) + 2 * q + ((j >> 1) & 1);
}

// The int8 values in bytes 0 and 2 of w as a BF16 pair (byte 0 low), exact:
// with m = b & 127 and s the sign bit, BF16 0x4300 | m is 128 + m and
// 0x4300 | (b & 128) is 128 or 256, so their difference is m - 128 s = b.
__device__ __forceinline__ uint32_t q8_bytes02(uint32_t w) {
  const uint32_t mag = (w & 0x007F007Fu) | 0x43004300u;
  const uint32_t sub = (w & 0x00800080u) | 0x43004300u;
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&mag),
                                   *reinterpret_cast<const __nv_bfloat162*>(&sub));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// A fragments of the two k-steps of one block from rows g and g + 8 (eight
// quants each, `r0` and `r1`): bytes 0, 2 / 1, 3 of the first word are
// k = 2q, 2q + 1 / 2q + 8, 2q + 9 of k-step 0; the second word the same for
// k-step 1 (kperm).
__device__ __forceinline__ void q8_afrags(const uint2 r0, const uint2 r1, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
  a0[0] = q8_bytes02(r0.x);
  a0[1] = q8_bytes02(r1.x);
  a0[2] = q8_bytes02(r0.x >> 8);
  a0[3] = q8_bytes02(r1.x >> 8);
  a1[0] = q8_bytes02(r0.y);
  a1[1] = q8_bytes02(r1.y);
  a1[2] = q8_bytes02(r0.y >> 8);
  a1[3] = q8_bytes02(r1.y >> 8);
}

// Stores the hi/lo split of four consecutive activations (columns p0 .. p0+3
// of a 32-column block, p0 % 4 == 0) into a staging row at their kperm
// positions: columns p0, p0 + 2 and p0 + 1, p0 + 3 are adjacent there.
__device__ __forceinline__ void q8_stage4(unsigned char* row_hi, unsigned char* row_lo, int block_col0, int p0,
                                          const float4 x) {
  uint2 hi, lo;
  split4(x, hi, lo);
  const int k02 = block_col0 + q8_kperm(p0);      // k of column p0; p0 + 2 follows it
  const int k13 = block_col0 + q8_kperm(p0 + 1);  // k of column p0 + 1; p0 + 3 follows it
  *reinterpret_cast<uint32_t*>(row_hi + 2 * k02) = __byte_perm(hi.x, hi.y, 0x5410);
  *reinterpret_cast<uint32_t*>(row_hi + 2 * k13) = __byte_perm(hi.x, hi.y, 0x7632);
  *reinterpret_cast<uint32_t*>(row_lo + 2 * k02) = __byte_perm(lo.x, lo.y, 0x5410);
  *reinterpret_cast<uint32_t*>(row_lo + 2 * k13) = __byte_perm(lo.x, lo.y, 0x7632);
}

// Q8_0 modes of the tensor-core kernels: 1 decodes the quants in registers
// inside the MMA loop (the layout above; fastest for one token group), 2
// widens the tile to BF16 once in shared memory right after it lands and
// runs the BF16 MMA loop with per-block scales (the second and later token
// groups reuse the widened tile: 4.9 -> 4.4-4.7 us per read at T = 5..8 on
// six streams, while one group measured 5 % slower than mode 1).  For mode 2
// the int8 rows land at byte Q8_OFF of the BF16 rows of the same tile.  Each
// row is widened in place: every lane loads its bytes of the row, the warp
// synchronises, then the lanes write the BF16 values from the row's start;
// rows do not overlap and inside a row all loads precede all stores.
// Widens ROWS int8 rows of COLS bytes (at byte `q8_off` of each row, rows
// `pitch` bytes apart) to BF16 at the start of the same rows.  Called by
// every thread of the CTA after the tile has landed; LANES_PER_ROW lanes
// take one row, each COLS / LANES_PER_ROW bytes (a multiple of 4).  A warp
// loads all its rows first, synchronises once, then stores them all.
template <int ROWS, int COLS, int LANES_PER_ROW>
__device__ __forceinline__ void q8_widen_rows(unsigned char* tile, int pitch, int q8_off, int warp, int lane) {
  constexpr int BPL = COLS / LANES_PER_ROW;  // bytes per lane
  constexpr int WPL = BPL / 4;               // words per lane
  constexpr int RPW = 32 / LANES_PER_ROW;    // rows per warp step
  constexpr int STEPS = ROWS / (kWarps * RPW);
  static_assert(COLS % LANES_PER_ROW == 0 && BPL % 4 == 0 && 32 % LANES_PER_ROW == 0, "whole words per lane");
  static_assert(ROWS % (kWarps * RPW) == 0, "every warp takes the same number of rows");
  const int sub = lane / LANES_PER_ROW, l = lane - sub * LANES_PER_ROW;
  uint32_t v[STEPS][WPL];
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const unsigned char* row = tile + (st * kWarps * RPW + warp * RPW + sub) * pitch;
#pragma unroll
    for (int i = 0; i < WPL; ++i) v[st][i] = *reinterpret_cast<const uint32_t*>(row + q8_off + BPL * l + 4 * i);
  }
  __syncwarp();
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    unsigned char* row = tile + (st * kWarps * RPW + warp * RPW + sub) * pitch;
#pragma unroll
    for (int i = 0; i < WPL; ++i) {
      *reinterpret_cast<uint2*>(row + 2 * (BPL * l + 4 * i)) =
          make_uint2(q8_bytes02(__byte_perm(v[st][i], 0, 0x4140)), q8_bytes02(__byte_perm(v[st][i], 0, 0x4342)));
    }
  }
}

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
template <int D, int KD, int NT, int Q8 = 0>
__global__ void __launch_bounds__(kThreads, tc_min_blocks<D, NT>()) hc_down_tc_kernel(const DownArgs a) {
  using G = Geo<D, KD>;
  using S = DownTcSmem<D, KD, NT, Q8>;
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

  const uint64_t t_entry = ptx::globaltimer_ns();
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  float* recv_ss = cluster.map_shared_rank(reinterpret_cast<float*>(smem + S::RECV), 0);
  float* recv_p = recv_ss + 4 * T;

  ptx::cluster_arrive_relaxed();
  constexpr int WROW = Q8 ? G::SLAB : G::SLAB * 2;  // bytes of one W_down row of the slab
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::fence_barrier_init();
      ptx::mbar_arrive_expect_tx(bar_w, (!Q8 && a.W_tiles) ? G::DN_ROWS * S::WPITCH : G::DN_ROWS * WROW);
    }
    __syncwarp();
    const uint64_t once = ptx::policy_evict_first();
    if (Q8 || a.W_tiles == nullptr) {
      const void* src = Q8 ? static_cast<const void*>(a.Wq + (size_t)(row0 + lane) * G::N + col0)
                           : static_cast<const void*>(a.W_down + (size_t)(row0 + lane) * G::N + col0);
      ptx::bulk_g2s(w_s + lane * S::WPITCH + S::Q8_OFF, src, WROW, bar_w, once);
    } else if (lane < kTileCopies) {
      static_assert(Q8 || S::WPITCH == G::DN_PITCH, "BF16 tiles at the tile order's pitch");
      copy_down_tile<G>(w_s, a.W_tiles, rg, slab, lane, bar_w, once);
    }
  }
  if constexpr (Q8) {
    // The slab's block scales of the CTA's 32 rows (binary16), copied
    // asynchronously: waited for with the weight tile, before the MMAs.
    constexpr int PIECES = S::NB / 4;  // 8-byte pieces per row
    for (int idx = tid; idx < G::DN_ROWS * PIECES; idx += kThreads) {
      const int r = idx / PIECES, c = idx - r * PIECES;
      ptx::cp_async8(smem + S::SC + (r * S::NB + 4 * c) * 2,
                     a.Wscale + (size_t)(row0 + r) * (G::N / 32) + col0 / 32 + 4 * c);
    }
  }
  // This thread's float4 of the w_norm slab goes straight to registers (it is
  // not written by the previous kernel): no shared copy, no barrier.
  const int c4 = tid;  // one float4 of the slab per thread and token
  static_assert(G::DN_F4 <= kThreads, "one float4 per thread and token");
  const float4 wn = c4 < G::DN_F4 ? __ldg(reinterpret_cast<const float4*>(a.w_norm + col0) + c4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
  // Late launch of the up kernel for independent reads of one token group
  // on the batch lanes, as in hc_down_kernel.
  const bool late_launch = a.late_launch && a.independent && a.T <= TG;
  if (!late_launch) ptx::launch_dependents();
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
  const uint32_t a_base = ptx::smem_u32(w_s + a_row * S::WPITCH + a_col * 2);
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
        if constexpr (Q8 == 1) {
          q8_stage4(xs + (2 * t) * S::XS_PITCH, xs + (2 * t + 1) * S::XS_PITCH, (4 * c4) & ~31, (4 * c4) & 31, x);
        } else {
          uint2 hi, lo;
          split4(x, hi, lo);  // tokens past tg carry zeros
          *reinterpret_cast<uint2*>(xs + (2 * t) * S::XS_PITCH + c4 * 8) = hi;
          *reinterpret_cast<uint2*>(xs + (2 * t + 1) * S::XS_PITCH + c4 * 8) = lo;
        }
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
    if (t0 == 0) {
      ok = wait_bar_from(bar_w, 0, a.err, kErrDownWeights, t_entry, first_wait_limit(a.wait_ns)) && ok;
      if constexpr (Q8 != 0) ptx::cp_async_wait_all();
      if constexpr (Q8 == 2) q8_widen_rows<G::DN_ROWS, G::SLAB, 32>(w_s, S::WPITCH, S::Q8_OFF, warp, lane);
    }
    __syncthreads();  // x (hi, lo), the per-warp sums of squares (and a widened tile) are complete
    if (tid < tg) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += ssw_s[w * TG + tid];
      recv_ss[rank * T + t0 + tid] = v;
    }

    // One k-step of 16 columns: B rows from the x staging, MMA into cc.
    auto kstep = [&](int ks, const uint32_t(&af)[4], float(&cc)[NT][4]) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3;
        if (n + 1 < NT) {
          ptx::ldsm_x4(ptx::smem_u32(xs + (n * 8 + b_row) * S::XS_PITCH + (b_col + ks * 16) * 2), b0, b1,
                       b2, b3);
          ptx::mma_bf16_16816(cc[n], af, b0, b1);
          ptx::mma_bf16_16816(cc[n + 1], af, b2, b3);
        } else {
          ptx::ldsm_x2(ptx::smem_u32(xs + (n * 8 + (lane & 7)) * S::XS_PITCH + (b_col + ks * 16) * 2), b0,
                       b1);
          ptx::mma_bf16_16816(cc[n], af, b0, b1);
        }
      }
    };
    // The two k-steps of one Q8_0 block into cc, started at zero.
    auto kstep_q8 = [&](int ks, const uint32_t(&a0)[4], const uint32_t(&a1)[4], float(&cc)[NT][4]) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
        if (n + 1 < NT) {
          ptx::ldsm_x4(ptx::smem_u32(xs + (n * 8 + b_row) * S::XS_PITCH + (b_col + ks * 16) * 2), b0, b1, b2, b3);
          ptx::ldsm_x4(ptx::smem_u32(xs + (n * 8 + b_row) * S::XS_PITCH + (b_col + ks * 16 + 16) * 2), c0, c1, c2,
                       c3);
          ptx::mma_bf16_16816_zero(cc[n], a0, b0, b1);
          ptx::mma_bf16_16816_zero(cc[n + 1], a0, b2, b3);
          ptx::mma_bf16_16816(cc[n], a1, c0, c1);
          ptx::mma_bf16_16816(cc[n + 1], a1, c2, c3);
        } else {
          ptx::ldsm_x2(ptx::smem_u32(xs + (n * 8 + (lane & 7)) * S::XS_PITCH + (b_col + ks * 16) * 2), b0, b1);
          ptx::ldsm_x2(ptx::smem_u32(xs + (n * 8 + (lane & 7)) * S::XS_PITCH + (b_col + ks * 16 + 16) * 2), c0, c1);
          ptx::mma_bf16_16816_zero(cc[n], a0, b0, b1);
          ptx::mma_bf16_16816(cc[n], a1, c0, c1);
        }
      }
    };
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    if constexpr (!Q8) {
      // Two accumulator sets (even and odd k-steps), added at the end: half
      // the dependent-MMA chain, a fixed order.
      float acc2[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) acc2[n][0] = acc2[n][1] = acc2[n][2] = acc2[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t afrag[4];
        ptx::ldsm_x4(a_base + ks * 32, afrag[0], afrag[1], afrag[2], afrag[3]);
        kstep(ks, afrag, (ks & 1) ? acc2 : acc);
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = __fadd_rn(acc[n][e], acc2[n][e]);
      }
    } else {
      // Q8_0: each 32-column block (two k-steps into one accumulator started
      // at zero) is scaled by its rows' block scales and added, blocks in
      // order.
      const int g = lane >> 2, q = lane & 3;
      const unsigned char* qa = w_s + (mt * 16 + g) * S::WPITCH + kp * KPART + 8 * q;
      const __half* sc = reinterpret_cast<const __half*>(smem + S::SC) + (mt * 16 + g) * S::NB + kp * (KPART / 32);
#pragma unroll 2  // fully unrolled, the 64-register variants spill
      for (int bk = 0; bk < KS / 2; ++bk) {
        uint32_t a0[4], a1[4];
        if constexpr (Q8 == 1) {
          q8_afrags(*reinterpret_cast<const uint2*>(qa + 32 * bk),
                    *reinterpret_cast<const uint2*>(qa + 8 * S::WPITCH + 32 * bk), a0, a1);
        } else {
          ptx::ldsm_x4(a_base + (2 * bk) * 32, a0[0], a0[1], a0[2], a0[3]);
          ptx::ldsm_x4(a_base + (2 * bk + 1) * 32, a1[0], a1[1], a1[2], a1[3]);
        }
        float blk[NT][4];
        kstep_q8(2 * bk, a0, a1, blk);
        const float s0 = __half2float(sc[bk]), s1 = __half2float(sc[8 * S::NB + bk]);  // rows g and g + 8
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          acc[n][0] = __fmaf_rn(s0, blk[n][0], acc[n][0]);
          acc[n][1] = __fmaf_rn(s0, blk[n][1], acc[n][1]);
          acc[n][2] = __fmaf_rn(s1, blk[n][2], acc[n][2]);
          acc[n][3] = __fmaf_rn(s1, blk[n][3], acc[n][3]);
        }
      }
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
  if (late_launch) ptx::launch_dependents();
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
template <int D, int KD, int NT, int Q8 = 0>
__global__ void __launch_bounds__(kThreads, tc_min_blocks<D, NT>()) hc_up_tc_kernel(const UpArgs a) {
  using G = Geo<D, KD>;
  using S = UpTcSmem<D, KD, NT, Q8>;
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
      ptx::mbar_arrive_expect_tx(bar_w, G::UP_ROWS * KD * (Q8 ? 1 : 2));
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
      if constexpr (Q8) {
        ptx::bulk_g2s(w_s + r * S::WPITCH + S::Q8_OFF, a.Wq + (size_t)grow * KD, KD, bar_w, once);
      } else {
        ptx::bulk_g2s(w_s + r * S::WPITCH, a.W_up + (size_t)grow * KD, KD * 2, bar_w, once);
      }
    }
  }
  if constexpr (Q8) {
    // The block scales of the CTA's 64 rows (binary16), copied
    // asynchronously: waited for with the weight tile, before the MMAs.
    constexpr int PIECES = G::UP_COLS * S::NB * 2 / 16;  // 16-byte pieces per stream
    for (int idx = tid; idx < kStreams * PIECES; idx += kThreads) {
      const int st = idx / PIECES, c = idx - st * PIECES;
      ptx::cp_async16(smem + S::SC + st * G::UP_COLS * S::NB * 2 + 16 * c,
                      reinterpret_cast<const unsigned char*>(a.Wscale + ((size_t)st * D + c0) * S::NB) + 16 * c);
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
  const uint32_t a_base = ptx::smem_u32(w_s + a_row * S::WPITCH + a_col * 2);
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
        if constexpr (Q8 == 1) {
          q8_stage4(ls + (2 * t) * S::LS_PITCH, ls + (2 * t + 1) * S::LS_PITCH, (4 * k4) & ~31, (4 * k4) & 31, l);
        } else {
          uint2 hi, lo;
          split4(l, hi, lo);  // tokens past tg carry zeros
          *reinterpret_cast<uint2*>(ls + (2 * t) * S::LS_PITCH + k4 * 8) = hi;
          *reinterpret_cast<uint2*>(ls + (2 * t + 1) * S::LS_PITCH + k4 * 8) = lo;
        }
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
    if (t0 == 0) {
      ok = wait_bar(bar_w, 0, a.err, kErrUpWeights) && ok;
      if constexpr (Q8 != 0) ptx::cp_async_wait_all();
      if constexpr (Q8 == 2) q8_widen_rows<G::UP_ROWS, KD, 16>(w_s, S::WPITCH, S::Q8_OFF, warp, lane);
    }
    __syncthreads();  // lo (hi, lo), R', the gates (and a widened tile) are in shared memory

    // One k-step of 16 along K: B rows from the lo staging, MMA into cc.
    auto kstep = [&](int ks, const uint32_t(&af)[4], float(&cc)[NT][4]) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3;
        if (n + 1 < NT) {
          ptx::ldsm_x4(ptx::smem_u32(ls + (n * 8 + b_row) * S::LS_PITCH + (b_col + ks * 16) * 2), b0, b1,
                       b2, b3);
          ptx::mma_bf16_16816(cc[n], af, b0, b1);
          ptx::mma_bf16_16816(cc[n + 1], af, b2, b3);
        } else {
          ptx::ldsm_x2(ptx::smem_u32(ls + (n * 8 + (lane & 7)) * S::LS_PITCH + (b_col + ks * 16) * 2), b0,
                       b1);
          ptx::mma_bf16_16816(cc[n], af, b0, b1);
        }
      }
    };
    // The two k-steps of one Q8_0 block into cc, started at zero.
    auto kstep_q8 = [&](int ks, const uint32_t(&a0)[4], const uint32_t(&a1)[4], float(&cc)[NT][4]) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
        if (n + 1 < NT) {
          ptx::ldsm_x4(ptx::smem_u32(ls + (n * 8 + b_row) * S::LS_PITCH + (b_col + ks * 16) * 2), b0, b1, b2, b3);
          ptx::ldsm_x4(ptx::smem_u32(ls + (n * 8 + b_row) * S::LS_PITCH + (b_col + ks * 16 + 16) * 2), c0, c1, c2,
                       c3);
          ptx::mma_bf16_16816_zero(cc[n], a0, b0, b1);
          ptx::mma_bf16_16816_zero(cc[n + 1], a0, b2, b3);
          ptx::mma_bf16_16816(cc[n], a1, c0, c1);
          ptx::mma_bf16_16816(cc[n + 1], a1, c2, c3);
        } else {
          ptx::ldsm_x2(ptx::smem_u32(ls + (n * 8 + (lane & 7)) * S::LS_PITCH + (b_col + ks * 16) * 2), b0, b1);
          ptx::ldsm_x2(ptx::smem_u32(ls + (n * 8 + (lane & 7)) * S::LS_PITCH + (b_col + ks * 16 + 16) * 2), c0, c1);
          ptx::mma_bf16_16816_zero(cc[n], a0, b0, b1);
          ptx::mma_bf16_16816(cc[n], a1, c0, c1);
        }
      }
    };
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    if constexpr (!Q8) {
      // Two accumulator sets (even and odd k-steps), added at the end: half
      // the dependent-MMA chain, a fixed order.
      float acc2[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) acc2[n][0] = acc2[n][1] = acc2[n][2] = acc2[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t afrag[4];
        ptx::ldsm_x4(a_base + ks * 32, afrag[0], afrag[1], afrag[2], afrag[3]);
        kstep(ks, afrag, (ks & 1) ? acc2 : acc);
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = __fadd_rn(acc[n][e], acc2[n][e]);
      }
    } else {
      // Q8_0: each 32-wide block of K (two k-steps into one accumulator
      // started at zero) is scaled by its rows' block scales and added,
      // blocks in order.
      const int g = lane >> 2, q = lane & 3;
      const unsigned char* qa = w_s + (mt * 16 + g) * S::WPITCH + kh * KHALF + 8 * q;
      const __half* sc = reinterpret_cast<const __half*>(smem + S::SC) + (mt * 16 + g) * S::NB + kh * (KHALF / 32);
#pragma unroll 2  // fully unrolled, the 64-register variants spill
      for (int bk = 0; bk < KS / 2; ++bk) {
        uint32_t a0[4], a1[4];
        if constexpr (Q8 == 1) {
          q8_afrags(*reinterpret_cast<const uint2*>(qa + 32 * bk),
                    *reinterpret_cast<const uint2*>(qa + 8 * S::WPITCH + 32 * bk), a0, a1);
        } else {
          ptx::ldsm_x4(a_base + (2 * bk) * 32, a0[0], a0[1], a0[2], a0[3]);
          ptx::ldsm_x4(a_base + (2 * bk + 1) * 32, a1[0], a1[1], a1[2], a1[3]);
        }
        float blk[NT][4];
        kstep_q8(2 * bk, a0, a1, blk);
        const float s0 = __half2float(sc[bk]), s1 = __half2float(sc[8 * S::NB + bk]);  // rows g and g + 8
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          acc[n][0] = __fmaf_rn(s0, blk[n][0], acc[n][0]);
          acc[n][1] = __fmaf_rn(s0, blk[n][1], acc[n][1]);
          acc[n][2] = __fmaf_rn(s1, blk[n][2], acc[n][2]);
          acc[n][3] = __fmaf_rn(s1, blk[n][3], acc[n][3]);
        }
      }
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
