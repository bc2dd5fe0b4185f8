// Q2_0 matrix-vector product (include/hc_q2.h): kernel and C ABI.
//
// y[c][r] = sum_j W[r][j] x[c][j] over Q2_0 weights, 1..4 columns: the QSA
// layers' attn_q projection of the decode windows (Strata pull request
// #2221, first paragraph and its kernel table: 2560 -> 12288, one to four
// columns, cold weights).
//
// Arithmetic.  The weights are the only large operand (2.25 bits a value), so
// the decoding has to cost less than the bytes.  A two-bit code q masked out
// of its 32-bit word in place, (w & (3 << 2j)), is the bit pattern of the IEEE
// binary16 subnormal q * 4^j * 2^-24, exact; the tensor cores take subnormal
// binary16 operands exactly.  So one AND per two codes gives the MMA's A
// operand (mma.sync m16n8k16, binary16 in, FP32 accumulate) with no offset to
// remove, if the B operand carries x * 4^-j for the k-slots of bit position j
// (codes at bits 0..9 of a 16-bit half take j = 0..4, bits 10..15 after one
// shift j = 0..2).  The MMA then sums 2^-24 * q * x; the -2 of the weight
// d * (q - 2) is a constant of each 64-value block and column, -2^-23 * sum(x),
// which seeds the accumulator.  x is scaled per column by a power of two that
// brings max|x| to [2^13, 2^14) and split into two binary16 terms, hi and lo
// (B columns 2c and 2c + 1): 22 significant bits.  Each block's sum is
// multiplied by the block's scale and added to the row's FP32 total; powers
// of two undo the scalings at the end.
//
// Schedule.  One persistent launch takes up to kLaunchProducts products of
// one shape that share no memory; their 32-row tiles form one list (product
// major) and CTA i takes tiles i, i + G, ... (G CTAs, as many as the device
// holds at once).  A tile is 32 rows x all columns: warp w takes rows
// 16 (w % 2) + g and + 8 over the (w / 2)-th quarter of the blocks, and the
// four quarters are added in a fixed order through shared memory.  The codes
// and scales of the next kStages - 1 tiles stream into a ring of shared-memory
// stages with cp.async while one tile is computed.  x is split into the B
// layout when a tile's product has another x than the tile before, so a
// batch over one x splits it once per CTA.
//
// Value order inside a block: MMA lane (g, t) (g = lane / 4, t = lane % 4)
// holds the 32-bit word t of the block for rows g and g + 8, values
// 16t .. 16t + 15; bits p and 16 + p of the word (values 16t + p/2 and
// 16t + 8 + p/2) form one binary16x2 register, pair i = p/2.  The B fragment
// of the same lane carries (x[16t + i], x[16t + 8 + i]) for the same i, so the
// MMA's k order is a permutation of the block's values that A and B share.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "hc_ptx.cuh"
#include "hc_q2.h"

#define HC_EXPORT extern "C" __attribute__((visibility("default")))

namespace hc {
namespace q2 {

constexpr int kThreads = 256;         // 8 warps (their split of a tile: the KPB template below)
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 32;             // rows of one tile
constexpr int kStages = 3;            // tiles in flight per CTA (one computed, two loading)
constexpr int kMinCols = 512;         // a quarter of a row is an even number of 64-value blocks
constexpr int kMaxCols = 4096;
constexpr int kMaxNcols = 4;
constexpr int kMaxRows = 1 << 24;
constexpr int kLaunchProducts = 120;  // products per launch (kernel parameters under 4 KB)
constexpr int kTarget = 13;           // x is scaled so that max|x| lies in [2^13, 2^14)

struct Product {
  const uint8_t* Wq;
  const uint16_t* Ws;
  const float* x;
  float* y;
};

struct Args {
  Product p[kLaunchProducts];
  int count;  // products in this launch
  int rows;
  int cols;
  int tiles;  // tiles of one product
};

// Shared-memory layout of one CTA for `cols` columns and NC input columns.
struct Layout {
  int nb;           // 64-value blocks of a row
  int code_pitch;   // bytes between rows of a code tile
  int scale_pitch;  // bytes between rows of a scale tile
  int stage;        // bytes of one stage (codes, then scales)
  int scales, xs, kb, wmax, red, bytes;
  __host__ __device__ Layout(int cols, int nc, int parts) {
    nb = cols / 64;
    // cols / 4 code bytes a row plus 16: the pitch in words is 4 * odd, so the
    // eight rows g of an MMA fragment fall on eight different groups of four
    // banks.
    code_pitch = cols / 4 + 16;
    scale_pitch = cols / 32;
    scales = kRows * code_pitch;
    stage = scales + kRows * scale_pitch;
    xs = kStages * stage;                  // [nb][2 halves][2 nc][4][16 B] binary16x2
    kb = xs + nb * 2 * (2 * nc) * 4 * 16;  // [nb][nc] float: accumulator seeds
    wmax = kb + nb * nc * 4;               // [8 warps][nc] float: max|x| per warp
    red = wmax + kWarps * nc * 4;          // [parts][32 rows][nc] float
    bytes = red + parts * kRows * nc * 4;
  }
};

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// D(16x8, fp32) = A(16x16, binary16, row) * B(16x8, binary16, col) + C.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                        float c0, float c1, float c2, float c3) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  mma_f16(d, a, b0, b1, d[0], d[1], d[2], d[3]);
}

// The eight A registers of one code word: pair i holds the codes at bits 2i
// and 16 + 2i (i < 5) or 2i of w >> 10 (i >= 5), as binary16 subnormals.
__device__ __forceinline__ void q2_decode(uint32_t w, uint32_t (&p)[8]) {
  const uint32_t w10 = w >> 10;
  p[0] = w & 0x00030003u;
  p[1] = w & 0x000C000Cu;
  p[2] = w & 0x00300030u;
  p[3] = w & 0x00C000C0u;
  p[4] = w & 0x03000300u;
  p[5] = w10 & 0x00030003u;
  p[6] = w10 & 0x000C000Cu;
  p[7] = w10 & 0x00300030u;
}

// 4^-j of pair i's bit position.
__device__ __forceinline__ float pair_factor(int i) {
  const int j = i < 5 ? i : i - 5;
  return __uint_as_float(static_cast<uint32_t>(127 - 2 * j) << 23);
}

// 2^e for -126 <= e <= 127.
__device__ __forceinline__ float pow2(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Two values as binary16x2 hi terms and lo terms (v = hi + lo to 22 bits),
// first value in the low half.
__device__ __forceinline__ void split_pair(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(v0, v1);
  const __half2 l = __floats2half2_rn(__fsub_rn(v0, __low2float(h)), __fsub_rn(v1, __high2float(h)));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Copy `pieces` 16-byte pieces of each of the first min(valid, kRows) rows at
// src (row stride src_pitch) to dst (row stride dst_pitch) with cp.async.
__device__ __forceinline__ void copy_rows(uint8_t* dst, int dst_pitch, const uint8_t* src, size_t src_pitch,
                                          int pieces, int valid, int warp, int lane) {
  const int rows = valid < kRows ? valid : kRows;
  if (pieces <= 32) {
    const int per = 32 / pieces;  // rows a warp copies at a time
    const int lr = lane / pieces, lc = lane - lr * pieces;
    if (lr >= per) return;
    for (int r = warp * per + lr; r < rows; r += kWarps * per) {
      ptx::cp_async16(dst + r * dst_pitch + 16 * lc, src + r * src_pitch + 16 * lc);
    }
  } else {
    for (int r = warp; r < rows; r += kWarps) {
      for (int c = lane; c < pieces; c += 32) ptx::cp_async16(dst + r * dst_pitch + 16 * c, src + r * src_pitch + 16 * c);
    }
  }
}

// A position in a CTA's list of tiles: tile r of product p.
struct Cursor {
  int p, r;
  __device__ void next(int step, int tiles) {
    r += step;
    while (r >= tiles) {
      r -= tiles;
      ++p;
    }
  }
};

// KPB > 0: the form for cols = 512 * KPB in which warp w takes both row
// groups over the w-th eighth of the blocks (KPB blocks) and keeps that
// eighth of x's B layout in registers for as long as x stays the same.
// KPB = 0: any width; warp w takes one row group over a quarter of the
// blocks and reads the B layout from shared memory.
template <int NC, int KPB>
__global__ void __launch_bounds__(kThreads, 2) hc_q2_matvec_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int kParts = KPB > 0 ? kWarps : 4;  // partial sums per row
  const Layout L(a.cols, NC, kParts);
  uint4* xs = reinterpret_cast<uint4*>(smem + L.xs);
  float* kb = reinterpret_cast<float*>(smem + L.kb);
  float* wmax = reinterpret_cast<float*>(smem + L.wmax);
  float* red = reinterpret_cast<float*>(smem + L.red);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int total = a.count * a.tiles;
  const int step = gridDim.x;
  const int bid = blockIdx.x;
  const int n_items = bid < total ? (total - bid + step - 1) / step : 0;
  const int nb = L.nb;

  auto issue = [&](const Cursor& c, int k) {
    const Product& pr = a.p[c.p];
    uint8_t* st = smem + (k % kStages) * L.stage;
    const int row0 = c.r * kRows;
    const size_t row_bytes = static_cast<size_t>(a.cols) / 4;
    copy_rows(st, L.code_pitch, pr.Wq + static_cast<size_t>(row0) * row_bytes, row_bytes, a.cols / 64,
              a.rows - row0, warp, lane);
    const size_t srow = static_cast<size_t>(a.cols) / 32;
    copy_rows(st + L.scales, L.scale_pitch, reinterpret_cast<const uint8_t*>(pr.Ws) + static_cast<size_t>(row0) * srow,
              srow, a.cols / 512, a.rows - row0, warp, lane);
  };
  const Cursor first{bid / a.tiles, bid % a.tiles};

  // Weights of the first tiles before the wait (they do not depend on
  // earlier kernels); x is read and y written after it.
  Cursor is = first;
  for (int k = 0; k < kStages - 1; ++k) {
    if (k < n_items) {
      issue(is, k);
      is.next(step, a.tiles);
    }
    cp_async_commit();
  }
  ptx::wait_prerequisites();
  ptx::launch_dependents();

  // Warp w: rows 16 rg + g and + 8 of a tile, blocks [kq nq, (kq + 1) nq)
  // (KPB = 0); or all 32 rows, blocks [w KPB, (w + 1) KPB).
  const int rg = KPB > 0 ? 0 : warp & 1, kq = KPB > 0 ? warp : warp >> 1;
  const int nq = KPB > 0 ? KPB : nb / 4, b0 = kq * nq;
  constexpr int kRegBlocks = KPB > 0 ? KPB : 1;
  uint4 breg_l[kRegBlocks], breg_h[kRegBlocks];  // B fragments of this warp's blocks (KPB > 0)
  float sreg[kRegBlocks];                         // their accumulator seeds
  const int co = (16 * rg + g) * L.code_pitch + 4 * t + 16 * b0;
  const int so = (16 * rg + g) * L.scale_pitch + 2 * b0;
  const bool has_b = g < 2 * NC;  // B columns past 2 NC are zero
  const uint4* bp = xs + g * 4 + t + (2 * b0) * (8 * NC);
  const float* kp = kb + b0 * NC + t;

  Cursor cs = first;
  const float* staged = nullptr;  // the x now in the B layout
  float unscale[NC];              // 2^-s of column c's scale 2^s
#pragma unroll
  for (int c = 0; c < NC; ++c) unscale[c] = 0.f;
  for (int k = 0; k < n_items; ++k) {
    if (k + kStages - 1 < n_items) {
      issue(is, k + kStages - 1);
      is.next(step, a.tiles);
    }
    cp_async_commit();
    cp_async_wait_group<kStages - 1>();
    __syncthreads();
    const Product& pr = a.p[cs.p];
    if (pr.x != staged) {
      // Scale of each column: 2^(13 - e) with 2^e <= max|x| < 2^(e + 1).
      const float* x = pr.x;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float m = 0.f;
        for (int i = tid; i < a.cols / 4; i += kThreads) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(x + static_cast<size_t>(c) * a.cols) + i);
          m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wmax[warp * NC + c] = m;
      }
      __syncthreads();
      float scale[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float m = wmax[c];
        for (int w = 1; w < kWarps; ++w) m = fmaxf(m, wmax[w * NC + c]);
        const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;
        const int s = kTarget - e < -126 ? -126 : (kTarget - e > 126 ? 126 : kTarget - e);
        scale[c] = pow2(s);
        unscale[c] = pow2(-s);
      }
      // The B layout: item (b, c, h, tt) holds the pairs (x[16 tt + i],
      // x[16 tt + 8 + i]) * scale * 4^-j(i), i = 4h .. 4h + 3, of block b,
      // column c, as hi terms (B column 2c) and lo terms (B column 2c + 1);
      // the eight items of a block and column sit in eight adjacent lanes,
      // which add their scaled values for the block's accumulator seed.
      for (int i = tid; i < nb * NC * 8; i += kThreads) {
        const int tt = i & 3, h = (i >> 2) & 1;
        const int rest = i >> 3;
        const int c = rest % NC, b = rest / NC;
        const float* xp = x + static_cast<size_t>(c) * a.cols + b * 64 + 16 * tt + 4 * h;
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(xp));
        const float4 v1 = __ldg(reinterpret_cast<const float4*>(xp + 8));
        float sc = scale[0];
#pragma unroll
        for (int cc = 1; cc < NC; ++cc) sc = c == cc ? scale[cc] : sc;
        const float r0[4] = {v0.x, v0.y, v0.z, v0.w}, r1[4] = {v1.x, v1.y, v1.z, v1.w};
        // powers of two: the sums and products below are the ones of the
        // scaled values, exactly
        float sum = 0.f;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          sum = __fadd_rn(sum, __fadd_rn(r0[u], r1[u]));
          const float f = __fmul_rn(sc, pair_factor(4 * h + u));
          split_pair(__fmul_rn(r0[u], f), __fmul_rn(r1[u], f), hi[u], lo[u]);
        }
        sum = __fmul_rn(sum, sc);
        uint4* plane = xs + (b * 2 + h) * (8 * NC);
        plane[(2 * c) * 4 + tt] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        plane[(2 * c + 1) * 4 + tt] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        // lanes 8m .. 8m + 7 hold the eight items of one (b, c)
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 1));
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 2));
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 4));
        if ((i & 7) == 0) kb[b * NC + c] = __fmul_rn(sum, -0x1.0p-23f);
      }
      staged = pr.x;
      __syncthreads();
      if constexpr (KPB > 0) {
#pragma unroll
        for (int b = 0; b < KPB; ++b) {
          breg_l[b] = has_b ? bp[(2 * b) * (8 * NC)] : make_uint4(0u, 0u, 0u, 0u);
          breg_h[b] = has_b ? bp[(2 * b + 1) * (8 * NC)] : make_uint4(0u, 0u, 0u, 0u);
          sreg[b] = t < NC ? kp[b * NC] : 0.f;
        }
      }
    }

    const uint8_t* st = smem + (k % kStages) * L.stage;
    if constexpr (KPB > 0) {
      // rows g, g + 8 (chain 0) and 16 + g, 24 + g (chain 1)
      const uint8_t* c0 = st + co;
      const int sp = L.scale_pitch / 2;  // halves between scale rows
      const __half* s0 = reinterpret_cast<const __half*>(st + L.scales + so);
      float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll
      for (int b = 0; b < KPB; ++b) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(c0 + 16 * b);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(c0 + 8 * L.code_pitch + 16 * b);
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(c0 + 16 * L.code_pitch + 16 * b);
        const uint32_t w3 = *reinterpret_cast<const uint32_t*>(c0 + 24 * L.code_pitch + 16 * b);
        uint32_t p0[8], p1[8], p2[8], p3[8];
        q2_decode(w0, p0);
        q2_decode(w1, p1);
        q2_decode(w2, p2);
        q2_decode(w3, p3);
        const uint4 bl = breg_l[b], bh = breg_h[b];
        const float seed = sreg[b];
        float d[4], e[4];
        const uint32_t a0[4] = {p0[0], p1[0], p0[1], p1[1]};
        const uint32_t f0[4] = {p2[0], p3[0], p2[1], p3[1]};
        mma_f16(d, a0, bl.x, bl.y, seed, 0.f, seed, 0.f);
        mma_f16(e, f0, bl.x, bl.y, seed, 0.f, seed, 0.f);
        const uint32_t a1[4] = {p0[2], p1[2], p0[3], p1[3]};
        const uint32_t f1[4] = {p2[2], p3[2], p2[3], p3[3]};
        mma_f16(d, a1, bl.z, bl.w);
        mma_f16(e, f1, bl.z, bl.w);
        const uint32_t a2[4] = {p0[4], p1[4], p0[5], p1[5]};
        const uint32_t f2[4] = {p2[4], p3[4], p2[5], p3[5]};
        mma_f16(d, a2, bh.x, bh.y);
        mma_f16(e, f2, bh.x, bh.y);
        const uint32_t a3[4] = {p0[6], p1[6], p0[7], p1[7]};
        const uint32_t f3[4] = {p2[6], p3[6], p2[7], p3[7]};
        mma_f16(d, a3, bh.z, bh.w);
        mma_f16(e, f3, bh.z, bh.w);
        t0 = __fmaf_rn(__half2float(s0[b]), __fadd_rn(d[0], d[1]), t0);
        t1 = __fmaf_rn(__half2float(s0[8 * sp + b]), __fadd_rn(d[2], d[3]), t1);
        t2 = __fmaf_rn(__half2float(s0[16 * sp + b]), __fadd_rn(e[0], e[1]), t2);
        t3 = __fmaf_rn(__half2float(s0[24 * sp + b]), __fadd_rn(e[2], e[3]), t3);
      }
      if (t < NC) {
        red[(kq * kRows + g) * NC + t] = t0;
        red[(kq * kRows + g + 8) * NC + t] = t1;
        red[(kq * kRows + g + 16) * NC + t] = t2;
        red[(kq * kRows + g + 24) * NC + t] = t3;
      }
    } else {
      const uint8_t* c0 = st + co;
      const uint8_t* c1 = c0 + 8 * L.code_pitch;
      const __half* s0 = reinterpret_cast<const __half*>(st + L.scales + so);
      const __half* s1 = reinterpret_cast<const __half*>(st + L.scales + so + 8 * L.scale_pitch);
      float tot0 = 0.f, tot1 = 0.f;
#pragma unroll 2
      for (int b = 0; b < nq; ++b) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(c0 + 16 * b);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(c1 + 16 * b);
        uint4 bl = make_uint4(0u, 0u, 0u, 0u), bh = bl;
        float seed = 0.f;
        if (has_b) {
          bl = bp[(2 * b) * (8 * NC)];
          bh = bp[(2 * b + 1) * (8 * NC)];
        }
        if (t < NC) seed = kp[b * NC];
        uint32_t p0[8], p1[8];
        q2_decode(w0, p0);
        q2_decode(w1, p1);
        float d[4];
        const uint32_t a0[4] = {p0[0], p1[0], p0[1], p1[1]};
        mma_f16(d, a0, bl.x, bl.y, seed, 0.f, seed, 0.f);
        const uint32_t a1[4] = {p0[2], p1[2], p0[3], p1[3]};
        mma_f16(d, a1, bl.z, bl.w);
        const uint32_t a2[4] = {p0[4], p1[4], p0[5], p1[5]};
        mma_f16(d, a2, bh.x, bh.y);
        const uint32_t a3[4] = {p0[6], p1[6], p0[7], p1[7]};
        mma_f16(d, a3, bh.z, bh.w);
        // d[0], d[1]: row g, column t (hi and lo terms); d[2], d[3]: row g + 8.
        tot0 = __fmaf_rn(__half2float(s0[b]), __fadd_rn(d[0], d[1]), tot0);
        tot1 = __fmaf_rn(__half2float(s1[b]), __fadd_rn(d[2], d[3]), tot1);
      }
      if (t < NC) {
        red[(kq * kRows + 16 * rg + g) * NC + t] = tot0;
        red[(kq * kRows + 16 * rg + g + 8) * NC + t] = tot1;
      }
    }
    __syncthreads();
    if (tid < kRows * NC) {
      const int i = tid / NC, c = tid - i * NC;
      float s = red[i * NC + c];
#pragma unroll
      for (int m = 1; m < kParts; ++m) s = __fadd_rn(s, red[(m * kRows + i) * NC + c]);
      float u = unscale[0];
#pragma unroll
      for (int cc = 1; cc < NC; ++cc) u = c == cc ? unscale[cc] : u;
      const int r = cs.r * kRows + i;
      if (r < a.rows) pr.y[static_cast<size_t>(c) * a.rows + r] = __fmul_rn(__fmul_rn(s, 0x1.0p24f), u);
    }
    cs.next(step, a.tiles);
  }
  cp_async_wait_group<0>();
}

// CTAs of one launch: as many as can run at once (the kernel is persistent),
// at most one per tile.
template <int NC, int KPB>
cudaError_t launch(const Args& a, cudaStream_t st) {
  static std::once_flag once[64];
  static cudaError_t configured[64];
  static int per_sm[64][kMaxCols / kMinCols + 1];
  static int sms[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    configured[dev] = cudaFuncSetAttribute(hc_q2_matvec_kernel<NC, KPB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Layout(kMaxCols, NC, KPB > 0 ? kWarps : 4).bytes);
    if (configured[dev] == cudaSuccess)
      configured[dev] = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    for (int i = 0; i <= kMaxCols / kMinCols; ++i) per_sm[dev][i] = 0;
  });
  if (configured[dev] != cudaSuccess) return configured[dev];
  const int smem = Layout(a.cols, NC, KPB > 0 ? kWarps : 4).bytes;
  int& n = per_sm[dev][a.cols / kMinCols];
  if (n == 0) {
    int v = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, hc_q2_matvec_kernel<NC, KPB>, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (v < 1) return cudaErrorInvalidConfiguration;
    n = v;
  }
  const long long tiles = static_cast<long long>(a.count) * a.tiles;
  const long long slots = static_cast<long long>(n) * sms[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles < slots ? tiles : slots));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hc_q2_matvec_kernel<NC, KPB>, a);
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

// Byte ranges of one product's operands.
struct Ranges {
  size_t wq, ws, x, y;
  Ranges(int rows, int cols, int ncols) {
    const size_t r = static_cast<size_t>(rows), c = static_cast<size_t>(cols), n = static_cast<size_t>(ncols);
    wq = r * c / 4;
    ws = r * (c / 64) * 2;
    x = n * c * 4;
    y = n * r * 4;
  }
};

int check_product(const uint8_t* Wq, const uint16_t* Wscale, const float* x, float* y, const Ranges& b) {
  if (!Wq || !Wscale || !x || !y) return HC_ERR_ARG;
  for (const void* p : {static_cast<const void*>(Wq), static_cast<const void*>(Wscale),
                        static_cast<const void*>(x), static_cast<const void*>(y)}) {
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return HC_ERR_ALIGN;
  }
  if (overlaps(y, b.y, Wq, b.wq) || overlaps(y, b.y, Wscale, b.ws) || overlaps(y, b.y, x, b.x)) return HC_ERR_ARG;
  return HC_OK;
}

int check_sizes(int rows, int cols, int ncols) {
  // rows <= 2^24 keeps the tile counts of a launch (products x rows / 32)
  // inside int
  if (rows < 1 || rows > kMaxRows || ncols < 1 || ncols > kMaxNcols) return HC_ERR_ARG;
  if (cols < kMinCols || cols > kMaxCols || cols % kMinCols != 0) return HC_ERR_SHAPE;
  return HC_OK;
}

// The register form for the pages' width (2560 columns: 5 blocks a warp) at
// 1..3 columns, the shared-memory form otherwise (measured on GB300, µs per
// product in a cold batch at 1 / 2 / 3 / 4 columns: register form 3.14 /
// 3.27 / 3.45 / 4.50, shared-memory form 3.51 / 3.59 / 3.82 / 3.58; at 4
// columns the register form is at its 128-register limit).
template <int NC>
cudaError_t launch_nc(const Args& a, cudaStream_t st) {
  if constexpr (NC < 4) {
    if (a.cols == 2560) return launch<NC, 5>(a, st);
  }
  return launch<NC, 0>(a, st);
}

cudaError_t launch_any(const Args& a, int ncols, cudaStream_t st) {
  switch (ncols) {
    case 1: return launch_nc<1>(a, st);
    case 2: return launch_nc<2>(a, st);
    case 3: return launch_nc<3>(a, st);
    default: return launch_nc<4>(a, st);
  }
}

}  // namespace q2
}  // namespace hc

HC_EXPORT int hc_q2_0_matvec(const uint8_t* Wq, const uint16_t* Wscale, int rows, int cols,
                             const float* x, int ncols, float* y, hc_stream_t stream) {
  const hc_q2_0_desc d{Wq, Wscale, x, y};
  if (!Wq || !Wscale || !x || !y) return HC_ERR_ARG;
  return hc_q2_0_matvec_batch(&d, 1, rows, cols, ncols, stream);
}

// Which launch each product of a batch goes to: a product joins the launch
// being assembled unless that launch holds kLaunchProducts products already
// or the product shares memory with one of them (reads an earlier y, or
// writes over an earlier operand).  Returns the number of launches.
static int plan_launches(const hc_q2_0_desc* descs, int count, const hc::q2::Ranges& b, int* launch) {
  using namespace hc::q2;
  int launches = 0, first = 0, in_launch = 0;
  for (int j = 0; j < count; ++j) {
    bool flush = in_launch == kLaunchProducts;
    for (int i = first; i < j && !flush; ++i) {
      const hc_q2_0_desc& d = descs[j];
      const hc_q2_0_desc& e = descs[i];
      flush = overlaps(d.x, b.x, e.y, b.y) || overlaps(d.Wq, b.wq, e.y, b.y) || overlaps(d.Wscale, b.ws, e.y, b.y) ||
              overlaps(d.y, b.y, e.y, b.y) || overlaps(d.y, b.y, e.x, b.x) || overlaps(d.y, b.y, e.Wq, b.wq) ||
              overlaps(d.y, b.y, e.Wscale, b.ws);
    }
    if (j == 0 || flush) {
      ++launches;
      first = j;
      in_launch = 0;
    }
    launch[j] = launches - 1;
    ++in_launch;
  }
  return launches;
}

HC_EXPORT int hc_q2_0_matvec_batch_plan(const hc_q2_0_desc* descs, int count, int rows, int cols, int ncols,
                                        int* launch) {
  using namespace hc::q2;
  if (!descs || !launch || count < 1) return HC_ERR_ARG;
  const int rc = check_sizes(rows, cols, ncols);
  if (rc != HC_OK) return rc;
  return plan_launches(descs, count, Ranges(rows, cols, ncols), launch);
}

HC_EXPORT int hc_q2_0_matvec_batch(const hc_q2_0_desc* descs, int count, int rows, int cols, int ncols,
                                   hc_stream_t stream) {
  using namespace hc::q2;
  if (!descs || count < 1) return HC_ERR_ARG;
  int rc = check_sizes(rows, cols, ncols);
  if (rc != HC_OK) return rc;
  const Ranges b(rows, cols, ncols);
  for (int j = 0; j < count; ++j) {
    rc = check_product(descs[j].Wq, descs[j].Wscale, descs[j].x, descs[j].y, b);
    if (rc != HC_OK) return rc;
  }
  std::vector<int> launch(static_cast<size_t>(count));
  plan_launches(descs, count, b, launch.data());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Args a;
  a.rows = rows;
  a.cols = cols;
  a.tiles = (rows + kRows - 1) / kRows;
  a.count = 0;
  for (int j = 0; j < count; ++j) {
    a.p[a.count++] = Product{descs[j].Wq, descs[j].Wscale, descs[j].x, descs[j].y};
    if (j + 1 == count || launch[j + 1] != launch[j]) {
      if (launch_any(a, ncols, st) != cudaSuccess) return HC_ERR_CUDA;
      a.count = 0;
    }
  }
  return HC_OK;
}
