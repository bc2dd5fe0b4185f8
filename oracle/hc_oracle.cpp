// Hyper-connection read: FP64 reference oracle.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct CPU
// statement of what the read computes.  Only the test suite, the smoke check
// and the benchmark's CPU-baseline / reference arm may load it.  The CUDA
// library never links, includes or calls it, and it shares no code with the
// CUDA library (no headers, tables or helpers).
//
// Sources (cited by page title and section):
//   [P4] "#2812 sycl: STRATA_GR_FUSED=1, the two-kernel BF16 hyper-connection
//        read (opt-in)", sections "Summary" and "What changed"
//        (gr_fused_down_kernel / gr_fused_up_kernel descriptions): the read is a
//        per-stream RMS norm, a BF16 down projection whose partial sums are
//        scaled by rs per stream, a BF16 up projection, then an epilogue that
//        commits the pending write, applies the gate and averages the
//        streams; R_out is the residual with the pending write committed.
//   [P1] Strata pull request #2070 (Turing up/down kernels), first paragraph:
//        a verify window runs 96 reads, each moving about 13 MB of BF16
//        projection weights.
//   The pages give no formula for the epilogue.  This library fixes it as
//        out = R' + sigmoid(g) * (W_up . lo),   m[c] = mean_s out[s, c],
//   with R' = fl32(R + P) the residual after the pending write P.
//
// Every floating-point step is done in double, in the order the formulas are
// written, with plain loops: no blocking, no fusion, no reordering.
//
// Geometry: n streams of width d, N = n*d rows, K = down width, T tokens.
// Activations are row-major [T][N] with element i = s*d + c (stream-major
// inside a token).  W_down is [K][N] BF16, W_up is [N][K] BF16, both
// row-major.  w_norm and gate have N entries.
//
// The Q8_0 read (hc_oracle_read_q8) is the same read over Q8_0 copies of the
// two projections [P4, sections "Summary" and "Extra Notes": the branch
// builds on an earlier one whose read takes Q8_0 copies of both projections
// (switched on by STRATA_HC_Q8=1), copies that cost device memory on top of
// the BF16 weights].  The pages give no block layout; this library reads Q8_0 as: every row of a
// weight matrix in blocks of 32 consecutive values along the dot-product axis
// (the columns of W_down [K][N], the columns of W_up [N][K]), each block one
// IEEE binary16 scale and 32 int8 values, weight = scale * q.  Quants and
// scales are two arrays: q [rows][cols] int8, scale [rows][cols / 32] binary16.
//
// The Q2_0 matrix-vector product (hc_oracle_q2_0_matvec) is the decode
// windows' other bandwidth-bound step [P3: Strata pull request #2221, first
// paragraph and the table "Kernel (2560 x 12288, cold weights ...)": the QSA
// layers' attn_q projection from 2560 inputs to 12288 outputs over Q2_0
// weights, for one to four columns].  The pages name the format and its
// 64-value blocks but not its bits; this library reads Q2_0 as: every row in
// blocks of 64 consecutive values, each block one IEEE binary16 scale d and
// 64 two-bit codes q in {0, 1, 2, 3}, weight = d * (q - 2); the codes of a
// row packed four to a byte, value j at byte j / 4, bits 2 * (j % 4) and
// 2 * (j % 4) + 1 (least significant first); codes and scales in separate
// arrays, Wq [rows][cols / 4] bytes and Wscale [rows][cols / 64] binary16.
// (The pages' 80 us at about 110 GB/s for 2560 x 12288 is about 8.8 MB per
// call: two bits per value and 16 bits per 64-value block give 8,847,360 B.)
//
// Parity status: every function below is pinned by the CPU tests (hand-expanded
// tiny cases under tests/golden/, closed forms, invariants, brute force).

#include <cmath>
#include <cstdint>
#include <cstring>

namespace {

// A BF16 value is the upper 16 bits of an IEEE binary32; widening it to
// double is exact.
double bf16_to_double(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
// bits; exponent 0 holds the subnormals (fraction * 2^-24), exponent 31 the
// infinities and NaNs.  Every binary16 value is exact in double.
double half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int exponent = (h >> 10) & 0x1F;
  const int fraction = h & 0x3FF;
  double v;
  if (exponent == 0) {
    v = std::ldexp(static_cast<double>(fraction), -24);
  } else if (exponent == 31) {
    v = fraction == 0 ? HUGE_VAL : std::nan("");
  } else {
    v = std::ldexp(static_cast<double>(1024 + fraction), exponent - 25);
  }
  return sign ? -v : v;
}

// One Q8_0 weight: row r, column j of a matrix with `cols` columns.
double q8_weight(const int8_t* q, const uint16_t* scale, int cols, int r, int j) {
  return half_to_double(scale[(size_t)r * (cols / 32) + j / 32]) *
         static_cast<double>(q[(size_t)r * cols + j]);
}

// One Q2_0 weight: row r, column j of a matrix with `cols` columns.
double q2_weight(const uint8_t* codes, const uint16_t* scale, int cols, int r, int j) {
  const uint8_t byte = codes[(size_t)r * (cols / 4) + j / 4];
  const int q = (byte >> (2 * (j % 4))) & 3;
  return half_to_double(scale[(size_t)r * (cols / 64) + j / 64]) * static_cast<double>(q - 2);
}

}  // namespace

extern "C" {

// Step 1 [P4 "Summary": R_out is "the pending write"; "What changed": the down
// kernel stages R' * w_norm].  R' = fl32(R + P).  The exact sum of two floats
// rounded once to binary32 is what a single fp32 round-to-nearest add gives;
// computing it in double first and rounding once is equivalent because
// double carries more than 2*24+2 bits.
void hc_oracle_commit(int N, int T, const float* R, const float* P, float* r_out) {
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < N; ++i) {
      double r = R[(size_t)t * N + i];
      double p = (P != nullptr) ? P[(size_t)t * N + i] : 0.0;
      r_out[(size_t)t * N + i] = static_cast<float>(r + p);
    }
  }
}

// Step 2 [P4, "What changed": the down kernel accumulates squares over its
// slab, and rs scales the partial sums stream by stream].
// ss[t][s] = sum_c R'[t][s*d+c]^2 ; rs[t][s] = 1 / sqrt(ss[t][s] / d + eps).
void hc_oracle_rms(int n, int d, int T, double eps, const float* r_prime,
                   double* ss, double* rs) {
  const int N = n * d;
  for (int t = 0; t < T; ++t) {
    for (int s = 0; s < n; ++s) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c) {
        double v = r_prime[(size_t)t * N + (size_t)s * d + c];
        acc += v * v;
      }
      ss[t * n + s] = acc;
      rs[t * n + s] = 1.0 / std::sqrt(acc / d + eps);
    }
  }
}

// Step 3 [P4 "What changed": R' * w_norm staged unscaled, the down
// projection's sums per stream, then "applies rs per stream, writes lo"].
// lo[t][k] = sum_s rs[t][s] * sum_c W_down[k][s*d+c] * (R'[t][s*d+c] * w_norm[s*d+c]).
void hc_oracle_down(int n, int d, int K, int T, const float* r_prime,
                    const float* w_norm, const uint16_t* W_down, const double* rs,
                    double* lo) {
  const int N = n * d;
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      double total = 0.0;
      for (int s = 0; s < n; ++s) {
        double stream_sum = 0.0;
        for (int c = 0; c < d; ++c) {
          const int i = s * d + c;
          double x = static_cast<double>(r_prime[(size_t)t * N + i]) *
                     static_cast<double>(w_norm[i]);
          stream_sum += bf16_to_double(W_down[(size_t)k * N + i]) * x;
        }
        total += rs[t * n + s] * stream_sum;
      }
      lo[(size_t)t * K + k] = total;
    }
  }
}

// Step 4 [P4 "What changed": gr_fused_up_kernel, the up projection].
// u[t][i] = sum_k W_up[i][k] * lo[t][k].
void hc_oracle_up(int N, int K, int T, const uint16_t* W_up, const double* lo,
                  double* u) {
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < N; ++i) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        acc += bf16_to_double(W_up[(size_t)i * K + k]) * lo[(size_t)t * K + k];
      }
      u[(size_t)t * N + i] = acc;
    }
  }
}

// Step 5 [P4, "What changed": the up kernel ends with the default read's
// epilogue, which commits the pending write, applies the gate and averages
// the streams; the formula is this library's reading, see the header].
// out[t][i] = R'[t][i] + sigmoid(g[i]) * u[t][i], sigmoid(x) = 1 / (1 + exp(-x));
// m[t][c] = (1/n) * sum_s out[t][s*d+c].
void hc_oracle_epilogue(int n, int d, int T, const float* r_prime, const float* gate,
                        const double* u, double* out, double* mean) {
  const int N = n * d;
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < N; ++i) {
      double g = gate[i];
      double sig = 1.0 / (1.0 + std::exp(-g));
      out[(size_t)t * N + i] =
          static_cast<double>(r_prime[(size_t)t * N + i]) + sig * u[(size_t)t * N + i];
    }
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int s = 0; s < n; ++s) acc += out[(size_t)t * N + (size_t)s * d + c];
      mean[(size_t)t * d + c] = acc / n;
    }
  }
}

// Step 3 over Q8_0 weights: hc_oracle_down with W_down[k][i] = the Q8_0
// value of row k, column i.
void hc_oracle_down_q8(int n, int d, int K, int T, const float* r_prime,
                       const float* w_norm, const int8_t* Wd_q, const uint16_t* Wd_scale,
                       const double* rs, double* lo) {
  const int N = n * d;
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      double total = 0.0;
      for (int s = 0; s < n; ++s) {
        double stream_sum = 0.0;
        for (int c = 0; c < d; ++c) {
          const int i = s * d + c;
          double x = static_cast<double>(r_prime[(size_t)t * N + i]) *
                     static_cast<double>(w_norm[i]);
          stream_sum += q8_weight(Wd_q, Wd_scale, N, k, i) * x;
        }
        total += rs[t * n + s] * stream_sum;
      }
      lo[(size_t)t * K + k] = total;
    }
  }
}

// Step 4 over Q8_0 weights: u[t][i] = sum_k W_up[i][k] * lo[t][k] with
// W_up[i][k] the Q8_0 value of row i, column k.
void hc_oracle_up_q8(int N, int K, int T, const int8_t* Wu_q, const uint16_t* Wu_scale,
                     const double* lo, double* u) {
  for (int t = 0; t < T; ++t) {
    for (int i = 0; i < N; ++i) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += q8_weight(Wu_q, Wu_scale, K, i, k) * lo[(size_t)t * K + k];
      u[(size_t)t * N + i] = acc;
    }
  }
}

// The binary16 value of h (exported for the tests of the decoding).
double hc_oracle_half(uint16_t h) { return half_to_double(h); }

// The whole Q8_0 read: steps 1, 2, 3 and 4 over Q8_0 weights, 5.  N and K
// must be multiples of 32.  Buffers as for hc_oracle_read.
int hc_oracle_read_q8(int n, int d, int K, int T, double eps, const float* R,
                      const float* P, const float* w_norm, const int8_t* Wd_q,
                      const uint16_t* Wd_scale, const int8_t* Wu_q, const uint16_t* Wu_scale,
                      const float* gate, float* r_out, double* ss, double* rs, double* lo,
                      double* u, double* out, double* mean) {
  if (n <= 0 || d <= 0 || K <= 0 || T <= 0 || eps < 0.0) return -1;
  if ((n * d) % 32 != 0 || K % 32 != 0) return -1;
  if (!R || !w_norm || !Wd_q || !Wd_scale || !Wu_q || !Wu_scale || !gate) return -1;
  if (!r_out || !ss || !rs || !lo || !u || !out || !mean) return -1;
  const int N = n * d;
  hc_oracle_commit(N, T, R, P, r_out);
  hc_oracle_rms(n, d, T, eps, r_out, ss, rs);
  hc_oracle_down_q8(n, d, K, T, r_out, w_norm, Wd_q, Wd_scale, rs, lo);
  hc_oracle_up_q8(N, K, T, Wu_q, Wu_scale, lo, u);
  hc_oracle_epilogue(n, d, T, r_out, gate, u, out, mean);
  return 0;
}

// The Q2_0 matrix-vector product [P3, first paragraph and the kernel table]:
// y[c][r] = sum_j W[r][j] * x[c][j] for columns c < ncols, with W[r][j] the
// Q2_0 value of row r, column j.  x [ncols][cols] float, y [ncols][rows]
// double.  cols must be a multiple of 64.  Returns 0, or -1 on a bad argument.
int hc_oracle_q2_0_matvec(int rows, int cols, int ncols, const uint8_t* Wq,
                          const uint16_t* Wscale, const float* x, double* y) {
  if (rows <= 0 || cols <= 0 || cols % 64 != 0 || ncols <= 0) return -1;
  if (!Wq || !Wscale || !x || !y) return -1;
  for (int c = 0; c < ncols; ++c) {
    for (int r = 0; r < rows; ++r) {
      double acc = 0.0;
      for (int j = 0; j < cols; ++j) {
        acc += q2_weight(Wq, Wscale, cols, r, j) * static_cast<double>(x[(size_t)c * cols + j]);
      }
      y[(size_t)c * rows + r] = acc;
    }
  }
  return 0;
}

// The whole read, steps 1-5 in order.  Any output pointer may be null except
// the scratch the later steps need; this entry point allocates its own
// intermediates only through the caller-provided buffers:
//   r_out [T][N] float, ss/rs [T][n], lo [T][K], u [T][N], out [T][N], mean [T][d].
// Returns 0 on success, -1 on a bad argument.
int hc_oracle_read(int n, int d, int K, int T, double eps, const float* R,
                   const float* P, const float* w_norm, const uint16_t* W_down,
                   const uint16_t* W_up, const float* gate, float* r_out, double* ss,
                   double* rs, double* lo, double* u, double* out, double* mean) {
  if (n <= 0 || d <= 0 || K <= 0 || T <= 0 || eps < 0.0) return -1;
  if (!R || !w_norm || !W_down || !W_up || !gate) return -1;
  if (!r_out || !ss || !rs || !lo || !u || !out || !mean) return -1;
  const int N = n * d;
  hc_oracle_commit(N, T, R, P, r_out);
  hc_oracle_rms(n, d, T, eps, r_out, ss, rs);
  hc_oracle_down(n, d, K, T, r_out, w_norm, W_down, rs, lo);
  hc_oracle_up(N, K, T, W_up, lo, u);
  hc_oracle_epilogue(n, d, T, r_out, gate, u, out, mean);
  return 0;
}

}  // extern "C"
