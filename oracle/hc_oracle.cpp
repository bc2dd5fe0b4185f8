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
//        scaled by rs per stream, a BF16 up projection, then an epilogue of
//        "pending write, gate, stream mean"; R_out is "the pending write".
//   [P1] Strata pull request #2070 (Turing up/down kernels), first paragraph:
//        96 reads per window, 13 MB of BF16 weights each.
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

// Step 2 [P4 "What changed": the slab's sums of squares; "rs per stream"].
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

// Step 5 [P4 "What changed": "the default read's epilogue: pending write,
// gate, stream mean"; the formula is this library's reading, see the header].
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
