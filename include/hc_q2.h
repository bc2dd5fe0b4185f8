/* Q2_0 matrix-vector product on GB300 (sm_103a): C ABI.
 *
 * The decode windows' other bandwidth-bound step: the QSA layers' attn_q
 * projection, 2560 inputs to 12288 outputs over Q2_0 weights, for one to
 * four columns at a time (Strata pull request #2221, first paragraph and the
 * table "Kernel (2560 x 12288, cold weights: six copies in rotation, 300
 * calls)").
 *
 *   y[c][r] = sum_j W[r][j] * x[c][j],   c < ncols, r < rows, j < cols.
 *
 * Q2_0 (the pages name the format and its 64-value blocks, not its bits;
 * this library reads it as): every row of W in blocks of 64 consecutive
 * values, each block one IEEE binary16 scale d and 64 two-bit codes
 * q in {0, 1, 2, 3}, weight = d * (q - 2).  The codes of a row are packed
 * four to a byte, value j at byte j / 4, bits 2 * (j % 4) and 2 * (j % 4) + 1
 * (least significant first).
 *
 * Layouts (row-major, contiguous, device memory, every pointer 16-byte
 * aligned):
 *   Wq     : uint8  [rows][cols / 4]   (codes)
 *   Wscale : uint16 [rows][cols / 64]  (binary16 bit patterns)
 *   x      : float  [ncols][cols]
 *   y      : float  [ncols][rows]
 *
 * Sizes: 1 <= rows <= 2^24; cols a multiple of 512, 512 <= cols <= 4096;
 * 1 <= ncols <= 4.
 *
 * Arithmetic: each weight is decoded exactly; x is scaled per column by a
 * power of two and split into two binary16 terms (22 significant bits); each
 * 64-value block's dot product is summed in FP32 on the tensor cores and
 * multiplied by the block's scale, and the blocks of a row are accumulated in
 * FP32 in a fixed order.  The result is deterministic: the same inputs give
 * the same bits on every call, alone, in a batch or in a CUDA graph.
 *
 * Ownership: the caller owns every buffer; the call allocates nothing.
 * y must not overlap Wq, Wscale or x.
 *
 * Asynchrony: one kernel is enqueued on `stream` (the calling thread's
 * current device); the call never synchronises and can be captured into a
 * CUDA graph.  The kernel is persistent (as many CTAs as the device holds at
 * once stream 32-row tiles through shared memory) and uses programmatic
 * dependent launch: it fetches the weights of its first tiles before it
 * waits for the preceding kernel in the stream, and reads x and writes y
 * only after that wait.  Wq and Wscale must therefore not be written by a
 * kernel that immediately precedes the call on the stream and itself
 * triggers its dependents early (kernels that do not use programmatic
 * completion, copies and memsets are always waited for in full).
 *
 * Errors (hc_status of hc_read.h): HC_ERR_ARG for a NULL pointer, rows
 * outside 1..2^24, ncols outside 1..4, y overlapping an input, or a batch
 * without products; HC_ERR_SHAPE for cols not supported; HC_ERR_ALIGN for a
 * pointer that is not 16-byte aligned; HC_ERR_CUDA for a launch error.
 * Nothing is enqueued on an error.  The kernel has no waits of its own.
 */
#ifndef HC_Q2_H
#define HC_Q2_H

#include <stdint.h>

#include "hc_read.h"

#ifdef __cplusplus
extern "C" {
#endif

int hc_q2_0_matvec(const uint8_t* Wq, const uint16_t* Wscale, int rows, int cols,
                   const float* x, int ncols, float* y, hc_stream_t stream);

/* One product of a batch: the buffers of hc_q2_0_matvec. */
typedef struct {
  const uint8_t* Wq;
  const uint16_t* Wscale;
  const float* x;
  float* y;
} hc_q2_0_desc;

/* Enqueue `count` products of one shape (rows, cols, ncols) on `stream`, in
 * order; each gives the bits hc_q2_0_matvec gives for the same buffers.
 * `descs` is host memory, read during the call only.  The arguments of every
 * product are checked before anything is enqueued.
 *
 * Products that share no memory (none reads an earlier product's y or
 * writes over an earlier product's operands) run in one persistent launch,
 * up to 120 at a time: their tiles stream through the GPU back to back, with
 * the next tiles' weights in flight while one is computed (x is prepared for
 * the tensor cores once per CTA while it stays the same), which a run of
 * independent products (the pages' cold sweep of 300 calls, or projections
 * that read one input) needs to keep HBM busy.  A product that does share
 * memory with an earlier one starts a new launch, which waits for all
 * earlier kernels in the stream as hc_q2_0_matvec does.  No product of the
 * batch reads x or writes y before every kernel enqueued ahead of the batch
 * has completed. */
int hc_q2_0_matvec_batch(const hc_q2_0_desc* descs, int count, int rows, int cols, int ncols,
                         hc_stream_t stream);

/* How hc_q2_0_matvec_batch would split this batch (same arguments): writes
 * launch[j], the launch product j goes to (0, 1, ... in order), and returns
 * the number of launches; HC_ERR_ARG for NULL pointers or no products,
 * HC_ERR_SHAPE / HC_ERR_ARG for sizes as hc_q2_0_matvec.  A product joins
 * the launch being assembled unless it holds 120 products already or the
 * product shares memory with one of them.  Host logic only: the pointers
 * are compared, never dereferenced, and no device is needed. */
int hc_q2_0_matvec_batch_plan(const hc_q2_0_desc* descs, int count, int rows, int cols, int ncols,
                              int* launch);

#ifdef __cplusplus
}
#endif

#endif /* HC_Q2_H */
