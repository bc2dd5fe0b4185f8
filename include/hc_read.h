/* hc_read.h - C ABI of the GB300 (sm_103a) hyper-connection read.
 *
 * The read (sources cited by page title and section):
 *   "#2812 sycl: STRATA_GR_FUSED=1, the two-kernel BF16 hyper-connection read
 *   (opt-in)", sections "Summary" and "What changed": the pending write is
 *   committed (R_out), a per-stream RMS norm's sums of squares give rs, the
 *   BF16 down projection of R' * w_norm is scaled by rs per stream into lo, and
 *   the BF16 up projection of lo feeds an epilogue of pending write, gate and
 *   stream mean.  Strata pull request #2070 (Turing up/down kernels): a verify
 *   window runs 96 reads, each moving about 13 MB of BF16 projection weights.  The pages give no formula for
 *   the epilogue; this library defines it as written below.
 *
 * For T tokens, n = 4 streams of width d, N = n*d, down width K, i = s*d + c:
 *   R'[t][i]  = fl32(R[t][i] + P[t][i])          (P = 0 when pending == NULL)
 *   ss[t][s]  = sum_c R'[t][s*d+c]^2,  rs[t][s] = 1 / sqrt(ss[t][s] / d + eps)
 *   lo[t][k]  = sum_s rs[t][s] * sum_c W_down[k][s*d+c] * R'[t][s*d+c] * w_norm[s*d+c]
 *   u[t][i]   = sum_k W_up[i][k] * lo[t][k]
 *   out[t][i] = R'[t][i] + sigmoid(gate[i]) * u[t][i]
 *   mean[t][c]= (1/n) * sum_s out[t][s*d+c]
 *
 * Supported geometries (compiled in): n = 4 with (d, K) = (2560, 320) or
 * (4096, 512).  1 <= T <= T_max <= 64.
 *
 * Layouts (all row-major, contiguous, device memory, 16-byte aligned):
 *   R, pending, out, r_out : float  [T][N]
 *   w_norm, gate           : float  [N]
 *   W_down                 : uint16 [K][N]  (BF16 bit patterns)
 *   W_up                   : uint16 [N][K]  (BF16 bit patterns)
 *   lo                     : float  [T][K]
 *   mean                   : float  [T][d]
 *   rs                     : float  [T][n]
 *
 * Ownership: the caller owns every tensor.  A handle owns its scratch (two
 * slots of per-stream partial sums, used by consecutive reads in turn, and an
 * error word), allocated and zeroed by hc_read_create and freed by
 * hc_read_destroy.
 *
 * Aliasing: out may equal R (in-place update of the residual).  pending must
 * not overlap out; lo, mean, r_out and rs must not overlap any input.
 *
 * Asynchrony: hc_read only validates and enqueues two kernels on `stream`; it
 * never synchronises.  Calls on one handle must be issued to one stream at a
 * time (the scratch belongs to the handle).  The call can be captured into a
 * CUDA graph; replays give the same bits as direct calls.  The kernels use
 * programmatic dependent launch: each kernel prefetches its BF16 weights,
 * w_norm and gate before it waits for the preceding kernel in the stream.
 * When the read takes nothing that the previous read enqueued on the same
 * stream by this library writes (the library compares address ranges), the
 * read also reads R and pending and computes before that wait, so the two
 * reads overlap on the GPU; its outputs are still written after the previous
 * read's.  The inputs of a read must therefore not be written by a kernel
 * that immediately precedes it on the stream and itself triggers its
 * dependents early (kernels that do not use programmatic completion, copies
 * and memsets are always waited for in full); callers whose own kernels do
 * that switch the overlap off per handle with hc_read_set_overlap.
 *
 * Errors: every entry point returns an hc_status (0 = HC_OK).  Argument errors
 * are detected on the host before anything is enqueued.  HC_ERR_CUDA reports
 * a CUDA runtime error at launch.  A kernel that gives up on a bounded wait
 * records it in the handle's error word; hc_read_check reports it as
 * HC_ERR_TIMEOUT until hc_read_reset clears it.
 */
#ifndef HC_READ_H
#define HC_READ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hc_read_s* hc_read_t;
typedef void* hc_stream_t;  /* a cudaStream_t; NULL = the legacy default stream */
typedef void* hc_graph_t;   /* an instantiated CUDA graph (cudaGraphExec_t) */

typedef enum {
  HC_OK = 0,
  HC_ERR_ARG = -1,      /* null handle/pointer, T out of range, bad eps, wrong device */
  HC_ERR_ALIGN = -2,    /* a pointer is not 16-byte aligned */
  HC_ERR_SHAPE = -3,    /* geometry not compiled in */
  HC_ERR_CUDA = -4,     /* CUDA runtime error (allocation, launch, capture) */
  HC_ERR_TIMEOUT = -5,  /* a kernel gave up on a bounded wait (see hc_read_check) */
  HC_ERR_TOO_LARGE = -6 /* T above the no-allocation entry point's maximum */
} hc_status;

/* Create a read handle for geometry (n, d, K) on CUDA device `device`, for up
 * to T_max tokens per call, with the RMS epsilon `eps` (>= 0).  Allocates and
 * zeroes the handle's scratch on that device (synchronous).  On success *h
 * holds the handle; on failure *h is NULL. */
int hc_read_create(hc_read_t* h, int n, int d, int K, int T_max, float eps, int device);

/* Enqueue one read of T tokens on `stream` (see the formulas above).
 * pending may be NULL (no pending write).  The calling thread's current CUDA
 * device must be the handle's device.  Outputs: out [T][N], mean [T][d],
 * lo [T][K]. */
int hc_read(hc_read_t h, const float* R, const float* w_norm, const uint16_t* W_down,
            const uint16_t* W_up, const float* gate, const float* pending, int T,
            float* out, float* mean, float* lo, hc_stream_t stream);

/* hc_read with two optional debug outputs: r_out [T][N] receives R' (the
 * committed residual, bit for bit one fp32 add), rs [T][n] the per-stream
 * inverse RMS.  Either may be NULL. */
int hc_read_ex(hc_read_t h, const float* R, const float* w_norm, const uint16_t* W_down,
               const uint16_t* W_up, const float* gate, const float* pending, int T,
               float* out, float* mean, float* lo, float* r_out, float* rs,
               hc_stream_t stream);

/* hc_read over Q8_0 copies of the two projections.
 *
 * The pages say that this two-kernel read follows the structure of an
 * earlier read over Q8_0 copies of the projections, switched on by
 * STRATA_HC_Q8=1 ("#2812 sycl: STRATA_GR_FUSED=1, the two-kernel BF16
 * hyper-connection read (opt-in)", sections "Summary" and "Extra Notes"),
 * but not how Q8_0 lays out its blocks.  This library reads Q8_0 as: every
 * row of a weight matrix in blocks of 32 consecutive values along the
 * dot-product axis, each block one IEEE binary16 scale and
 * 32 int8 values, weight = scale * q, with quants and scales in separate
 * arrays:
 *   Wd_q     [K][n*d] int8,   Wd_scale [K][n*d/32] binary16 bits (W_down),
 *   Wu_q     [n*d][K] int8,   Wu_scale [n*d][K/32] binary16 bits (W_up),
 * row-major.  Everything else as hc_read_ex (the same norm, partial sums,
 * epilogue and outputs).  Every pointer, scales included, must be 16-byte
 * aligned (HC_ERR_ALIGN).  The MMA takes the int8 values as BF16 (exact)
 * and applies each block's scale to the block's FP32 sum. */
int hc_read_q8(hc_read_t h, const float* R, const float* w_norm, const int8_t* Wd_q,
               const uint16_t* Wd_scale, const int8_t* Wu_q, const uint16_t* Wu_scale,
               const float* gate, const float* pending, int T, float* out, float* mean, float* lo,
               float* r_out, float* rs, hc_stream_t stream);

/* One read of a batch: the arguments of hc_read, same meaning and layouts. */
typedef struct {
  const float* R;
  const float* w_norm;
  const uint16_t* W_down;
  const uint16_t* W_up;
  const float* gate;
  const float* pending;  /* NULL = no pending write */
  float* out;
  float* mean;
  float* lo;
} hc_read_desc;

/* Enqueue `count` reads of T tokens each on `stream`, in order: the reads of a
 * verify window (the pages' engine runs 96 per window, one per layer; Strata
 * pull request #2070, first paragraph), or any list of reads.
 *
 * Read j may take as R the previous read's out (the same pointer): a chained
 * read, whose input then never leaves the chip.  Otherwise R and pending of
 * read j must not overlap an output (out, mean, lo) of an earlier read of the
 * batch, and pending must not overlap the read's own out (HC_ERR_ARG).  Each
 * read's outputs are those of hc_read with the same arguments; reads may
 * reuse one set of output buffers.  `descs` is host memory, read during the
 * call only.
 *
 * The reads fall into groups (hc_read_batch_groups): two reads share a group
 * when an output of one overlaps an input or output of the other, directly or
 * through other reads.  With two or more groups the batch runs read by read
 * on up to 6 internal streams of the handle, each group on one of them in
 * the batch's order, forked from `stream` and joined back into it with
 * events (graph capture included); every read's bits are those of hc_read.
 * Reads sharing nothing then overlap on the device, which is what the
 * hardware needs: one read is a chain of dependent steps (about 5 us) that
 * keeps HBM busy for only 2 us of it.
 *
 * A batch that is one group (a chain, or reads reusing one set of outputs),
 * for (d, K) = (2560, 320) and T <= 4 on a device that can hold it, runs as
 * one persistent kernel per 224 reads: 128 CTAs, one per SM, that must all
 * be resident at once (a cooperative launch).  Do not run two such batches
 * at the same time on one device (two streams or two threads): a kernel that
 * cannot get its 128 SMs gives up after its bounded waits and reports
 * HC_ERR_TIMEOUT through hc_read_check.  Other one-group batches run read by
 * read on `stream` as hc_read does.  hc_read_reset also clears the
 * persistent kernel's abort word; its exchange state needs no reset. */
int hc_read_batch(hc_read_t h, const hc_read_desc* descs, int count, int T, hc_stream_t stream);

/* How hc_read_batch would run this batch (same arguments): 0 read by read on
 * the caller's stream, 1 as the persistent kernel, L >= 2 on L internal
 * streams; HC_ERR_ARG for a NULL handle or descs, no reads or T outside
 * 1..T_max.  Enqueues nothing. */
int hc_read_batch_plan(hc_read_t h, const hc_read_desc* descs, int count, int T);

/* Most internal streams hc_read_batch may use on this handle (default and
 * upper bound 6; 0 or 1: every batch stays on the caller's stream, as one
 * persistent kernel or read by read).  Returns the previous setting, or
 * HC_ERR_ARG for a NULL handle or lanes < 0.  Not thread-safe against a
 * concurrent hc_read_batch on the same handle. */
int hc_read_set_batch_lanes(hc_read_t h, int lanes);

/* The groups of a batch of `count` T-token reads of geometry (n, d, K): writes
 * group[j] (groups numbered 0, 1, ... in order of first appearance) and
 * returns the number of groups, or HC_ERR_ARG.  Reads j and k share a group
 * when a byte range of one's outputs (out [T][n d] fp32, mean [T][d] fp32,
 * lo [T][K] fp32) overlaps one of the other's inputs (R, pending, w_norm,
 * gate, W_down, W_up) or outputs, or through a chain of such overlaps.
 * Host logic only: the pointers are compared, never dereferenced, and no
 * device is needed. */
int hc_read_batch_groups(const hc_read_desc* descs, int count, int n, int d, int K, int T, int* group);

/* One Q8_0 read of a batch: the arguments of hc_read_q8, same meaning and
 * layouts. */
typedef struct {
  const float* R;
  const float* w_norm;
  const int8_t* Wd_q;
  const uint16_t* Wd_scale;
  const int8_t* Wu_q;
  const uint16_t* Wu_scale;
  const float* gate;
  const float* pending;  /* NULL = no pending write */
  float* out;
  float* mean;
  float* lo;
} hc_read_q8_desc;

/* hc_read_batch over Q8_0 reads: the same rules on the reads' buffers, the
 * same groups (the scale arrays count as inputs) and the same internal
 * streams.  The persistent kernel takes BF16 weights only, so a one-group
 * Q8_0 batch runs read by read on `stream`.  Alignment as hc_read_q8. */
int hc_read_batch_q8(hc_read_t h, const hc_read_q8_desc* descs, int count, int T, hc_stream_t stream);

/* How hc_read_batch_q8 would run this batch: 0 read by read on the caller's
 * stream, L >= 2 on L internal streams; HC_ERR_ARG as hc_read_batch_plan.
 * Enqueues nothing. */
int hc_read_batch_q8_plan(hc_read_t h, const hc_read_q8_desc* descs, int count, int T);

/* hc_read_batch_groups for Q8_0 reads: the inputs are R, pending, w_norm,
 * gate, Wd_q and Wu_q ([K][n d] and [n d][K] bytes) and Wd_scale and Wu_scale
 * ([K][n d / 32] and [n d][K / 32] binary16); HC_ERR_ARG also when n d or K
 * is not a multiple of 32.  Host logic only. */
int hc_read_batch_q8_groups(const hc_read_q8_desc* descs, int count, int n, int d, int K, int T, int* group);

/* 1 if hc_read_batch on this handle runs batches of T-token reads as the
 * persistent kernel, 0 if it runs them read by read; HC_ERR_ARG for a NULL
 * handle or T outside 1..T_max. */
int hc_read_batch_persistent(hc_read_t h, int T);

/* Synchronise with the handle's device and report the kernels' error word:
 * HC_OK, or HC_ERR_TIMEOUT if any kernel gave up on a bounded wait since the
 * last hc_read_reset. */
int hc_read_check(hc_read_t h);

/* The error word itself (synchronises the device), or a negative hc_status.
 * Bits: 1 and 2 the down kernel's w_norm and W_down copies, 4 and 8 the up
 * kernel's gate and W_up copies, 16 a ring slot of hc_read_batch's persistent
 * kernel that did not land, 32 a ring slot its producer could not reuse, 64 a
 * cluster exchange (partial sums or lo) and 128 the global exchange that did
 * not complete in time. */
int64_t hc_read_error_word(hc_read_t h);

/* Re-zero the handle's error word on `stream` (after HC_ERR_TIMEOUT). */
int hc_read_reset(hc_read_t h, hc_stream_t stream);

/* Free the handle's scratch.  Synchronises with the handle's device first.
 * NULL is ignored. */
void hc_read_destroy(hc_read_t h);

/* Bytes of device scratch a handle holds (for accounting). */
int64_t hc_read_scratch_bytes(hc_read_t h);

/* Limit, in nanoseconds counted from the kernel's start, of the first
 * bulk-copy wait of the down kernel of every later read enqueued through this
 * handle (hc_read, hc_read_ex, hc_read_q8 and the reads of batches that run
 * on the internal streams).  0 restores the default, which is also the
 * largest value taken: 1 s.  A read whose down kernel reaches that wait after
 * the limit gives up on it whether or not the copy has landed: its results
 * are void, the copy is still drained before the kernel exits, and
 * hc_read_check reports HC_ERR_TIMEOUT (bit 1 or 2 of hc_read_error_word)
 * until hc_read_reset.  This is how the timeout path is exercised on purpose
 * (a limit of a few nanoseconds); no other wait takes the setting.  Not
 * thread-safe against a concurrent read on the same handle.  HC_ERR_ARG for
 * a NULL handle. */
int hc_read_set_wait_limit(hc_read_t h, uint64_t ns);

/* Whether reads on this handle may overlap the read enqueued before them on
 * the same stream (1, the default) or always wait for it in full (0).  With
 * 1, a read that takes nothing the previous read wrote reads R and pending
 * and computes before its dependency wait (see "Asynchrony" above); callers
 * whose own kernels trigger their dependents early and write a read's inputs
 * just before it should pass 0.  Returns the previous setting, or HC_ERR_ARG
 * for a NULL handle or a value other than 0 or 1.  Not thread-safe against a
 * concurrent read on the same handle. */
int hc_read_set_overlap(hc_read_t h, int enabled);

/* Weights in tile order: optional second copies of a W_down or W_up, laid
 * out so that every CTA of the read kernels fetches its weight tile as one
 * contiguous block instead of many row segments far apart in [K][N] or
 * [N][K].  The values are the same, and so is every bit of every result; the
 * gain is DRAM efficiency (measured at d = 2560 in a cold batch: about 8 %
 * less time per read at T = 2..4, 4-5 % at T = 9..16, 3-4 % at T = 32, 2 %
 * at T = 64, within 1 % at T = 5..8).  Reads whose kernels have no tiled
 * path keep reading the weights themselves.
 *
 * hc_read_down_tiles_bytes: size of a W_down's copy for this handle's
 * geometry, or -1 for a NULL handle.  At d = 2560, K = 320: 13,189,120
 * bytes, the 32-row tiles of the BF16 reads with T = 2..4 (6,635,520 bytes:
 * rows at a 1,296-byte pitch) followed by the 64-row tiles of the
 * tensor-memory kernels (T >= 5; 6,553,600 bytes in the 128-byte swizzle of
 * their shared memory).  At d = 4096, K = 512: the 32-row tiles alone,
 * 16,908,288 bytes, which every T reads.
 *
 * hc_read_up_tiles_bytes: size of a W_up's copy (6,553,600 bytes at
 * d = 2560, read by the up kernel of T >= 9; 0 at d = 4096, where no kernel
 * takes one), or -1 for a NULL handle.
 *
 * hc_read_register_down_tiles / hc_read_register_up_tiles: write the copy of
 * W_down ([K][N] BF16) or W_up ([N][K] BF16), on the handle's device, into
 * `tiles` (caller-owned device memory of the size above, disjoint from the
 * weights) on `stream`, wait for it, and register the pair: every later read
 * through this handle whose W_down (W_up) is this pointer fetches its tiles
 * from `tiles` where its kernels can.  A registration replaces one of the
 * same pointer.  `tiles` must stay allocated and the weights unchanged until
 * the matching forget call or hc_read_destroy (register again after
 * changing the weights); graphs captured meanwhile keep using `tiles`.  Not
 * during stream capture.  HC_ERR_ARG for a NULL handle or pointer, a
 * capturing stream, overlapping buffers or another device; HC_ERR_ALIGN if
 * either pointer is not 16-byte aligned; HC_ERR_SHAPE for up tiles at a
 * geometry without a kernel that takes them; HC_ERR_CUDA if the copy fails.
 *
 * hc_read_forget_down_tiles / hc_read_forget_up_tiles: drop the registration
 * of a W_down (W_up), all of them for NULL; later reads read the weights
 * themselves.  HC_ERR_ARG for a NULL handle.  None of these calls is
 * thread-safe against a concurrent read on the same handle. */
int64_t hc_read_down_tiles_bytes(hc_read_t h);
int hc_read_register_down_tiles(hc_read_t h, const void* W_down, void* tiles, hc_stream_t stream);
int hc_read_forget_down_tiles(hc_read_t h, const void* W_down);
int64_t hc_read_up_tiles_bytes(hc_read_t h);
int hc_read_register_up_tiles(hc_read_t h, const void* W_up, void* tiles, hc_stream_t stream);
int hc_read_forget_up_tiles(hc_read_t h, const void* W_up);

/* hc_read without a handle and without any device allocation.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory when they need the read: engines that
 * reserve nearly all of HBM for weights and KV cache at start-up (a later
 * cudaMalloc fails), code that runs inside another framework's allocator,
 * and code paths that cannot afford cudaMalloc's implicit device-wide
 * synchronisation.  hc_read_create needs cudaMalloc for its scratch; this
 * entry point uses a fixed scratch array compiled into the library instead
 * (HC_NOALLOC_SCRATCH_BYTES, held on every device that loads the library
 * until the process exits) and calls no allocating routine.
 *
 * Geometry (n, d, K) and eps are passed per call (same supported set as
 * hc_read_create); 1 <= T <= HC_NOALLOC_MAX_T, larger T returns
 * HC_ERR_TOO_LARGE.  Other arguments, layouts and errors as hc_read.  The
 * current device must be the device the pointers live on.
 *
 * The first call on a device sets that device up (it looks up the scratch
 * array's device address and sets kernel attributes); make that first call
 * before any stream capture.  Every call on a device shares the one scratch
 * array: calls that overlap on the GPU (two streams, or two threads) race and
 * give wrong results, so serialise them.  The array keeps what the last call
 * left there: the partial sums need no clearing (each call writes all it
 * reads), and the error word, which starts at zero when the library is
 * loaded, collects the calls' bounded-wait failures until
 * hc_read_noalloc_check reads and clears it.  No call runs every read in
 * independent mode: each waits for the kernel before it in full. */
#define HC_NOALLOC_MAX_T 8
#define HC_NOALLOC_SCRATCH_BYTES (4 * HC_NOALLOC_MAX_T * 512 * 4 + 256)
int hc_read_noalloc(int n, int d, int K, float eps, const float* R, const float* w_norm,
                    const uint16_t* W_down, const uint16_t* W_up, const float* gate,
                    const float* pending, int T, float* out, float* mean, float* lo,
                    hc_stream_t stream);

/* The no-allocation entry point's counterpart of hc_read_check, for the
 * current device: synchronises the device, then returns HC_ERR_TIMEOUT if a
 * kernel of an hc_read_noalloc call gave up on a bounded wait since the last
 * hc_read_noalloc_check (and clears that record), HC_OK if none did or no
 * call has run on the device, HC_ERR_CUDA on a runtime error.  Allocates
 * nothing. */
int hc_read_noalloc_check(void);

/* Static text for a status code. */
const char* hc_status_str(int status);

/* CUDA-graph helpers for callers without a graph API of their own.
 * hc_graph_begin starts a thread-local stream capture on `stream`;
 * hc_graph_end ends it and instantiates the graph into *exec;
 * hc_graph_launch replays it on `stream`; hc_graph_destroy frees it. */
int hc_graph_begin(hc_stream_t stream);
int hc_graph_end(hc_stream_t stream, hc_graph_t* exec);
int hc_graph_launch(hc_graph_t exec, hc_stream_t stream);
void hc_graph_destroy(hc_graph_t exec);

#ifdef __cplusplus
}
#endif

#endif /* HC_READ_H */
