// Host side of the C ABI declared in include/hc_read.h: handle and scratch
// management, argument validation, kernel selection and launch with
// programmatic dependent launch, CUDA-graph helpers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <algorithm>
#include <mutex>
#include <new>
#include <numeric>
#include <unordered_map>
#include <vector>

#include "hc_kernels.cuh"
#include "hc_kernels_tc.cuh"
#include "hc_kernels_umma.cuh"
#include "hc_kernels_wide.cuh"
#include "hc_read.h"
#include "hc_window.cuh"

#define HC_EXPORT extern "C" __attribute__((visibility("default")))

// Streams hc_read_batch spreads independent reads over.  Measured on GB300
// (cold reads, d = 2560): one stream 5.2 us per read at T = 1; 4 / 6 / 8
// streams 2.60 / 2.52 / 2.51 us; at T = 8 6.9 -> 3.88 / 3.79 / 3.82 us.
constexpr int kBatchLanes = 6;

// Reads of at least this many tokens (d = 2560) take the wide tensor-memory
// pair (hc_kernels_wide.cuh).
constexpr int kWideMinT = 9;
// ... and from this many tokens the wide up kernel runs 32-token passes.
constexpr int kUpPass32MinT = 49;

// The tensor maps of the weight matrices a handle has seen, by address:
// W_down in boxes of 64 columns x 64 rows (the tensor-memory down kernels),
// W_up in boxes of 64 columns x 16 rows (the wide up kernel).  A map holds
// only the address, sizes and strides, so an entry stays valid for the
// handle's geometry whatever the memory holds.
struct MapCache {
  static constexpr int kSlots = 64;
  const void* base[2][kSlots];  // [0] W_down, [1] W_up
  CUtensorMap maps[2][kSlots];
  unsigned next[2];
};

struct hc_read_s {
  int n, d, K, T_max, device;
  float eps;
  void* scratch;
  size_t scratch_bytes;
  float* part[2];  // two slots of [4][T_max][K] rs-scaled per-stream partials
  unsigned* err;
  int parity;      // slot of the next read
  // Persistent multi-read kernel (d = 2560, K = 320 only): exchange packets,
  // published output tiles, per-CTA epoch bases, abort word.
  bool window;     // the kernel's 128 CTAs fit co-resident on this device
  unsigned* xbuf;
  unsigned* xss;
  unsigned* mbuf;
  unsigned* gen;
  size_t window_bytes;  // xbuf, mbuf, gen, abort word: zeroed by hc_read_reset
  unsigned* abort_flag;
  // Internal streams on which hc_read_batch runs groups of reads that share
  // no memory side by side (each with its own partial-sum slots), forked from
  // and joined back into the caller's stream with events.
  struct Lane {
    cudaStream_t st;
    cudaEvent_t done;
    float* part[2];
    int parity;
  } lanes[kBatchLanes];
  MapCache* map_cache;  // created on first use
  // W_down -> its tile-ordered copies, W_up -> its (hc_read_register_down_tiles,
  // hc_read_register_up_tiles); created on first use.
  std::unordered_map<const void*, const void*>* down_tiles;
  std::unordered_map<const void*, const void*>* up_tiles;
  unsigned long long wait_ns;  // limit of the down kernels' first bulk-copy wait (0: the default)
  bool overlap;       // reads may overlap their predecessor (independent mode), hc_read_set_overlap
  int nlanes;         // lanes created (0: batches run on the caller's stream only)
  int batch_lanes;    // most lanes a batch may use (hc_read_set_batch_lanes)
  cudaEvent_t fork;
};

namespace {

using hc::DownArgs;
using hc::UpArgs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The batch lanes' streams and events (on the current device).
cudaError_t create_lanes(hc_read_s* h) {
  cudaError_t e = cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  for (int l = 0; l < kBatchLanes; ++l) {
    e = cudaStreamCreateWithFlags(&h->lanes[l].st, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
    e = cudaEventCreateWithFlags(&h->lanes[l].done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      cudaStreamDestroy(h->lanes[l].st);
      return e;
    }
    h->nlanes = l + 1;
  }
  h->batch_lanes = h->nlanes;
  return cudaSuccess;
}

void destroy_lanes(hc_read_s* h) {
  for (int l = 0; l < h->nlanes; ++l) {
    cudaEventDestroy(h->lanes[l].done);
    cudaStreamDestroy(h->lanes[l].st);
  }
  if (h->fork != nullptr) cudaEventDestroy(h->fork);
  h->nlanes = 0;
  h->fork = nullptr;
}

// Launch configuration with programmatic dependent launch and, when
// cluster_x > 1, thread-block clusters of cluster_x CTAs along x.
cudaLaunchConfig_t pdl_config(dim3 grid, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr,
                              unsigned cluster_x, unsigned threads = hc::kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cfg;
}

template <int D, int KD, bool Q8, int TT>
cudaError_t configure_down_s() {
  return cudaFuncSetAttribute(hc::hc_down_s_kernel<D, KD, Q8, TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              hc::StreamGeo<D, KD, Q8, TT>::BYTES);
}

template <int D, int KD, int TT>
cudaError_t configure_one() {
  cudaError_t e = cudaFuncSetAttribute(hc::hc_down_kernel<D, KD, TT, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       hc::DownSmem<D, KD, TT>::BYTES_MAX);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(hc::hc_down_kernel<D, KD, TT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           hc::DownSmem<D, KD, TT>::BYTES_MAX);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(hc::hc_up_kernel<D, KD, TT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              hc::UpSmem<D, KD, TT>::BYTES_MAX);
}

template <int D, int KD, int NT, int Q8>
cudaError_t configure_tc() {
  cudaError_t e = cudaFuncSetAttribute(hc::hc_down_tc_kernel<D, KD, NT, Q8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       hc::DownTcSmem<D, KD, NT, Q8>::BYTES_MAX);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(hc::hc_up_tc_kernel<D, KD, NT, Q8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              hc::UpTcSmem<D, KD, NT, Q8>::BYTES_MAX);
}

template <int D, int KD>
cudaError_t configure_umma() {
  return cudaFuncSetAttribute(hc::hc_down_u_kernel<D, KD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              hc::UGeo<D, KD>::DN_BYTES);
}

template <int D, int KD>
cudaError_t configure_wide() {
  using W = hc::WGeo<D, KD>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(hc::hc_down_w1_kernel<D, KD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                W::d1_bytes(W::TP))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(hc::hc_down_w_kernel<D, KD, 2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                W::DN_BYTES_MAX)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(hc::hc_down_w_kernel<D, KD, 2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                W::DN_BYTES_MAX)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(hc::hc_down_w_kernel<D, KD, 4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                W::DN_BYTES_MAX)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(hc::hc_down_w_kernel<D, KD, 4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                W::DN_BYTES_MAX)) != cudaSuccess)
    return e;
  using P16 = hc::UpPass<D, KD, 16>;
  using P32 = hc::UpPass<D, KD, 32>;
  if ((e = cudaFuncSetAttribute(hc::hc_up_w_kernel<D, KD, false, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                P16::up_bytes(16))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(hc::hc_up_w_kernel<D, KD, true, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                P16::up_bytes(kUpPass32MinT - 1))) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(hc::hc_up_w_kernel<D, KD, true, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              P32::up_bytes(W::TW));
}

template <int D, int KD>
cudaError_t configure_geometry() {
  cudaError_t e;
  if constexpr (D == 2560) {
    if ((e = configure_down_s<D, KD, false, 1>()) != cudaSuccess || (e = configure_down_s<D, KD, true, 1>()) != cudaSuccess ||
        (e = configure_down_s<D, KD, true, 2>()) != cudaSuccess ||
        (e = cudaFuncSetAttribute(hc::hc_up_kernel<D, KD, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  hc::UpSmem<D, KD, 1, true>::BYTES_MAX)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(hc::hc_up_kernel<D, KD, 2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  hc::UpSmem<D, KD, 2, true>::BYTES_MAX)) != cudaSuccess)
      return e;
    if ((e = configure_umma<D, KD>()) != cudaSuccess) return e;
    if ((e = configure_wide<D, KD>()) != cudaSuccess) return e;
  }
  if ((e = configure_one<D, KD, 1>()) != cudaSuccess) return e;
  if ((e = configure_tc<D, KD, 1, 0>()) != cudaSuccess) return e;
  if ((e = configure_tc<D, KD, 2, 0>()) != cudaSuccess) return e;
  if ((e = configure_tc<D, KD, 1, 1>()) != cudaSuccess) return e;
  if ((e = configure_tc<D, KD, 1, 2>()) != cudaSuccess) return e;
  return configure_tc<D, KD, 2, 2>();
}

template <int D, int KD, int TT>
cudaError_t launch_pair(const DownArgs& da, const UpArgs& ua, cudaStream_t st) {
  using G = hc::Geo<D, KD>;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t c1 = pdl_config(dim3(G::SLABS, G::ROW_GROUPS),
                                      hc::DownSmem<D, KD, TT>::bytes(da.T), st, attr,
                                      G::SLABS_PER_STREAM);
  cudaError_t e = da.W_tiles ? cudaLaunchKernelEx(&c1, hc::hc_down_kernel<D, KD, TT, true>, da)
                             : cudaLaunchKernelEx(&c1, hc::hc_down_kernel<D, KD, TT, false>, da);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr2[2];
  cudaLaunchConfig_t c2 = pdl_config(dim3(G::UP_CTAS), hc::UpSmem<D, KD, TT>::bytes(ua.T), st,
                                      attr2, 1);
  return cudaLaunchKernelEx(&c2, hc::hc_up_kernel<D, KD, TT>, ua);
}

// The stream-wide down kernel (no cluster), TT tokens held in registers.
template <int D, int KD, bool Q8, int TT>
cudaError_t launch_down_s(const DownArgs& da, cudaStream_t st) {
  using S = hc::StreamGeo<D, KD, Q8, TT>;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t c = pdl_config(dim3(S::ROW_GROUPS, hc::kStreams), S::BYTES, st, attr, 1);
  return cudaLaunchKernelEx(&c, hc::hc_down_s_kernel<D, KD, Q8, TT>, da);
}

// T = 1 at d = 2560: the stream-wide down kernel (no cluster) with the
// CUDA-core up kernel.
template <int D, int KD>
cudaError_t launch_pair_s(const DownArgs& da, const UpArgs& ua, cudaStream_t st) {
  using G = hc::Geo<D, KD>;
  cudaError_t e = launch_down_s<D, KD, false, 1>(da, st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr2[2];
  cudaLaunchConfig_t c2 = pdl_config(dim3(G::UP_CTAS), hc::UpSmem<D, KD, 1>::bytes(ua.T), st, attr2, 1);
  return cudaLaunchKernelEx(&c2, hc::hc_up_kernel<D, KD, 1>, ua);
}

template <int D, int KD, int NT, int Q8 = 0>
cudaError_t launch_pair_tc(const DownArgs& da, const UpArgs& ua, cudaStream_t st) {
  using G = hc::Geo<D, KD>;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t c1 = pdl_config(dim3(G::SLABS, G::ROW_GROUPS),
                                      hc::DownTcSmem<D, KD, NT, Q8>::bytes(da.T), st, attr,
                                      G::SLABS_PER_STREAM);
  cudaError_t e = cudaLaunchKernelEx(&c1, hc::hc_down_tc_kernel<D, KD, NT, Q8>, da);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr2[2];
  cudaLaunchConfig_t c2 = pdl_config(dim3(G::UP_CTAS), hc::UpTcSmem<D, KD, NT, Q8>::bytes(ua.T), st,
                                      attr2, 1);
  return cudaLaunchKernelEx(&c2, hc::hc_up_tc_kernel<D, KD, NT, Q8>, ua);
}

// The Q8_0 CUDA-core up kernel (token groups of TT).
template <int D, int KD, int TT>
cudaError_t launch_up_q8_cc(const UpArgs& ua, cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t c = pdl_config(dim3(hc::Geo<D, KD>::UP_CTAS), hc::UpSmem<D, KD, TT, true>::bytes(ua.T), st,
                                     attr, 1);
  return cudaLaunchKernelEx(&c, hc::hc_up_kernel<D, KD, TT, true>, ua);
}

// The driver's tensor-map encoder (null when the driver does not offer it;
// the reads then take the mma.sync kernels).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor map of a row-major BF16 matrix [rows][cols] read in boxes of 64
// columns x box_rows rows with the 128-byte swizzle.
bool encode_bf16_tiles(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-memory down kernel (all T <= 8 in one pass) and the mma.sync
// up kernel of 4-token groups (d = 2560, K = 320), for T = 5..8.  Measured
// on six streams with independent reads: 3.42 -> 3.14 us per read at T = 5,
// 3.56 -> 3.26 at T = 8; at T = 2..4 the pair is 2-3 % slower than the
// mma.sync pair, which keeps those.  The choice depends on the read's shape
// only, never on what ran before it, so a read's bits do not depend on its
// history (direct calls, batches and graph replays agree).
template <int D, int KD>
cudaError_t launch_pair_u(const DownArgs& da, const UpArgs& ua, const CUtensorMap& w_down, cudaStream_t st) {
  using U = hc::UGeo<D, KD>;
  using G = hc::Geo<D, KD>;
  hc::DownUArgs dargs;
  dargs.w = w_down;
  dargs.a = da;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t c1 = pdl_config(dim3(U::CHUNKS, U::ROW_GROUPS), U::DN_BYTES, st, attr, U::CPS, U::THREADS);
  cudaError_t e = cudaLaunchKernelEx(&c1, hc::hc_down_u_kernel<D, KD>, dargs);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr2[2];
  cudaLaunchConfig_t c2 = pdl_config(dim3(G::UP_CTAS), hc::UpTcSmem<D, KD, 1>::bytes(ua.T), st, attr2, 1);
  return cudaLaunchKernelEx(&c2, hc::hc_up_tc_kernel<D, KD, 1>, ua);
}

// The wide tensor-memory pair (d = 2560, K = 320, T >= kWideMinT): both
// projections on tcgen05 with every weight byte read once for all T tokens,
// tokens in passes of 16, the up kernel's lo combined once per cluster;
// shared memory sized by T, three CTAs per SM.
template <int D, int KD>
cudaError_t launch_pair_w(const DownArgs& da, const UpArgs& ua, const CUtensorMap& w_down, const CUtensorMap& w_up,
                          cudaStream_t st) {
  using W = hc::WGeo<D, KD>;
  hc::DownUArgs dargs;
  dargs.w = w_down;
  dargs.a = da;
  cudaLaunchAttribute attr[2];
  // T <= 16: the single-pass instantiations.
  const bool multi = da.T > W::TP;
  cudaLaunchConfig_t c1 = pdl_config(dim3(W::CHUNKS, W::ROW_GROUPS), W::dn_bytes(da.T), st, attr, W::CPS, W::THREADS);
  // Down kernel: T <= 16 the single pass (measured 4 % faster there than
  // the K-slice ring), above it the ring with 2 or 4 tokens per staging
  // thread (8-10 % faster at T = 17..48 than 16-token passes).
  if (da.T <= W::TP) c1.dynamicSmemBytes = W::d1_bytes(da.T);
  const bool hasp = da.P != nullptr;
  cudaError_t e = da.T <= W::TP ? cudaLaunchKernelEx(&c1, hc::hc_down_w1_kernel<D, KD>, dargs)
                  : da.T <= 32  ? (hasp ? cudaLaunchKernelEx(&c1, hc::hc_down_w_kernel<D, KD, 2, true>, dargs)
                                        : cudaLaunchKernelEx(&c1, hc::hc_down_w_kernel<D, KD, 2, false>, dargs))
                  : hasp        ? cudaLaunchKernelEx(&c1, hc::hc_down_w_kernel<D, KD, 4, true>, dargs)
                                : cudaLaunchKernelEx(&c1, hc::hc_down_w_kernel<D, KD, 4, false>, dargs);
  if (e != cudaSuccess) return e;
  hc::UpWArgs uargs;
  uargs.w = w_up;
  uargs.a = ua;
  cudaLaunchAttribute attr2[2];
  // Up kernel: one 16-token pass (T <= 16), 16-token passes (three CTAs per
  // SM, T <= 48), or 32-token passes (two CTAs per SM either way, half the
  // passes).
  if (ua.T >= kUpPass32MinT) {
    cudaLaunchConfig_t c2 = pdl_config(dim3(W::UP_CTAS), hc::UpPass<D, KD, 32>::up_bytes(ua.T), st, attr2, W::UCL,
                                       W::THREADS);
    return cudaLaunchKernelEx(&c2, hc::hc_up_w_kernel<D, KD, true, 32>, uargs);
  }
  cudaLaunchConfig_t c2 = pdl_config(dim3(W::UP_CTAS), hc::UpPass<D, KD, 16>::up_bytes(ua.T), st, attr2, W::UCL,
                                     W::THREADS);
  return multi ? cudaLaunchKernelEx(&c2, hc::hc_up_w_kernel<D, KD, true, 16>, uargs)
               : cudaLaunchKernelEx(&c2, hc::hc_up_w_kernel<D, KD, false, 16>, uargs);
}

// From T = 2 on the tensor-core kernels are faster on GB300 (measured: T=2
// 6.1 vs 6.7 us, T=8 7.9 vs 11.1 us per read); at T = 1 the CUDA-core kernels
// are (5.2 vs 6.0 us): the MMA path stages four tokens there.  At d = 2560,
// up to T = 8, the kernels of one 4-token group run the tokens in one or two
// groups: they fit four CTAs per SM, and reads of a batch overlap better
// (measured on six streams at T = 6: 3.50 us per read against 3.83 with
// 8-token groups).  At d = 4096 (two CTAs per SM either way) 8-token groups
// stay faster from T = 5 (8.5 against 9.0 us).
template <int D, int KD>
cudaError_t launch_geometry(int T, const DownArgs& da, const UpArgs& ua, cudaStream_t st,
                            const CUtensorMap* w_down, const CUtensorMap* w_up = nullptr) {
  if constexpr (D == 2560) {
    if (T == 1) return launch_pair_s<D, KD>(da, ua, st);
  } else {
    if (T == 1) return launch_pair<D, KD, 1>(da, ua, st);
  }
  if constexpr (D == 2560) {
    if (w_down != nullptr && w_up != nullptr && T >= kWideMinT) return launch_pair_w<D, KD>(da, ua, *w_down, *w_up, st);
    if (w_down != nullptr && T <= hc::UGeo<D, KD>::TMAX) return launch_pair_u<D, KD>(da, ua, *w_down, st);
  }
  constexpr int kOneGroupMaxT = D == 2560 ? 8 : 4;
  return T <= kOneGroupMaxT ? launch_pair_tc<D, KD, 1>(da, ua, st) : launch_pair_tc<D, KD, 2>(da, ua, st);
}

// The Q8_0 read: at T = 1, 2 and d = 2560 the stream-wide down kernel and the
// CUDA-core up kernel, elsewhere the tensor-core kernels, token groups as for
// BF16.  One token group: quants
// decoded in registers (mode 1); several groups: the tile widened once in
// shared memory (mode 2), reused by every group.
template <int D, int KD>
cudaError_t launch_geometry_q8(int T, const DownArgs& da, const UpArgs& ua, cudaStream_t st) {
  constexpr int kOneGroupMaxT = D == 2560 ? 8 : 4;
  if constexpr (D == 2560) {
    if (T == 1) {
      // The stream-wide down kernel over the quants (no cluster) and the
      // CUDA-core up kernel: for one token its decoding costs the chain less
      // than the tensor-core kernel's fragment decoding.
      cudaError_t e = launch_down_s<D, KD, true, 1>(da, st);
      if (e != cudaSuccess) return e;
      return launch_up_q8_cc<D, KD, 1>(ua, st);
    }
    if (T == 2) {
      // The stream-wide down kernel with both tokens in registers and the
      // CUDA-core up kernel with both tokens.  Four tokens (T = 3, 4) cost
      // more than they save in either kernel: 96 registers a thread in the
      // down kernel, spills at 64 in the up kernel.
      cudaError_t e = launch_down_s<D, KD, true, 2>(da, st);
      if (e != cudaSuccess) return e;
      return launch_up_q8_cc<D, KD, 2>(ua, st);
    }
  }
  if (T <= 4) return launch_pair_tc<D, KD, 1, 1>(da, ua, st);
  return T <= kOneGroupMaxT ? launch_pair_tc<D, KD, 1, 2>(da, ua, st) : launch_pair_tc<D, KD, 2, 2>(da, ua, st);
}

// Q8_0 weights of a read (quants and block scales of both projections).
struct Q8Weights {
  const int8_t* Wd_q;
  const uint16_t* Wd_scale;
  const int8_t* Wu_q;
  const uint16_t* Wu_scale;
};

// ---- Which reads may overlap their predecessor.
// For every (device, stream) the output ranges of the last read enqueued
// there are kept.  A read whose inputs overlap none of them runs in
// independent mode.  Work the caller enqueues between two reads is always
// waited for in full (only kernels of this library trigger their dependents
// early), so only the previous read matters.
struct Range {
  uintptr_t lo, hi;
};

struct LastRead {
  int device;
  void* stream;
  bool valid;
  Range outs[5];  // out, mean, lo, r_out, rs
};

constexpr int kTrackedStreams = 64;
std::mutex g_track_mutex;
LastRead g_track[kTrackedStreams];
unsigned g_track_next;

Range range_of(const void* p, size_t bytes) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(p);
  return Range{b, p != nullptr ? b + bytes : b};
}

// One read as the host handles it: BF16 projections (W_down, W_up) or Q8_0
// ones (q8.Wd_q set, W_down and W_up null).
struct ReadDesc {
  const float* R;
  const float* pending;
  const float* w_norm;
  const float* gate;
  const uint16_t* W_down;
  const uint16_t* W_up;
  Q8Weights q8;
  float* out;
  float* mean;
  float* lo;
  bool is_q8() const { return q8.Wd_q != nullptr; }
};

constexpr int kReadInputs = 8;

// The byte ranges a T-token read takes as inputs: R, pending, w_norm, gate,
// the two projections and (Q8_0) their block scales.
void input_ranges(const ReadDesc& q, size_t N, int K, int T, Range (&r)[kReadInputs]) {
  r[0] = range_of(q.R, T * N * 4);
  r[1] = range_of(q.pending, T * N * 4);
  r[2] = range_of(q.w_norm, N * 4);
  r[3] = range_of(q.gate, N * 4);
  if (q.is_q8()) {
    r[4] = range_of(q.q8.Wd_q, N * K);
    r[5] = range_of(q.q8.Wu_q, N * K);
    r[6] = range_of(q.q8.Wd_scale, N * K / 32 * 2);
    r[7] = range_of(q.q8.Wu_scale, N * K / 32 * 2);
  } else {
    r[4] = range_of(q.W_down, N * K * 2);
    r[5] = range_of(q.W_up, N * K * 2);
    r[6] = range_of(nullptr, 0);
    r[7] = range_of(nullptr, 0);
  }
}

// Its outputs out, mean and lo.
void output_ranges(const ReadDesc& q, int n, int d, int K, int T, Range (&r)[3]) {
  r[0] = range_of(q.out, (size_t)T * n * d * 4);
  r[1] = range_of(q.mean, (size_t)T * d * 4);
  r[2] = range_of(q.lo, (size_t)T * K * 4);
}

ReadDesc from_desc(const hc_read_desc& d) {
  return ReadDesc{d.R, d.pending, d.w_norm, d.gate, d.W_down, d.W_up, Q8Weights{}, d.out, d.mean, d.lo};
}

ReadDesc from_desc(const hc_read_q8_desc& d) {
  return ReadDesc{d.R,      d.pending, d.w_norm, d.gate, nullptr, nullptr,
                  Q8Weights{d.Wd_q, d.Wd_scale, d.Wu_q, d.Wu_scale}, d.out, d.mean, d.lo};
}

// Records this read's outputs for (device, stream); returns whether its inputs
// are disjoint from the outputs of the previous read recorded there.
bool record_and_check(int device, void* stream, const Range (&ins)[kReadInputs], const Range (&outs)[5]) {
  std::lock_guard<std::mutex> lock(g_track_mutex);
  LastRead* slot = nullptr;
  for (auto& e : g_track) {
    if (e.valid && e.device == device && e.stream == stream) {
      slot = &e;
      break;
    }
  }
  bool independent = false;
  if (slot != nullptr) {
    independent = true;
    for (const Range& i : ins) {
      if (i.lo == i.hi) continue;
      for (const Range& o : slot->outs) {
        if (o.lo != o.hi && i.lo < o.hi && o.lo < i.hi) independent = false;
      }
    }
  } else {
    slot = &g_track[g_track_next++ % kTrackedStreams];
  }
  slot->device = device;
  slot->stream = stream;
  slot->valid = true;
  for (int k = 0; k < 5; ++k) slot->outs[k] = outs[k];
  return independent;
}

// Drops what is kept for (device, stream): the next read there waits for
// everything before it in full.
void forget_stream(int device, void* stream) {
  std::lock_guard<std::mutex> lock(g_track_mutex);
  for (auto& e : g_track) {
    if (e.valid && e.device == device && e.stream == stream) e.valid = false;
  }
}

// ---- Persistent multi-read kernel (hc_window.cuh), d = 2560, K = 320, T <= 4.
using WinG1 = hc::WinGeo<2560, 320, 1>;
constexpr size_t kXbufWords = (size_t)hc::kWinXSlots * hc::kWinCluster * (hc::kWinCtas / hc::kWinCluster) *
                              hc::kWinTmaxAlloc * WinG1::KQ;
constexpr size_t kXssWords = (size_t)hc::kWinXSlots * hc::kWinTmaxAlloc * (hc::kWinCtas / hc::kWinCluster) * 2;
constexpr size_t kMbufWords = (size_t)hc::kWinXSlots * hc::kStreams * hc::kWinTmaxAlloc * 2560;

cudaLaunchConfig_t window_config(cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(hc::kWinCtas);
  cfg.blockDim = dim3(WinG1::THREADS);
  cfg.dynamicSmemBytes = WinG1::BYTES;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = hc::kWinCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // The CTAs wait on one another: they must all be resident at once.
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[2].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 3;
  return cfg;
}

// Whether the current device can hold the window kernel's 32 clusters of
// four CTAs (one CTA per SM) at once.
bool window_fits() {
  if (cudaFuncSetAttribute(hc::hc_window_kernel<2560, 320, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           WinG1::BYTES) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchAttribute attr[3];
  cudaLaunchConfig_t cfg = window_config(nullptr, attr);
  cfg.numAttrs = 1;  // the cluster shape only
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, hc::hc_window_kernel<2560, 320, 1>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return clusters >= hc::kWinCtas / hc::kWinCluster;
}

bool overlaps(const Range& a, const Range& b) {
  return a.lo != a.hi && b.lo != b.hi && a.lo < b.hi && b.lo < a.hi;
}

bool geometry_supported(int n, int d, int K) {
  return n == hc::kStreams && ((d == 2560 && K == 320) || (d == 4096 && K == 512));
}

}  // namespace

HC_EXPORT int hc_read_create(hc_read_t* out, int n, int d, int K, int T_max, float eps, int device) {
  if (out == nullptr) return HC_ERR_ARG;
  *out = nullptr;
  if (!geometry_supported(n, d, K)) return HC_ERR_SHAPE;
  if (T_max < 1 || T_max > hc::kMaxT || !(eps >= 0.0f) || device < 0) return HC_ERR_ARG;

  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return HC_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return HC_ERR_CUDA;

  cudaError_t e = (d == 2560) ? configure_geometry<2560, 320>() : configure_geometry<4096, 512>();
  hc_read_s* h = nullptr;
  if (e == cudaSuccess) {
    h = new (std::nothrow) hc_read_s();
    if (h == nullptr) {
      cudaSetDevice(prev);
      return HC_ERR_ARG;
    }
    h->n = n;
    h->d = d;
    h->K = K;
    h->T_max = T_max;
    h->device = device;
    h->eps = eps;
    h->wait_ns = 0;
    h->overlap = true;
    const size_t part_b = round_up((size_t)n * T_max * K * sizeof(float), 256);
    const size_t err_b = 256;
    h->window = d == 2560 && window_fits();
    const size_t xbuf_b = h->window ? round_up(kXbufWords * 4, 256) : 0;
    const size_t xss_b = h->window ? round_up(kXssWords * 4, 256) : 0;
    const size_t mbuf_b = h->window ? round_up(kMbufWords * 4, 256) : 0;
    const size_t gen_b = h->window ? round_up(hc::kWinCtas * sizeof(unsigned), 256) + 256 : 0;
    const size_t lanes_b = kBatchLanes * 2 * part_b;
    h->scratch_bytes = 2 * part_b + err_b + xbuf_b + xss_b + mbuf_b + gen_b + lanes_b;
    e = cudaMalloc(&h->scratch, h->scratch_bytes);
    if (e == cudaSuccess) {
      char* base = static_cast<char*>(h->scratch);
      h->part[0] = reinterpret_cast<float*>(base);
      h->part[1] = reinterpret_cast<float*>(base + part_b);
      h->err = reinterpret_cast<unsigned*>(base + 2 * part_b);
      h->parity = 0;
      // Window state, contiguous (hc_read_reset zeroes it in one go):
      // xbuf | xss | mbuf | gen[128] | abort word.
      char* wb = base + 2 * part_b + err_b;
      h->window_bytes = xbuf_b + xss_b + mbuf_b + gen_b;
      h->xbuf = h->window ? reinterpret_cast<unsigned*>(wb) : nullptr;
      h->xss = h->window ? reinterpret_cast<unsigned*>(wb + xbuf_b) : nullptr;
      h->mbuf = h->window ? reinterpret_cast<unsigned*>(wb + xbuf_b + xss_b) : nullptr;
      h->gen = h->window ? reinterpret_cast<unsigned*>(wb + xbuf_b + xss_b + mbuf_b) : nullptr;
      h->abort_flag = h->window ? reinterpret_cast<unsigned*>(wb + h->window_bytes - 256) : nullptr;
      char* lb = wb + h->window_bytes;
      for (int l = 0; l < kBatchLanes; ++l) {
        h->lanes[l].part[0] = reinterpret_cast<float*>(lb + (2 * l) * part_b);
        h->lanes[l].part[1] = reinterpret_cast<float*>(lb + (2 * l + 1) * part_b);
        h->lanes[l].parity = 0;
      }
      e = cudaMemset(h->scratch, 0, h->scratch_bytes);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e == cudaSuccess) e = create_lanes(h);
    } else {
      h->scratch = nullptr;
    }
  }
  cudaSetDevice(prev);
  if (e != cudaSuccess) {
    if (h != nullptr) {
      if (cudaSetDevice(h->device) == cudaSuccess) {
        destroy_lanes(h);
        if (h->scratch != nullptr) cudaFree(h->scratch);
        cudaSetDevice(prev);
      }
      delete h;
    }
    return HC_ERR_CUDA;
  }
  *out = h;
  return HC_OK;
}

namespace {

// Whether a BF16 read takes a tensor-memory down kernel: d = 2560 and
// 5 <= T <= 8 (hc_down_u_kernel) or T >= kWideMinT (the wide pair, whose up
// kernel also takes a W_up map).
bool takes_umma(int d, int T) { return d == 2560 && T > 4 && (T <= hc::UGeo<2560, 320>::TMAX || T >= kWideMinT); }
bool takes_wide(int d, int T) { return d == 2560 && T >= kWideMinT; }

// A weight map from the handle's cache (which = 0: W_down [K][N] in boxes of
// 64 x 64; 1: W_up [N][K] in boxes of 64 x 16); null when the driver offers
// no tensor-map encoder.
const CUtensorMap* weight_map(hc_read_t h, int which, const void* base) {
  MapCache* c = h->map_cache;
  if (c == nullptr) {
    c = h->map_cache = new (std::nothrow) MapCache();
    if (c == nullptr) return nullptr;
  }
  for (int i = 0; i < MapCache::kSlots; ++i) {
    if (c->base[which][i] == base) return &c->maps[which][i];
  }
  const int i = (int)(c->next[which]++ % MapCache::kSlots);
  c->base[which][i] = nullptr;
  const uint64_t N = (uint64_t)h->n * h->d;
  const bool done = which == 0 ? encode_bf16_tiles(&c->maps[which][i], base, h->K, N, 64)
                               : encode_bf16_tiles(&c->maps[which][i], base, N, h->K, 16);
  if (!done) return nullptr;
  c->base[which][i] = base;
  return &c->maps[which][i];
}

// The W_down tensor map of a read that takes a tensor-memory down kernel;
// null: the read takes the mma.sync kernels.
const CUtensorMap* down_map_for(hc_read_t h, const ReadDesc& q, int T) {
  if (q.is_q8() || !takes_umma(h->d, T)) return nullptr;
  return weight_map(h, 0, q.W_down);
}

// The W_up tensor map of a read that takes the wide pair (else null).
const CUtensorMap* up_map_for(hc_read_t h, const ReadDesc& q, int T) {
  if (q.is_q8() || !takes_wide(h->d, T)) return nullptr;
  return weight_map(h, 1, q.W_up);
}

// The tile-ordered copy registered for a weight, or null.
const void* tiles_for(const std::unordered_map<const void*, const void*>* m, const void* W) {
  if (m == nullptr) return nullptr;
  const auto it = m->find(W);
  return it == m->end() ? nullptr : it->second;
}

// The down-tile buffer: the 32-row tiles, then (d = 2560, where the
// tensor-memory kernels run) the 64-row swizzled tiles.
template <int D, int KD>
constexpr size_t down_tiles_rows_bytes() {
  using G = hc::Geo<D, KD>;
  return (size_t)G::ROW_GROUPS * G::SLABS * G::DN_ROWS * G::DN_PITCH;
}
constexpr size_t kSwTilesBytes = (size_t)4 * 2560 * 320 * 2;  // all of W_down or W_up at d = 2560, K = 320

size_t down_tiles_bytes(int d) {
  return d == 2560 ? down_tiles_rows_bytes<2560, 320>() + kSwTilesBytes : down_tiles_rows_bytes<4096, 512>();
}

template <int D, int KD>
cudaError_t launch_pack_down_tiles(const void* W_down, void* tiles, cudaStream_t st) {
  using G = hc::Geo<D, KD>;
  hc::hc_pack_down_tiles_kernel<D, KD><<<dim3(G::SLABS, G::ROW_GROUPS), hc::kThreads, 0, st>>>(
      static_cast<const uint16_t*>(W_down), static_cast<uint16_t*>(tiles));
  if constexpr (D == 2560) {
    using W = hc::WGeo<D, KD>;
    hc::hc_pack_down_sw_kernel<D, KD><<<dim3(W::CHUNKS, W::ROW_GROUPS), 256, 0, st>>>(
        static_cast<const uint16_t*>(W_down),
        reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(tiles) + down_tiles_rows_bytes<D, KD>()));
  }
  return cudaGetLastError();
}

// Enqueues one validated read on `st` with partial-sum slot `part` (the two
// kernels of the read; the caller alternates between its two slots).
int enqueue_read(hc_read_t h, float* part, int device, const ReadDesc& q, int T, float* r_out, float* rs,
                 cudaStream_t st, bool on_lanes = false) {
  const size_t N = (size_t)h->n * h->d;
  Range ins[kReadInputs];
  input_ranges(q, N, h->K, T, ins);
  const Range outs[5] = {range_of(q.out, T * N * 4),  range_of(q.mean, (size_t)T * h->d * 4),
                         range_of(q.lo, (size_t)T * h->K * 4), range_of(r_out, T * N * 4),
                         range_of(rs, (size_t)T * h->n * 4)};
  const int independent = (record_and_check(device, st, ins, outs) && h->overlap) ? 1 : 0;

  DownArgs da{};
  da.R = q.R;
  da.P = q.pending;
  da.w_norm = q.w_norm;
  da.W_down = q.W_down;
  da.W_tiles = q.is_q8() ? nullptr : tiles_for(h->down_tiles, q.W_down);
  da.W_tiles_sw = (da.W_tiles != nullptr && h->d == 2560)
                      ? static_cast<const unsigned char*>(da.W_tiles) + down_tiles_rows_bytes<2560, 320>()
                      : nullptr;
  da.Wq = q.q8.Wd_q;
  da.Wscale = q.q8.Wd_scale;
  da.part = part;
  da.err = h->err;
  da.rs_out = rs;
  da.T = T;
  da.T_max = h->T_max;
  da.independent = independent;
  da.late_launch = on_lanes ? 1 : 0;
  da.eps = h->eps;
  da.wait_ns = h->wait_ns;

  UpArgs ua{};
  ua.R = q.R;
  ua.P = q.pending;
  ua.gate = q.gate;
  ua.W_up = q.W_up;
  ua.Wq = q.q8.Wu_q;
  ua.Wscale = q.q8.Wu_scale;
  ua.part = part;
  ua.out = q.out;
  ua.mean = q.mean;
  ua.lo = q.lo;
  ua.r_out = r_out;
  ua.err = h->err;
  ua.T = T;
  ua.T_max = h->T_max;
  ua.independent = independent;
  ua.W_up_tiles = q.is_q8() ? nullptr : tiles_for(h->up_tiles, q.W_up);

  cudaError_t e;
  if (q.is_q8()) {
    e = (h->d == 2560) ? launch_geometry_q8<2560, 320>(T, da, ua, st) : launch_geometry_q8<4096, 512>(T, da, ua, st);
  } else {
    e = (h->d == 2560) ? launch_geometry<2560, 320>(T, da, ua, st, down_map_for(h, q, T), up_map_for(h, q, T))
                       : launch_geometry<4096, 512>(T, da, ua, st, nullptr);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky launch error for this thread
    return HC_ERR_CUDA;
  }
  return HC_OK;
}

// Argument checks of one read: required pointers set, every pointer 16-byte
// aligned (Q8_0 scales included: they are copied in 8- and 16-byte pieces).
int check_read(const ReadDesc& q, const float* r_out, const float* rs) {
  if (!q.R || !q.w_norm || !q.gate || !q.out || !q.mean || !q.lo) return HC_ERR_ARG;
  if (q.is_q8() ? (!q.q8.Wd_scale || !q.q8.Wu_q || !q.q8.Wu_scale || q.W_down || q.W_up) : (!q.W_down || !q.W_up)) {
    return HC_ERR_ARG;
  }
  const void* ptrs[] = {q.R,           q.w_norm,      q.W_down, q.W_up, q.q8.Wd_q, q.q8.Wd_scale, q.q8.Wu_q,
                        q.q8.Wu_scale, q.gate,        q.pending, q.out, q.mean,    q.lo,          r_out,
                        rs};
  for (const void* p : ptrs) {
    if (p != nullptr && !aligned16(p)) return HC_ERR_ALIGN;
  }
  return HC_OK;
}

// One checked read on the handle's own partial-sum slots.
int single_read(hc_read_t h, const ReadDesc& q, int T, float* r_out, float* rs, hc_stream_t stream) {
  if (h == nullptr) return HC_ERR_ARG;
  if (T < 1 || T > h->T_max) return HC_ERR_ARG;
  const int c = check_read(q, r_out, rs);
  if (c != HC_OK) return c;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return HC_ERR_CUDA;
  if (cur != h->device) return HC_ERR_ARG;
  float* part = h->part[h->parity];
  h->parity ^= 1;
  return enqueue_read(h, part, cur, q, T, r_out, rs, static_cast<cudaStream_t>(stream));
}

}  // namespace

HC_EXPORT int hc_read_ex(hc_read_t h, const float* R, const float* w_norm, const uint16_t* W_down,
                         const uint16_t* W_up, const float* gate, const float* pending, int T,
                         float* out, float* mean, float* lo, float* r_out, float* rs,
                         hc_stream_t stream) {
  if (W_down == nullptr || W_up == nullptr) return HC_ERR_ARG;
  return single_read(h, ReadDesc{R, pending, w_norm, gate, W_down, W_up, Q8Weights{}, out, mean, lo}, T, r_out, rs,
                     stream);
}

HC_EXPORT int hc_read_q8(hc_read_t h, const float* R, const float* w_norm, const int8_t* Wd_q,
                         const uint16_t* Wd_scale, const int8_t* Wu_q, const uint16_t* Wu_scale,
                         const float* gate, const float* pending, int T, float* out, float* mean, float* lo,
                         float* r_out, float* rs, hc_stream_t stream) {
  if (Wd_q == nullptr) return HC_ERR_ARG;
  return single_read(
      h, ReadDesc{R, pending, w_norm, gate, nullptr, nullptr, Q8Weights{Wd_q, Wd_scale, Wu_q, Wu_scale}, out, mean, lo},
      T, r_out, rs, stream);
}

HC_EXPORT int hc_read(hc_read_t h, const float* R, const float* w_norm, const uint16_t* W_down,
                      const uint16_t* W_up, const float* gate, const float* pending, int T,
                      float* out, float* mean, float* lo, hc_stream_t stream) {
  return hc_read_ex(h, R, w_norm, W_down, W_up, gate, pending, T, out, mean, lo, nullptr, nullptr,
                    stream);
}

namespace {

int find_root(std::vector<int>& parent, int x) {
  while (parent[x] != x) {
    parent[x] = parent[parent[x]];
    x = parent[x];
  }
  return x;
}

// Groups of a batch's reads that must run in order: two reads share a group
// when an output of one overlaps an input or an output of the other, directly
// or through other reads.  group[j] numbers the groups in order of first
// appearance; returns how many there are.
int group_reads(const ReadDesc* descs, int count, int n, int d, int K, int T, int* group) {
  const size_t N = (size_t)n * d;
  struct Out {
    Range r;
    int read;
  };
  std::vector<Out> outs;
  outs.reserve(3 * (size_t)count);
  for (int j = 0; j < count; ++j) {
    Range rs[3];
    output_ranges(descs[j], n, d, K, T, rs);
    for (const Range& r : rs) {
      if (r.lo != r.hi) outs.push_back({r, j});
    }
  }
  std::sort(outs.begin(), outs.end(), [](const Out& a, const Out& b) { return a.r.lo < b.r.lo; });
  std::vector<uintptr_t> hi_max(outs.size());
  for (size_t i = 0; i < outs.size(); ++i) hi_max[i] = std::max(i ? hi_max[i - 1] : 0, outs[i].r.hi);
  std::vector<int> parent(count);
  std::iota(parent.begin(), parent.end(), 0);
  for (int j = 0; j < count; ++j) {
    Range mine[kReadInputs + 3];
    Range ins[kReadInputs];
    Range own[3];
    input_ranges(descs[j], N, K, T, ins);
    output_ranges(descs[j], n, d, K, T, own);
    std::copy(ins, ins + kReadInputs, mine);
    std::copy(own, own + 3, mine + kReadInputs);
    for (const Range& m : mine) {
      if (m.lo == m.hi) continue;
      // Outputs starting below m.hi, walked down while one of them may still
      // reach above m.lo.
      const auto first_after = std::lower_bound(outs.begin(), outs.end(), m.hi,
                                                [](const Out& o, uintptr_t v) { return o.r.lo < v; });
      for (ptrdiff_t i = (first_after - outs.begin()) - 1; i >= 0 && hi_max[i] > m.lo; --i) {
        if (outs[i].r.hi > m.lo && outs[i].read != j) {
          parent[find_root(parent, outs[i].read)] = find_root(parent, j);
        }
      }
    }
  }
  std::vector<int> id(count, -1);
  int groups = 0;
  for (int j = 0; j < count; ++j) {
    const int r = find_root(parent, j);
    if (id[r] < 0) id[r] = groups++;
    group[j] = id[r];
  }
  return groups;
}

// Runs the reads of a batch on the handle's lanes, group g on lane g mod L,
// each lane in the batch's order; forks from and joins back into `caller`.
int run_lanes(hc_read_t h, const ReadDesc* descs, int count, int T, const int* group, int lanes, int device,
              cudaStream_t caller) {
  if (cudaEventRecord(h->fork, caller) != cudaSuccess) {
    cudaGetLastError();
    return HC_ERR_CUDA;
  }
  int forked = 0;
  for (; forked < lanes; ++forked) {
    // A lane's first read waits in full for whatever preceded the batch.
    forget_stream(device, h->lanes[forked].st);
    if (cudaStreamWaitEvent(h->lanes[forked].st, h->fork, 0) != cudaSuccess) break;
  }
  int status = forked == lanes ? HC_OK : HC_ERR_CUDA;
  for (int j = 0; j < count && status == HC_OK; ++j) {
    hc_read_s::Lane& ln = h->lanes[group[j] % lanes];
    float* part = ln.part[ln.parity];
    ln.parity ^= 1;
    status = enqueue_read(h, part, device, descs[j], T, nullptr, nullptr, ln.st, true);
  }
  // Every forked lane joins, also after a failure: a capture must not end
  // with work left on a lane.
  for (int l = 0; l < forked; ++l) {
    if (cudaEventRecord(h->lanes[l].done, h->lanes[l].st) != cudaSuccess ||
        cudaStreamWaitEvent(caller, h->lanes[l].done, 0) != cudaSuccess) {
      status = HC_ERR_CUDA;
    }
  }
  if (status != HC_OK) cudaGetLastError();
  // The caller's next read waits for the whole batch.
  forget_stream(device, caller);
  return status;
}

// How many lanes a batch with `groups` groups runs on (0: not on lanes).
int lanes_for(hc_read_t h, int groups) {
  const int most = std::min(h->nlanes, h->batch_lanes);
  return (groups >= 2 && most >= 2) ? std::min(groups, most) : 0;
}

// One launch of the persistent kernel over descs[0..count) (count <= kWinMaxReads).
int launch_window(hc_read_t h, const ReadDesc* descs, int count, int T, cudaStream_t st) {
  hc::WinArgs* a = new (std::nothrow) hc::WinArgs();
  if (a == nullptr) return HC_ERR_ARG;
  a->xbuf = h->xbuf;
  a->xss = h->xss;
  a->mbuf = h->mbuf;
  a->gen = h->gen;
  a->abort_flag = h->abort_flag;
  a->err = h->err;
  a->count = count;
  a->T = T;
  a->eps = h->eps;
  for (int j = 0; j < count; ++j) {
    const ReadDesc& d = descs[j];
    a->rd[j] = hc::WinRead{d.R, d.pending, d.w_norm, d.W_down, d.W_up, d.gate, d.out, d.mean, d.lo};
    a->chained[j] = (j > 0 && d.R == descs[j - 1].out) ? 1 : 0;
  }
  cudaLaunchAttribute attr[3];
  cudaLaunchConfig_t cfg = window_config(st, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, hc::hc_window_kernel<2560, 320, 1>, *a);
  delete a;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return HC_ERR_CUDA;
  }
  return HC_OK;
}

// Whether the persistent kernel covers a batch of T-token reads on this handle
// (BF16 weights only).
bool window_covers(hc_read_t h, int T, bool q8) { return !q8 && h->window && T <= 4; }

// Argument checks of a whole batch (see hc_read_batch).
int check_batch(hc_read_t h, const ReadDesc* descs, int count, int T) {
  const size_t N = (size_t)h->n * h->d;
  for (int j = 0; j < count; ++j) {
    const ReadDesc& d = descs[j];
    const int c = check_read(d, nullptr, nullptr);
    if (c != HC_OK) return c;
    if (d.is_q8() != descs[0].is_q8()) return HC_ERR_ARG;
    const Range p_in = range_of(d.pending, T * N * 4);
    if (overlaps(p_in, range_of(d.out, T * N * 4))) return HC_ERR_ARG;
    // Inputs may not depend on earlier reads of the batch, except R taking
    // the previous read's out exactly (a chained read, whose R is never
    // loaded by the persistent kernel: it is the previous read's output
    // tile, still on chip).
    const bool chained = j > 0 && d.R == descs[j - 1].out;
    const Range r_in = chained ? range_of(nullptr, 0) : range_of(d.R, T * N * 4);
    for (int i = 0; i < j; ++i) {
      Range outs[3];
      output_ranges(descs[i], h->n, h->d, h->K, T, outs);
      for (const Range& o : outs) {
        if (overlaps(r_in, o) || overlaps(p_in, o)) return HC_ERR_ARG;
      }
    }
  }
  return HC_OK;
}

// How a checked batch runs: 0 read by read, 1 the persistent kernel, L >= 2 lanes.
int plan_batch(hc_read_t h, const ReadDesc* descs, int count, int T, int* group) {
  if (count >= 2 && lanes_for(h, count) >= 2) {
    const int lanes = lanes_for(h, group_reads(descs, count, h->n, h->d, h->K, T, group));
    if (lanes >= 2) return lanes;
  }
  return window_covers(h, T, descs[0].is_q8()) ? 1 : 0;
}

int run_batch(hc_read_t h, const std::vector<ReadDesc>& descs, int T, hc_stream_t stream) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return HC_ERR_CUDA;
  if (cur != h->device) return HC_ERR_ARG;
  const int count = (int)descs.size();
  const int c = check_batch(h, descs.data(), count, T);
  if (c != HC_OK) return c;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int> group(count);
  const int plan = plan_batch(h, descs.data(), count, T, group.data());
  if (plan >= 2) return run_lanes(h, descs.data(), count, T, group.data(), plan, cur, st);
  if (plan == 0) {
    for (const ReadDesc& d : descs) {
      float* part = h->part[h->parity];
      h->parity ^= 1;
      const int r = enqueue_read(h, part, cur, d, T, nullptr, nullptr, st);
      if (r != HC_OK) return r;
    }
    return HC_OK;
  }
  for (int j0 = 0; j0 < count; j0 += hc::kWinMaxReads) {
    const int r = launch_window(h, descs.data() + j0, std::min(count - j0, hc::kWinMaxReads), T, st);
    if (r != HC_OK) return r;
  }
  // A later hc_read that consumes the last read's outputs must wait for them.
  const size_t N = (size_t)h->n * h->d;
  const ReadDesc& last = descs[count - 1];
  Range ins[kReadInputs];
  input_ranges(last, N, h->K, T, ins);
  const Range outs[5] = {range_of(last.out, T * N * 4), range_of(last.mean, (size_t)T * h->d * 4),
                         range_of(last.lo, (size_t)T * h->K * 4), range_of(nullptr, 0), range_of(nullptr, 0)};
  record_and_check(cur, stream, ins, outs);
  return HC_OK;
}

template <class Desc>
std::vector<ReadDesc> read_descs(const Desc* descs, int count) {
  std::vector<ReadDesc> v;
  v.reserve(count);
  for (int j = 0; j < count; ++j) v.push_back(from_desc(descs[j]));
  return v;
}

}  // namespace

HC_EXPORT int hc_read_batch_persistent(hc_read_t h, int T) {
  if (h == nullptr || T < 1 || T > h->T_max) return HC_ERR_ARG;
  return window_covers(h, T, false) ? 1 : 0;
}

HC_EXPORT int hc_read_batch(hc_read_t h, const hc_read_desc* descs, int count, int T, hc_stream_t stream) {
  if (h == nullptr || descs == nullptr || count < 1) return HC_ERR_ARG;
  if (T < 1 || T > h->T_max) return HC_ERR_ARG;
  for (int j = 0; j < count; ++j) {
    if (descs[j].W_down == nullptr || descs[j].W_up == nullptr) return HC_ERR_ARG;
  }
  return run_batch(h, read_descs(descs, count), T, stream);
}

HC_EXPORT int hc_read_batch_q8(hc_read_t h, const hc_read_q8_desc* descs, int count, int T, hc_stream_t stream) {
  if (h == nullptr || descs == nullptr || count < 1) return HC_ERR_ARG;
  if (T < 1 || T > h->T_max) return HC_ERR_ARG;
  for (int j = 0; j < count; ++j) {
    if (descs[j].Wd_q == nullptr) return HC_ERR_ARG;
  }
  return run_batch(h, read_descs(descs, count), T, stream);
}

HC_EXPORT int hc_read_batch_plan(hc_read_t h, const hc_read_desc* descs, int count, int T) {
  if (h == nullptr || descs == nullptr || count < 1 || T < 1 || T > h->T_max) return HC_ERR_ARG;
  std::vector<int> group(count);
  return plan_batch(h, read_descs(descs, count).data(), count, T, group.data());
}

HC_EXPORT int hc_read_batch_q8_plan(hc_read_t h, const hc_read_q8_desc* descs, int count, int T) {
  if (h == nullptr || descs == nullptr || count < 1 || T < 1 || T > h->T_max) return HC_ERR_ARG;
  std::vector<int> group(count);
  const std::vector<ReadDesc> v = read_descs(descs, count);
  for (const ReadDesc& d : v) {
    if (!d.is_q8()) return HC_ERR_ARG;
  }
  return plan_batch(h, v.data(), count, T, group.data());
}

HC_EXPORT int hc_read_set_batch_lanes(hc_read_t h, int lanes) {
  if (h == nullptr || lanes < 0) return HC_ERR_ARG;
  const int prev = h->batch_lanes;
  h->batch_lanes = std::min(lanes, kBatchLanes);
  return prev;
}

HC_EXPORT int hc_read_batch_groups(const hc_read_desc* descs, int count, int n, int d, int K, int T,
                                   int* group) {
  if (descs == nullptr || group == nullptr || count < 1 || T < 1 || n < 1 || d < 1 || K < 1) return HC_ERR_ARG;
  return group_reads(read_descs(descs, count).data(), count, n, d, K, T, group);
}

HC_EXPORT int hc_read_batch_q8_groups(const hc_read_q8_desc* descs, int count, int n, int d, int K, int T,
                                      int* group) {
  if (descs == nullptr || group == nullptr || count < 1 || T < 1 || n < 1 || d < 1 || K < 1) return HC_ERR_ARG;
  // Scale rows are K/32 or n*d/32 binary16 values: both widths multiples of 32.
  if ((n * d) % 32 != 0 || K % 32 != 0) return HC_ERR_ARG;
  return group_reads(read_descs(descs, count).data(), count, n, d, K, T, group);
}

HC_EXPORT int hc_read_check(hc_read_t h) {
  if (h == nullptr) return HC_ERR_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return HC_ERR_CUDA;
  if (cudaSetDevice(h->device) != cudaSuccess) return HC_ERR_CUDA;
  unsigned word = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost);
  cudaSetDevice(prev);
  if (e != cudaSuccess) return HC_ERR_CUDA;
  return word == 0 ? HC_OK : HC_ERR_TIMEOUT;
}

HC_EXPORT int64_t hc_read_error_word(hc_read_t h) {
  if (h == nullptr) return HC_ERR_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return HC_ERR_CUDA;
  if (cudaSetDevice(h->device) != cudaSuccess) return HC_ERR_CUDA;
  unsigned word = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost);
  cudaSetDevice(prev);
  if (e != cudaSuccess) return HC_ERR_CUDA;
  return static_cast<int64_t>(word);
}

HC_EXPORT int hc_read_reset(hc_read_t h, hc_stream_t stream) {
  if (h == nullptr) return HC_ERR_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return HC_ERR_CUDA;
  if (cur != h->device) return HC_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(h->err, 0, sizeof(unsigned), st);
  // The persistent kernel's exchange words, epoch bases and abort word start over.
  if (e == cudaSuccess && h->xbuf != nullptr) e = cudaMemsetAsync(h->xbuf, 0, h->window_bytes, st);
  return e == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

HC_EXPORT void hc_read_destroy(hc_read_t h) {
  if (h == nullptr) return;
  int prev = -1;
  if (cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(h->device) == cudaSuccess) {
    cudaDeviceSynchronize();
    destroy_lanes(h);
    cudaFree(h->scratch);
    cudaSetDevice(prev);
  }
  delete h->map_cache;
  delete h->down_tiles;
  delete h->up_tiles;
  delete h;
}

HC_EXPORT int hc_read_set_wait_limit(hc_read_t h, uint64_t ns) {
  if (h == nullptr) return HC_ERR_ARG;
  h->wait_ns = ns;
  return HC_OK;
}

HC_EXPORT int hc_read_set_overlap(hc_read_t h, int enabled) {
  if (h == nullptr || enabled < 0 || enabled > 1) return HC_ERR_ARG;
  const int prev = h->overlap ? 1 : 0;
  h->overlap = enabled != 0;
  return prev;
}

HC_EXPORT int64_t hc_read_down_tiles_bytes(hc_read_t h) {
  if (h == nullptr) return -1;
  return static_cast<int64_t>(down_tiles_bytes(h->d));
}

HC_EXPORT int64_t hc_read_up_tiles_bytes(hc_read_t h) {
  if (h == nullptr) return -1;
  return h->d == 2560 ? static_cast<int64_t>(kSwTilesBytes) : 0;
}

namespace {

// Writes `tiles` from W (on `stream`, waited for) and registers W -> tiles in *map.
int register_tiles(hc_read_t h, std::unordered_map<const void*, const void*>*& map, const void* W, size_t w_bytes,
                   void* tiles, size_t tile_bytes, hc_stream_t stream, bool up) {
  if (h == nullptr || W == nullptr || tiles == nullptr) return HC_ERR_ARG;
  if (!aligned16(W) || !aligned16(tiles)) return HC_ERR_ALIGN;
  if (tile_bytes == 0) return HC_ERR_SHAPE;
  if (overlaps(range_of(W, w_bytes), range_of(tiles, tile_bytes))) return HC_ERR_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return HC_ERR_CUDA;
  if (cur != h->device) return HC_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The copy completes before this returns: a read enqueued later may load
  // its weights before it waits for the kernels ahead of it.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return HC_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return HC_ERR_ARG;
  cudaError_t e;
  if (up) {
    using Wg = hc::WGeo<2560, 320>;
    hc::hc_pack_up_sw_kernel<2560, 320><<<Wg::UP_CTAS, 256, 0, st>>>(static_cast<const uint16_t*>(W),
                                                                     static_cast<uint16_t*>(tiles));
    e = cudaGetLastError();
  } else {
    e = h->d == 2560 ? launch_pack_down_tiles<2560, 320>(W, tiles, st) : launch_pack_down_tiles<4096, 512>(W, tiles, st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return HC_ERR_CUDA;
  }
  try {
    if (map == nullptr) map = new std::unordered_map<const void*, const void*>();
    (*map)[W] = tiles;
  } catch (...) {
    return HC_ERR_CUDA;
  }
  return HC_OK;
}

int forget_tiles(hc_read_t h, std::unordered_map<const void*, const void*>* map, const void* W) {
  if (h == nullptr) return HC_ERR_ARG;
  if (map != nullptr) {
    if (W == nullptr) {
      map->clear();
    } else {
      map->erase(W);
    }
  }
  return HC_OK;
}

}  // namespace

HC_EXPORT int hc_read_register_down_tiles(hc_read_t h, const void* W_down, void* tiles, hc_stream_t stream) {
  if (h == nullptr) return HC_ERR_ARG;
  return register_tiles(h, h->down_tiles, W_down, (size_t)h->K * h->n * h->d * 2, tiles, down_tiles_bytes(h->d),
                        stream, false);
}

HC_EXPORT int hc_read_forget_down_tiles(hc_read_t h, const void* W_down) {
  return forget_tiles(h, h == nullptr ? nullptr : h->down_tiles, W_down);
}

HC_EXPORT int hc_read_register_up_tiles(hc_read_t h, const void* W_up, void* tiles, hc_stream_t stream) {
  if (h == nullptr) return HC_ERR_ARG;
  return register_tiles(h, h->up_tiles, W_up, (size_t)h->K * h->n * h->d * 2, tiles,
                        static_cast<size_t>(hc_read_up_tiles_bytes(h)), stream, true);
}

HC_EXPORT int hc_read_forget_up_tiles(hc_read_t h, const void* W_up) {
  return forget_tiles(h, h == nullptr ? nullptr : h->up_tiles, W_up);
}

HC_EXPORT int64_t hc_read_scratch_bytes(hc_read_t h) {
  return h == nullptr ? -1 : static_cast<int64_t>(h->scratch_bytes);
}

HC_EXPORT const char* hc_status_str(int status) {
  switch (status) {
    case HC_OK: return "ok";
    case HC_ERR_ARG: return "invalid argument";
    case HC_ERR_ALIGN: return "pointer not 16-byte aligned";
    case HC_ERR_SHAPE: return "geometry not supported";
    case HC_ERR_CUDA: return "CUDA runtime error";
    case HC_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
    case HC_ERR_TOO_LARGE: return "T exceeds the no-allocation entry point's maximum";
    default: return "unknown status";
  }
}

HC_EXPORT int hc_graph_begin(hc_stream_t stream) {
  cudaError_t e = cudaStreamBeginCapture(static_cast<cudaStream_t>(stream),
                                         cudaStreamCaptureModeThreadLocal);
  return e == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

HC_EXPORT int hc_graph_end(hc_stream_t stream, hc_graph_t* exec) {
  if (exec == nullptr) return HC_ERR_ARG;
  *exec = nullptr;
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(static_cast<cudaStream_t>(stream), &g);
  if (e != cudaSuccess) return HC_ERR_CUDA;
  cudaGraphExec_t ge = nullptr;
  e = cudaGraphInstantiate(&ge, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return HC_ERR_CUDA;
  *exec = ge;
  return HC_OK;
}

HC_EXPORT int hc_graph_launch(hc_graph_t exec, hc_stream_t stream) {
  if (exec == nullptr) return HC_ERR_ARG;
  cudaError_t e = cudaGraphLaunch(static_cast<cudaGraphExec_t>(exec), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

HC_EXPORT void hc_graph_destroy(hc_graph_t exec) {
  if (exec != nullptr) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(exec));
}

// ---------------------------------------------------------------------------
// No-allocation entry point.  Its scratch is one file-scope device array
// (one slot of rs-scaled per-stream partials and the error word), sized for
// the largest supported geometry (K = 512) at T <= HC_NOALLOC_MAX_T.  Host
// code must not hand the array's name to a kernel (on the host it only stands
// for the symbol); the device address is looked up once per device with
// cudaGetSymbolAddress.
namespace {

constexpr size_t kNoallocPartBytes = (size_t)4 * HC_NOALLOC_MAX_T * 512 * sizeof(float);
constexpr size_t kNoallocTailBytes = 256;  // the error word
static_assert(kNoallocPartBytes + kNoallocTailBytes == HC_NOALLOC_SCRATCH_BYTES,
              "scratch size in the header and here disagree");

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_scratch_addr[kMaxDevices];

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[HC_NOALLOC_SCRATCH_BYTES];

HC_EXPORT int hc_read_noalloc(int n, int d, int K, float eps, const float* R, const float* w_norm,
                              const uint16_t* W_down, const uint16_t* W_up, const float* gate,
                              const float* pending, int T, float* out, float* mean, float* lo,
                              hc_stream_t stream) {
  if (!geometry_supported(n, d, K)) return HC_ERR_SHAPE;
  if (!(eps >= 0.0f) || T < 1) return HC_ERR_ARG;
  if (T > HC_NOALLOC_MAX_T) return HC_ERR_TOO_LARGE;
  if (!R || !w_norm || !W_down || !W_up || !gate || !out || !mean || !lo) return HC_ERR_ARG;
  const void* ptrs[] = {R, w_norm, W_down, W_up, gate, pending, out, mean, lo};
  for (const void* p : ptrs) {
    if (p != nullptr && !aligned16(p)) return HC_ERR_ALIGN;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HC_ERR_CUDA;

  // Set-up, once per device, with that device current: the scratch array's
  // device address and the kernels' shared-memory attributes.
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_scratch_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return HC_ERR_CUDA;
      }
      if (configure_geometry<2560, 320>() != cudaSuccess ||
          configure_geometry<4096, 512>() != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
      }
      g_noalloc_scratch_addr[dev] = addr;
    }
    base = g_noalloc_scratch_addr[dev];
  }

  char* b = static_cast<char*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The error word collects the calls' bounded-wait failures until
  // hc_read_noalloc_check reads and clears it (it starts at zero: the array
  // is zero-initialised when the library is loaded).  The partial-sum slot
  // needs no clearing: every call writes the part it reads.
  unsigned* err = reinterpret_cast<unsigned*>(b + kNoallocPartBytes);
  // Keep this stream's record of the last read current, so that a later read
  // that consumes these outputs waits for them.  (This path has one scratch
  // slot and always waits for the previous kernel before it computes.)
  const size_t N = (size_t)n * d;
  Range ins[kReadInputs];
  input_ranges(ReadDesc{R, pending, w_norm, gate, W_down, W_up, Q8Weights{}, out, mean, lo}, N, K, T, ins);
  const Range outs[5] = {range_of(out, T * N * 4), range_of(mean, (size_t)T * d * 4),
                         range_of(lo, (size_t)T * K * 4), range_of(nullptr, 0),
                         range_of(nullptr, 0)};
  record_and_check(dev, stream, ins, outs);

  DownArgs da{};
  da.R = R;
  da.P = pending;
  da.w_norm = w_norm;
  da.W_down = W_down;
  da.part = reinterpret_cast<float*>(b);
  da.err = err;
  da.rs_out = nullptr;
  da.T = T;
  da.T_max = HC_NOALLOC_MAX_T;
  da.independent = 0;
  da.eps = eps;

  UpArgs ua{};
  ua.R = R;
  ua.P = pending;
  ua.gate = gate;
  ua.W_up = W_up;
  ua.part = reinterpret_cast<float*>(b);
  ua.out = out;
  ua.mean = mean;
  ua.lo = lo;
  ua.r_out = nullptr;
  ua.err = err;
  ua.T = T;
  ua.T_max = HC_NOALLOC_MAX_T;
  ua.independent = 0;

  // The same kernels as a handle's read; the W_down tensor map is encoded
  // per call (a host structure, no allocation).
  CUtensorMap w_down;
  const bool mapped = takes_umma(d, T) && encode_bf16_tiles(&w_down, W_down, K, (uint64_t)n * d, 64);
  cudaError_t e = (d == 2560) ? launch_geometry<2560, 320>(T, da, ua, st, mapped ? &w_down : nullptr)
                              : launch_geometry<4096, 512>(T, da, ua, st, nullptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return HC_ERR_CUDA;
  }
  return HC_OK;
}

HC_EXPORT int hc_read_noalloc_check(void) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HC_ERR_CUDA;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    base = g_noalloc_scratch_addr[dev];
  }
  if (base == nullptr) return HC_OK;  // no call has run on this device
  unsigned* err = reinterpret_cast<unsigned*>(static_cast<char*>(base) + kNoallocPartBytes);
  unsigned word = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0u) e = cudaMemset(err, 0, sizeof word);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return HC_ERR_CUDA;
  }
  return word == 0u ? HC_OK : HC_ERR_TIMEOUT;
}
