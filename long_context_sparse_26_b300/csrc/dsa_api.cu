// libdsa: C ABI for DSA sparse attention with IndexShare on B300 (sm_103a).
// Host side: argument validation, workspace layout, TMA descriptors and the
// launch sequence of each entry point.  Every entry point only enqueues work on
// the caller's stream; nothing here allocates device memory or synchronizes.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "dsa.h"
#include "common.cuh"
#include "indexer.cuh"
#include "sparse_mla.cuh"
#include "sparse_mla_tc.cuh"
#include "topk.cuh"

namespace {

using dsa::attn::kMaxLayers;

// The indexer counts the top-k's first digit: both sides must agree on it.
static_assert(dsa::indexer::kHistBins == dsa::topk::kBins0 && dsa::indexer::kHistShift == dsa::topk::kShift0 &&
                  dsa::indexer::kHistRowStride == dsa::topk::kGhistStride,
              "indexer histogram and top-k digit 0 disagree");

constexpr int kIdxHeads = 64, kIdxDim = 128, kHeads = 64, kLora = 512, kRope = 64, kMaxTopk = 2048;
constexpr int kMaxDevices = 64;
constexpr long long kMaxRowsY = 65535;  // grid.y limit for (chunk, row) launches

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches `kernel` as a programmatic dependent of the kernel before it on
// the stream: its blocks may be scheduled while that kernel finishes, and
// every one of them executes griddepcontrol.wait before reading what that
// kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args) {
  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}
// The same, in thread-block clusters of cx consecutive blocks.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                     unsigned cx, Args &&...args) {
  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cx;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceState {
  int sms = 0;
  bool attrs_set = false;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// The indexer's instantiations: query-group size x key format (bf16; FP8
// with contiguous or paged scales; paged bf16 keys are a runtime path of the
// bf16 kernels), and for one query per group whether the epilogue counts the
// top-k's histograms.  Each needs its shared-memory attribute set once per
// device; a launch picks one.
template <int QG, bool F8, bool PGS, bool HIST>
struct IndexerInst {
  using C = dsa::indexer::Cfg<QG, F8, HIST>;
  static bool set_attr() {
    return cudaFuncSetAttribute(dsa::indexer::indexer_scores_kernel<QG, F8, PGS, HIST>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) == cudaSuccess;
  }
  static void launch(unsigned grid, const CUtensorMap &tk, const CUtensorMap &tq, const dsa::indexer::Params &p,
                     cudaStream_t stream) {
    dsa::indexer::indexer_scores_kernel<QG, F8, PGS, HIST><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tk, tq, p);
  }
};

template <bool F8, bool PGS>
struct IndexerFamily {
  static bool set_attrs() {
    return IndexerInst<1, F8, PGS, false>::set_attr() && IndexerInst<1, F8, PGS, true>::set_attr() &&
           IndexerInst<2, F8, PGS, false>::set_attr() && IndexerInst<4, F8, PGS, false>::set_attr();
  }
  // hist: QG == 1 only
  static void launch(int QG, bool hist, unsigned grid, const CUtensorMap &tk, const CUtensorMap &tq,
                     const dsa::indexer::Params &p, cudaStream_t stream) {
    if (QG == 1 && hist)
      IndexerInst<1, F8, PGS, true>::launch(grid, tk, tq, p, stream);
    else if (QG == 1)
      IndexerInst<1, F8, PGS, false>::launch(grid, tk, tq, p, stream);
    else if (QG == 2)
      IndexerInst<2, F8, PGS, false>::launch(grid, tk, tq, p, stream);
    else
      IndexerInst<4, F8, PGS, false>::launch(grid, tk, tq, p, stream);
  }
};

bool set_indexer_attrs() {
  return IndexerFamily<false, false>::set_attrs() && IndexerFamily<true, false>::set_attrs() &&
         IndexerFamily<true, true>::set_attrs();
}

// Per-device facts and one-time kernel attributes.  Returns false on a CUDA error.
bool device_state(DeviceState **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &s = g_dev[dev];
  if (!s.attrs_set) {
    if (cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    bool ok = true;
    ok &= set_indexer_attrs();
    ok &= cudaFuncSetAttribute(dsa::mla::sparse_mla_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dsa::mla::kSmemBytes) == cudaSuccess;
    ok &= cudaFuncSetAttribute(dsa::mla::sparse_mla_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dsa::mla::kSmemBytes) == cudaSuccess;
    ok &= cudaFuncSetAttribute(dsa::topk::topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dsa::topk::kSelectSmem) == cudaSuccess;
    ok &= cudaFuncSetAttribute(dsa::topk::topk_chunk_scan_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dsa::topk::kScanSelectSmem) == cudaSuccess;
    if (!ok) return false;
    if (g_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.attrs_set = true;
  }
  *out = &s;
  return true;
}

// 2D bf16 tensor map over a row-major [rows, 128] matrix, 128-byte swizzle,
// box = 64 columns x box_rows rows.
bool make_tmap_128(CUtensorMap *map, const void *ptr, unsigned long long rows, unsigned box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kIdxDim * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D tensor map over a row-major [rows, 128] matrix of E4M3 bytes, 128-byte
// swizzle, box = the whole 128-byte row x box_rows rows.
bool make_tmap_e4m3_128(CUtensorMap *map, const void *ptr, unsigned long long rows, unsigned box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kIdxDim)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kIdxDim), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D bf16 tensor map over a row-major [rows, 576] matrix (the query heads of
// an attention call), 128-byte swizzle, box = 64 columns x box_rows rows.
bool make_tmap_576(CUtensorMap *map, const void *ptr, unsigned long long rows, unsigned box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kLora + kRope), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>((kLora + kRope) * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

dsa_status_t check_config(const dsa_config_t *c) {
  if (c == nullptr) return DSA_ERR_INVALID_ARG;
  if (c->n_idx_heads != kIdxHeads || c->idx_dim != kIdxDim || c->kv_lora_rank != kLora || c->rope_dim != kRope ||
      c->n_heads != kHeads)
    return DSA_ERR_UNSUPPORTED;
  if (c->topk < 1 || c->topk > kMaxTopk || c->topk_freq < 1) return DSA_ERR_UNSUPPORTED;
  if (!(c->sm_scale > 0.0f) || !std::isfinite(c->sm_scale)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// A block-table description for B sequences of context T.
dsa_status_t check_pages(const dsa_pages_t *pg, int B, int T) {
  if (pg == nullptr || pg->block_table == nullptr) return DSA_ERR_INVALID_ARG;
  if (pg->page_size < 64 || pg->page_size % 64 != 0) return DSA_ERR_UNSUPPORTED;
  if (pg->num_pages <= 0 || pg->max_pages <= 0) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(pg->max_pages) * pg->page_size < T) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(pg->num_pages) * pg->page_size >= (1LL << 31)) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * pg->max_pages >= (1LL << 31)) return DSA_ERR_INVALID_ARG;
  if (!aligned16(pg->block_table)) return DSA_ERR_ALIGNMENT;
  return DSA_OK;
}

// No query rows (B or Q zero, none negative): a valid call with nothing to do.
inline bool empty_call(int B, int Q, int T) { return (B == 0 || Q == 0) && B >= 0 && Q >= 0 && T >= 0; }

dsa_status_t check_sizes(int B, int Q, int T) {
  if (B <= 0 || Q <= 0 || T <= 0) return DSA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * Q;
  if (rows > kMaxRowsY) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * T >= (1LL << 31)) return DSA_ERR_INVALID_ARG;    // TMA row coordinate
  if (rows * kIdxHeads >= (1LL << 31)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// ---------------------------------------------------------------------------
// Launch shapes and workspace layout (one definition for sizing and launching)
// ---------------------------------------------------------------------------
struct TopkShape {
  int nchunk = 1, chunk = 0;
};

TopkShape topk_shape(int rows, int T, int sms) {
  TopkShape s;
  if (rows >= 2 * sms) {
    s.nchunk = 1;
    s.chunk = T;
    return s;
  }
  // (chunk, row) blocks: at most one wave of the scan (two blocks per SM)
  const int target = 2 * sms;
  int n = target / rows;
  const int max_chunks = (T + 4095) / 4096;  // chunks of at least 4096 scores
  n = n < max_chunks ? n : max_chunks;
  n = n < dsa::topk::kThreads ? n : dsa::topk::kThreads;  // the select block prefix-sums one count per thread
  n = n < 1 ? 1 : n;
  s.chunk = static_cast<int>(align_up((T + n - 1) / n, 1024));
  s.nchunk = (T + s.chunk - 1) / s.chunk;
  return s;
}

struct AttnShape {
  int nsplit = 1, bps = 1;
  // one split per (layer, row) unit, except that the units from tail_base
  // on (the last, partial wave) take tail_nsplit splits of tail_bps windows
  long long tail_base = 0;
  int tail_nsplit = 0, tail_bps = 0;
  // (layer, row) units whose splits leave fp32 partials, and splits each
  long long partial_units(long long rowsL) const { return tail_nsplit > 0 ? rowsL - tail_base : (nsplit > 1 ? rowsL : 0); }
  int partial_splits() const { return tail_nsplit > 0 ? tail_nsplit : nsplit; }
};

constexpr int kSplitCost = 7;  // windows' worth of a split's partial (written, then read by the combine)

// Splits of each row's index slots over blocks (one block per SM at a time):
// the fewest waves x windows per block, where a split also costs its fp32
// partial.  With one split per unit, the units of a last, partial wave are
// split further when that shortens it, so that wave runs as wide as the GPU
// (wave quantisation: 512 units on 148 SMs leave a fourth wave 46% full).
AttnShape attn_shape(long long rowsL, int K, int sms) {
  AttnShape best;
  const int nblocks = (K + dsa::mla::kKeys - 1) / dsa::mla::kKeys;
  long long best_cost = -1;
  for (int ns = 1; ns <= 16 && ns <= nblocks; ++ns) {
    const int bps = (nblocks + ns - 1) / ns;
    const int nsr = (nblocks + bps - 1) / bps;
    const long long waves = (rowsL * nsr + sms - 1) / sms;
    const long long cost = waves * (bps + (nsr > 1 ? kSplitCost : 0));
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best.nsplit = nsr;
      best.bps = bps;
    }
  }
  if (best.nsplit == 1) {
    const long long full = rowsL / sms * sms;
    const long long rem = rowsL - full;
    if (full > 0 && rem > 0) {
      long long s = sms / rem;
      s = s < 16 ? s : 16;
      s = s < nblocks ? s : nblocks;
      const int bps = static_cast<int>((nblocks + s - 1) / s);
      if (s >= 2 && bps + kSplitCost < nblocks) {
        best.tail_base = full;
        best.tail_bps = bps;
        best.tail_nsplit = (nblocks + bps - 1) / bps;
      }
    }
  }
  return best;
}

struct Layout {
  size_t scores = 0, ghist = 0, done = 0, counts = 0, cand = 0, idx = 0, part_o = 0, part_ml = 0, total = 0;
  TopkShape ts;
};

size_t attn_partial_bytes(long long rowsL, int K, int sms, size_t *ml_bytes) {
  const AttnShape a = attn_shape(rowsL, K, sms);
  const size_t tiles = static_cast<size_t>(a.partial_units(rowsL)) * a.partial_splits();
  *ml_bytes = tiles * kHeads * 2 * sizeof(float);
  return tiles * kHeads * kLora * sizeof(float);
}

Layout layout(int B, int Q, int T, int n_layers, int K, int sms) {
  Layout L;
  const long long rows = static_cast<long long>(B) * Q;
  L.ts = topk_shape(static_cast<int>(rows), T, sms);
  size_t off = 0;
  L.scores = off;  // offset 0: a group call leaves its scores at the start of the workspace (dsa.h)
  off = align_up(off + static_cast<size_t>(rows) * T * sizeof(float), 256);
  // chunked top-k: digit-0 histograms and per-row chunk tickets (zeroed by
  // one memset, so they are adjacent), per-chunk candidate counts, then room
  // for T candidates per row
  L.ghist = off;
  if (L.ts.nchunk > 1) off += static_cast<size_t>(rows) * dsa::topk::kGhistStride * 4;
  L.done = off;
  if (L.ts.nchunk > 1) off = align_up(off + static_cast<size_t>(rows) * 4, 256);
  L.counts = off;
  if (L.ts.nchunk > 1) off = align_up(off + static_cast<size_t>(rows) * L.ts.nchunk * 4, 256);
  L.cand = off;
  if (L.ts.nchunk > 1) off = align_up(off + static_cast<size_t>(rows) * T * 8, 256);
  L.idx = off;
  off = align_up(off + static_cast<size_t>(rows) * K * sizeof(int32_t), 256);
  // partials: the largest need over a single-layer call and an n_layers call
  size_t ml1 = 0, mln = 0;
  const size_t po1 = attn_partial_bytes(rows, K, sms, &ml1);
  const size_t pon = attn_partial_bytes(rows * n_layers, K, sms, &mln);
  L.part_o = off;
  off = align_up(off + (po1 > pon ? po1 : pon), 256);
  L.part_ml = off;
  off = align_up(off + (ml1 > mln ? ml1 : mln), 256);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// Launch helpers (arguments already validated)
// ---------------------------------------------------------------------------
// ghist: when non-null (and Q == 1), the indexer also counts the top-k's
// digit-0 histograms into it (which must be zeroed before).
// FP8 caches: q_idx / k_idx point at E4M3 bytes and the two scale arrays
// are given (both null for bf16).
dsa_status_t launch_indexer(const DeviceState &dev, const void *q_idx, const float *w, const void *k_idx,
                            const int32_t *q_pos, int B, int Q, int T, float *scores, cudaStream_t stream,
                            uint32_t *ghist = nullptr, const dsa_pages_t *pages = nullptr,
                            const float *q_scale = nullptr, const float *k_scale = nullptr) {
  const bool f8 = k_scale != nullptr;
  const int QG = Q == 1 ? 1 : (Q == 2 ? 2 : 4);
  CUtensorMap tk, tq;
  auto tmap = f8 ? make_tmap_e4m3_128 : make_tmap_128;
  if (pages != nullptr) {
    if (!tmap(&tk, k_idx, static_cast<unsigned long long>(pages->num_pages) * pages->page_size, 64))
      return DSA_ERR_CUDA;
  } else if (!tmap(&tk, k_idx, static_cast<unsigned long long>(B) * T, dsa::indexer::kTileKeys)) {
    return DSA_ERR_CUDA;
  }
  if (!tmap(&tq, q_idx, static_cast<unsigned long long>(B) * Q * kIdxHeads, QG * kIdxHeads)) return DSA_ERR_CUDA;
  dsa::indexer::Params p;
  p.w = w;
  p.q_pos = q_pos;
  p.scores = scores;
  p.B = B;
  p.Q = Q;
  p.T = T;
  p.ngroups = (Q + QG - 1) / QG;
  // keys per unit of work: 256 for FP8 keys with one query per group, else 128
  const int unit_keys = (f8 && QG == 1) ? dsa::indexer::Cfg<1, true>::kUnitKeys : dsa::indexer::kTileKeys;
  p.ntiles = (T + unit_keys - 1) / unit_keys;
  p.units = static_cast<long long>(B) * p.ngroups * p.ntiles;
  p.stream_keys = p.ngroups == 1 ? 1 : 0;
  p.block_table = pages ? pages->block_table : nullptr;
  p.page_size = pages ? pages->page_size : 0;
  p.max_pages = pages ? pages->max_pages : 0;
  p.num_pages = pages ? pages->num_pages : 0;
  p.k_scale = k_scale;
  p.q_scale = q_scale;
  p.ghist = QG == 1 ? ghist : nullptr;
  const long long grid = p.units < dev.sms ? p.units : dev.sms;
  const unsigned g = static_cast<unsigned>(grid);
  const bool hist = p.ghist != nullptr;
  if (!f8)
    IndexerFamily<false, false>::launch(QG, hist, g, tk, tq, p, stream);
  else if (pages == nullptr)
    IndexerFamily<true, false>::launch(QG, hist, g, tk, tq, p, stream);
  else  // paged FP8 keys: the scales are a paged pool too
    IndexerFamily<true, true>::launch(QG, hist, g, tk, tq, p, stream);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Clears the chunked top-k's histograms and counters (before the indexer when
// it counts the digit-0 histogram itself).
dsa_status_t clear_topk_state(const Layout &L, uint8_t *ws, cudaStream_t stream) {
  if (L.ts.nchunk <= 1) return DSA_OK;
  return cudaMemsetAsync(ws + L.ghist, 0, L.counts - L.ghist, stream) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// hist_done: the digit-0 histograms were already counted (by the indexer).
dsa_status_t launch_topk(const Layout &L, uint8_t *ws, const float *scores, const int32_t *q_pos, int rows, int T,
                         int K, int32_t *idx, cudaStream_t stream, bool hist_done = false) {
  using namespace dsa::topk;
  if (L.ts.nchunk == 1) {
    topk_row_kernel<<<rows, kThreads, kSelectSmem, stream>>>(scores, q_pos, T, K, idx);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  ChunkParams p;
  p.scores = scores;
  p.q_pos = q_pos;
  p.T = T;
  p.K = K;
  p.rows = rows;
  p.chunk = L.ts.chunk;
  p.nchunk = L.ts.nchunk;
  p.ghist = reinterpret_cast<uint32_t *>(ws + L.ghist);
  p.done = reinterpret_cast<uint32_t *>(ws + L.done);
  p.counts = reinterpret_cast<uint32_t *>(ws + L.counts);
  p.cand = reinterpret_cast<uint64_t *>(ws + L.cand);
  p.idx = idx;
  const dim3 grid(p.nchunk, rows);
  if (!hist_done) {
    if (clear_topk_state(L, ws, stream) != DSA_OK) return DSA_ERR_CUDA;
    topk_chunk_hist_kernel<<<grid, kThreads, 0, stream>>>(p);
  }
  if (launch_dependent(topk_chunk_scan_select_kernel, grid, dim3(kThreads), kScanSelectSmem, stream, p) != cudaSuccess)
    return DSA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Enqueues the tensor-core attention kernel (and the split combine) for
// filled-in Params over B sequences; encodes each layer's tensor maps.
// How many clusters of cx attention blocks the current device runs at once
// (cached per device, row format and cluster size; 0 when it cannot).
int attention_clusters(bool fp8, int cx) {
  static int cache[kMaxDevices][2][9];
  static bool init = false;
  int dev = 0;
  if (cx < 2 || cx > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!init) {
    for (auto &d : cache)
      for (auto &f : d)
        for (int &c : f) c = -1;
    init = true;
  }
  int &c = cache[dev][fp8 ? 1 : 0][cx];
  if (c < 0) {
    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof(lc));
    lc.gridDim = dim3(static_cast<unsigned>(cx) * 64);
    lc.blockDim = dim3(fp8 ? dsa::mla::Roles<true>::kThreads : dsa::mla::Roles<false>::kThreads);
    lc.dynamicSmemBytes = dsa::mla::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cx);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    const cudaError_t e =
        fp8 ? cudaOccupancyMaxActiveClusters(&n, dsa::mla::sparse_mla_tc_kernel<true>, &lc)
            : cudaOccupancyMaxActiveClusters(&n, dsa::mla::sparse_mla_tc_kernel<false>, &lc);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    c = n;
  }
  return c;
}

dsa_status_t enqueue_attention(const dsa::attn::Params &p_in, int B, cudaStream_t stream) {
  (void)B;
  dsa::attn::Params p = p_in;
  dsa::mla::Maps maps;
  std::memset(&maps, 0, sizeof(maps));
  for (int l = 0; l < p.n_layers; ++l)
    if (!make_tmap_576(&maps.q[l], p.q[l], static_cast<unsigned long long>(p.rows) * kHeads, kHeads))
      return DSA_ERR_CUDA;
  const long long rowsL = static_cast<long long>(p.n_layers) * p.rows;
  const long long blocks = p.tail_nsplit > 0 ? p.tail_base + (rowsL - p.tail_base) * p.tail_nsplit : rowsL * p.nsplit;
  // Several splits per unit, all units in one wave of clusters: each unit's
  // splits form a cluster that merges them itself (no partials in global
  // memory, no combine launch).
  p.cluster = (p.tail_nsplit == 0 && (p.nsplit == 2 || p.nsplit == 4 || p.nsplit == 8) &&
               attention_clusters(p.kv_fp8 != 0, p.nsplit) >= rowsL)
                  ? 1
                  : 0;
  // a programmatic dependent launch: the blocks may start (barriers, tensor
  // memory, the query panels) while the kernel before them on the stream
  // finishes; they wait for it (griddepcontrol.wait) before reading idx
  const dim3 grid(static_cast<unsigned>(blocks));
  const dim3 block(p.kv_fp8 ? dsa::mla::Roles<true>::kThreads : dsa::mla::Roles<false>::kThreads);
  cudaError_t e;
  if (p.cluster)
    e = p.kv_fp8 ? launch_dependent_cluster(dsa::mla::sparse_mla_tc_kernel<true>, grid, block, dsa::mla::kSmemBytes,
                                            stream, static_cast<unsigned>(p.nsplit), maps, p)
                 : launch_dependent_cluster(dsa::mla::sparse_mla_tc_kernel<false>, grid, block, dsa::mla::kSmemBytes,
                                            stream, static_cast<unsigned>(p.nsplit), maps, p);
  else
    e = p.kv_fp8 ? launch_dependent(dsa::mla::sparse_mla_tc_kernel<true>, grid, block, dsa::mla::kSmemBytes, stream,
                                    maps, p)
                 : launch_dependent(dsa::mla::sparse_mla_tc_kernel<false>, grid, block, dsa::mla::kSmemBytes, stream,
                                    maps, p);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  if (!p.cluster && (p.nsplit > 1 || p.tail_nsplit > 0)) {
    const long long cunits = p.tail_nsplit > 0 ? rowsL - p.tail_base : rowsL;
    const dim3 cgrid(kHeads, static_cast<unsigned>(cunits));
    if (launch_dependent(dsa::attn::combine_kernel, cgrid, dim3(128), 0, stream, p) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

inline int B_of(int rows, int Q) { return rows / Q; }

// Attention over n_layers layers (or draft steps) that share one index set.
// kv[l] points at bf16 rows, or at FP8 latent rows when kv_fp8.
dsa_status_t launch_attention(const DeviceState &dev, const Layout &L, uint8_t *ws, const dsa_bf16_t *const *q,
                              const void *const *kv, dsa_bf16_t *const *out, float *const *lse, int n_layers,
                              const int32_t *idx, int rows, int Q, int T, int K, float sm_scale,
                              cudaStream_t stream, const dsa_pages_t *pages = nullptr, bool kv_fp8 = false) {
  dsa::attn::Params p;
  std::memset(&p, 0, sizeof(p));
  for (int l = 0; l < n_layers; ++l) {
    p.q[l] = reinterpret_cast<const __nv_bfloat16 *>(q[l]);
    p.kv[l] = kv[l];
    p.out[l] = reinterpret_cast<__nv_bfloat16 *>(out[l]);
    p.lse[l] = lse ? lse[l] : nullptr;
  }
  p.kv_fp8 = kv_fp8 ? 1 : 0;
  p.idx = idx;
  p.n_layers = n_layers;
  p.Q = Q;
  p.T = T;
  p.K = K;
  p.rows = rows;
  const AttnShape a = attn_shape(static_cast<long long>(rows) * n_layers, K, dev.sms);
  p.nsplit = a.nsplit;
  p.blocks_per_split = a.bps;
  p.tail_base = static_cast<int>(a.tail_base);
  p.tail_nsplit = a.tail_nsplit;
  p.tail_bps = a.tail_bps;
  p.part_o = reinterpret_cast<float *>(ws + L.part_o);
  p.part_ml = reinterpret_cast<float *>(ws + L.part_ml);
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  if (pages != nullptr) {
    p.block_table = pages->block_table;
    p.page_size = pages->page_size;
    p.max_pages = pages->max_pages;
    p.num_pages = pages->num_pages;
  }
  return enqueue_attention(p, B_of(rows, Q), stream);
}

#define DSA_TRY(expr)                 \
  do {                                \
    const dsa_status_t s_ = (expr);   \
    if (s_ != DSA_OK) return s_;      \
  } while (0)

// One IndexShare group (sizes and config already checked): the indexer and
// top-k once, then every layer over the same index set.  `pages` (nullable)
// describes a paged key cache and paged latent caches; kv[l] holds FP8
// latent rows when kv_fp8.
dsa_status_t group_forward(const dsa_config_t *cfg, const void *q_idx, const float *w, const void *k_idx,
                           const int32_t *q_pos, const dsa_bf16_t *const *q, const void *const *kv,
                           int n_layers, int B, int Q, int T, dsa_bf16_t *const *out, int32_t *idx_out, void *ws,
                           size_t ws_bytes, cudaStream_t st, const dsa_pages_t *pages,
                           const float *q_scale = nullptr, const float *k_scale = nullptr, bool kv_fp8 = false) {
  if (n_layers < 1 || n_layers > kMaxLayers) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Q * n_layers > kMaxRowsY) return DSA_ERR_INVALID_ARG;
  if (!q_idx || !w || !k_idx || !q_pos || !q || !kv || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(q_pos) || (idx_out && !aligned16(idx_out)))
    return DSA_ERR_ALIGNMENT;
  for (int l = 0; l < n_layers; ++l) {
    if (!q[l] || !kv[l] || !out[l]) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q[l]) || !aligned16(kv[l]) || !aligned16(out[l])) return DSA_ERR_ALIGNMENT;
  }
  if (ws == nullptr) return DSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, n_layers, cfg->topk, dev->sms);
  if (ws_bytes < L.total) return DSA_ERR_WORKSPACE;
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  float *scores = reinterpret_cast<float *>(wsb + L.scores);
  int32_t *idx = idx_out ? idx_out : reinterpret_cast<int32_t *>(wsb + L.idx);
  // IndexShare: the indexer and top-k run once for the whole group ...
  // one query per sequence: the indexer counts the top-k's first histogram
  const bool fuse_hist = Q == 1 && L.ts.nchunk > 1;
  if (fuse_hist) DSA_TRY(clear_topk_state(L, wsb, st));
  DSA_TRY(launch_indexer(*dev, q_idx, w, k_idx, q_pos, B, Q, T, scores, st,
                         fuse_hist ? reinterpret_cast<uint32_t *>(wsb + L.ghist) : nullptr, pages, q_scale,
                         k_scale));
  DSA_TRY(launch_topk(L, wsb, scores, q_pos, B * Q, T, cfg->topk, idx, st, fuse_hist));
  // ... and every layer of the group attends over the same index set.
  return launch_attention(*dev, L, wsb, q, kv, out, nullptr, n_layers, idx, B * Q, Q, T, cfg->topk, cfg->sm_scale,
                          st, pages, kv_fp8);
}

}  // namespace

extern "C" {

void dsa_config_default(dsa_config_t *cfg) {
  if (cfg == nullptr) return;
  cfg->n_idx_heads = kIdxHeads;
  cfg->idx_dim = kIdxDim;
  cfg->topk = kMaxTopk;
  cfg->topk_freq = 4;
  cfg->kv_lora_rank = kLora;
  cfg->rope_dim = kRope;
  cfg->n_heads = kHeads;
  cfg->sm_scale = 1.0f / std::sqrt(static_cast<float>(kLora + kRope));
  cfg->index_share_for_mtp = 1;
}

size_t dsa_workspace_bytes(const dsa_config_t *cfg, int B, int Q, int T, int n_layers) {
  if (check_config(cfg) == DSA_OK && empty_call(B, Q, T) && n_layers >= 1 && n_layers <= kMaxLayers) return 256;
  if (check_config(cfg) != DSA_OK || check_sizes(B, Q, T) != DSA_OK || n_layers < 1 || n_layers > kMaxLayers)
    return 0;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return 0;
  return layout(B, Q, T, n_layers, cfg->topk, dev->sms).total;
}

dsa_status_t dsa_indexer_scores(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                const dsa_bf16_t *k_idx, const int32_t *q_pos, int B, int Q, int T, float *scores,
                                dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q_idx || !w || !k_idx || !q_pos || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(q_pos) || !aligned16(scores))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  return launch_indexer(*dev, q_idx, w, k_idx, q_pos, B, Q, T, scores, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_topk_select(const dsa_config_t *cfg, const float *scores, const int32_t *q_pos, int B, int Q, int T,
                             int32_t *idx, void *ws, size_t ws_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!scores || !q_pos || !idx) return DSA_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(q_pos) || !aligned16(idx) || (ws && !aligned16(ws))) return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, 1, cfg->topk, dev->sms);
  if (L.ts.nchunk > 1 && (ws == nullptr || ws_bytes < L.total)) return DSA_ERR_WORKSPACE;
  return launch_topk(L, static_cast<uint8_t *>(ws), scores, q_pos, B * Q, T, cfg->topk, idx,
                     reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_sparse_mla_attn(const dsa_config_t *cfg, const dsa_bf16_t *q, const dsa_bf16_t *kv,
                                 const int32_t *idx, int B, int Q, int T, dsa_bf16_t *out, float *lse, void *ws,
                                 size_t ws_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (ws && !aligned16(ws)))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, 1, cfg->topk, dev->sms);
  if (attn_shape(static_cast<long long>(B) * Q, cfg->topk, dev->sms).nsplit > 1 &&
      (ws == nullptr || ws_bytes < L.total))
    return DSA_ERR_WORKSPACE;
  const dsa_bf16_t *qs[1] = {q};
  const void *kvs[1] = {kv};
  dsa_bf16_t *outs[1] = {out};
  float *lses[1] = {lse};
  return launch_attention(*dev, L, static_cast<uint8_t *>(ws), qs, kvs, outs, lses, 1, idx, B * Q, Q, T, cfg->topk,
                          cfg->sm_scale, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_indexshare_group_forward(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                          const dsa_bf16_t *k_idx, const int32_t *q_pos, const dsa_bf16_t *const *q,
                                          const dsa_bf16_t *const *kv, int n_layers, int B, int Q, int T,
                                          dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                          dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  return group_forward(cfg, q_idx, w, k_idx, q_pos, q, reinterpret_cast<const void *const *>(kv), n_layers, B, Q, T,
                       out, idx_out, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream), nullptr);
}

dsa_status_t dsa_sparse_mla_attn_shared(const dsa_config_t *cfg, const dsa_bf16_t *const *q,
                                        const dsa_bf16_t *const *kv, int n_layers, const int32_t *idx, int B,
                                        int Q, int T, dsa_bf16_t *const *out, void *ws, size_t ws_bytes,
                                        dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (n_layers < 1 || n_layers > kMaxLayers) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Q * n_layers > kMaxRowsY) return DSA_ERR_INVALID_ARG;
  if (!q || !kv || !out || !idx) return DSA_ERR_INVALID_ARG;
  if (!aligned16(idx) || (ws && !aligned16(ws))) return DSA_ERR_ALIGNMENT;
  for (int l = 0; l < n_layers; ++l) {
    if (!q[l] || !kv[l] || !out[l]) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q[l]) || !aligned16(kv[l]) || !aligned16(out[l])) return DSA_ERR_ALIGNMENT;
  }
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, n_layers, cfg->topk, dev->sms);
  if (attn_shape(static_cast<long long>(B) * Q * n_layers, cfg->topk, dev->sms).nsplit > 1 &&
      (ws == nullptr || ws_bytes < L.total))
    return DSA_ERR_WORKSPACE;
  return launch_attention(*dev, L, static_cast<uint8_t *>(ws), q, reinterpret_cast<const void *const *>(kv), out,
                          nullptr, n_layers, idx, B * Q, Q, T, cfg->topk, cfg->sm_scale,
                          reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_mtp_draft_attn(const dsa_config_t *cfg, const int32_t *idx0, const dsa_bf16_t *q_steps,
                                const dsa_bf16_t *kv, int S, int B, int T, dsa_bf16_t *out, void *ws, size_t ws_bytes,
                                dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (!cfg->index_share_for_mtp) return DSA_ERR_UNSUPPORTED;
  if (empty_call(B, S, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, 1, T));
  if (S < 1 || S > kMaxLayers || static_cast<long long>(S) * B > kMaxRowsY) return DSA_ERR_INVALID_ARG;
  if (!idx0 || !q_steps || !kv || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(idx0) || !aligned16(q_steps) || !aligned16(kv) || !aligned16(out) || (ws && !aligned16(ws)))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, 1, T, S, cfg->topk, dev->sms);
  if (attn_shape(static_cast<long long>(B) * S, cfg->topk, dev->sms).nsplit > 1 &&
      (ws == nullptr || ws_bytes < L.total))
    return DSA_ERR_WORKSPACE;
  const dsa_bf16_t *qs[kMaxLayers];
  const void *kvs[kMaxLayers];
  dsa_bf16_t *outs[kMaxLayers];
  const size_t qstep = static_cast<size_t>(B) * kHeads * (kLora + kRope);
  const size_t ostep = static_cast<size_t>(B) * kHeads * kLora;
  for (int s = 0; s < S; ++s) {
    qs[s] = q_steps + s * qstep;
    kvs[s] = kv;  // KV share: every draft step reads the target's cache only
    outs[s] = out + s * ostep;
  }
  return launch_attention(*dev, L, static_cast<uint8_t *>(ws), qs, kvs, outs, nullptr, S, idx0, B, 1, T, cfg->topk,
                          cfg->sm_scale, reinterpret_cast<cudaStream_t>(stream));
}


dsa_status_t dsa_indexer_scores_paged(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                      const dsa_bf16_t *k_pool, const dsa_pages_t *pages, const int32_t *q_pos, int B,
                                      int Q, int T, float *scores, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  if (!q_idx || !w || !k_pool || !q_pos || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_pool) || !aligned16(q_pos) || !aligned16(scores))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  return launch_indexer(*dev, q_idx, w, k_pool, q_pos, B, Q, T, scores, reinterpret_cast<cudaStream_t>(stream),
                        nullptr, pages);
}

dsa_status_t dsa_sparse_mla_attn_paged(const dsa_config_t *cfg, const dsa_bf16_t *q, const dsa_bf16_t *kv_pool,
                                       const dsa_pages_t *pages, const int32_t *idx, int B, int Q, int T,
                                       dsa_bf16_t *out, float *lse, void *ws, size_t ws_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  if (!q || !kv_pool || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (ws && !aligned16(ws)))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, 1, cfg->topk, dev->sms);
  if (attn_shape(static_cast<long long>(B) * Q, cfg->topk, dev->sms).nsplit > 1 &&
      (ws == nullptr || ws_bytes < L.total))
    return DSA_ERR_WORKSPACE;
  const dsa_bf16_t *qs[1] = {q};
  const void *kvs[1] = {kv_pool};
  dsa_bf16_t *outs[1] = {out};
  float *lses[1] = {lse};
  return launch_attention(*dev, L, static_cast<uint8_t *>(ws), qs, kvs, outs, lses, 1, idx, B * Q, Q, T, cfg->topk,
                          cfg->sm_scale, reinterpret_cast<cudaStream_t>(stream), pages);
}

dsa_status_t dsa_indexshare_group_forward_paged(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                                const dsa_bf16_t *k_pool, const int32_t *q_pos,
                                                const dsa_bf16_t *const *q, const dsa_bf16_t *const *kv_pools,
                                                int n_layers, const dsa_pages_t *pages, int B, int Q, int T,
                                                dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                                dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  return group_forward(cfg, q_idx, w, k_pool, q_pos, q, reinterpret_cast<const void *const *>(kv_pools), n_layers, B,
                       Q, T, out, idx_out, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream), pages);
}

dsa_status_t dsa_indexer_scores_fp8(const dsa_config_t *cfg, const uint8_t *q_idx8, const float *q_scale,
                                    const float *w, const uint8_t *k_idx8, const float *k_scale, const int32_t *q_pos,
                                    int B, int Q, int T, float *scores, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q_idx8 || !q_scale || !w || !k_idx8 || !k_scale || !q_pos || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx8) || !aligned16(q_scale) || !aligned16(w) || !aligned16(k_idx8) || !aligned16(k_scale) ||
      !aligned16(q_pos) || !aligned16(scores))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  return launch_indexer(*dev, q_idx8, w, k_idx8, q_pos, B, Q, T, scores, reinterpret_cast<cudaStream_t>(stream),
                        nullptr, nullptr, q_scale, k_scale);
}

dsa_status_t dsa_indexshare_group_forward_fp8(const dsa_config_t *cfg, const uint8_t *q_idx8, const float *q_scale,
                                              const float *w, const uint8_t *k_idx8, const float *k_scale,
                                              const int32_t *q_pos, const dsa_bf16_t *const *q,
                                              const dsa_bf16_t *const *kv, int n_layers, int B, int Q, int T,
                                              dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                              dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q_scale || !k_scale) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_scale) || !aligned16(k_scale)) return DSA_ERR_ALIGNMENT;
  return group_forward(cfg, q_idx8, w, k_idx8, q_pos, q, reinterpret_cast<const void *const *>(kv), n_layers, B, Q,
                       T, out, idx_out, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream), nullptr, q_scale, k_scale);
}

dsa_status_t dsa_sparse_mla_attn_fp8(const dsa_config_t *cfg, const dsa_bf16_t *q, const uint8_t *kv8,
                                     const int32_t *idx, int B, int Q, int T, dsa_bf16_t *out, float *lse, void *ws,
                                     size_t ws_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q || !kv8 || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv8) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (ws && !aligned16(ws)))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, 1, cfg->topk, dev->sms);
  if (attn_shape(static_cast<long long>(B) * Q, cfg->topk, dev->sms).nsplit > 1 &&
      (ws == nullptr || ws_bytes < L.total))
    return DSA_ERR_WORKSPACE;
  const dsa_bf16_t *qs[1] = {q};
  const void *kvs[1] = {kv8};
  dsa_bf16_t *outs[1] = {out};
  float *lses[1] = {lse};
  return launch_attention(*dev, L, static_cast<uint8_t *>(ws), qs, kvs, outs, lses, 1, idx, B * Q, Q, T, cfg->topk,
                          cfg->sm_scale, reinterpret_cast<cudaStream_t>(stream), nullptr, true);
}

dsa_status_t dsa_indexshare_group_forward_fp8kv(const dsa_config_t *cfg, const uint8_t *q_idx8,
                                                const float *q_scale, const float *w, const uint8_t *k_idx8,
                                                const float *k_scale, const int32_t *q_pos, const dsa_bf16_t *const *q,
                                                const uint8_t *const *kv8, int n_layers, int B, int Q, int T,
                                                dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                                dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q_scale || !k_scale) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_scale) || !aligned16(k_scale)) return DSA_ERR_ALIGNMENT;
  return group_forward(cfg, q_idx8, w, k_idx8, q_pos, q, reinterpret_cast<const void *const *>(kv8), n_layers, B, Q,
                       T, out, idx_out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, q_scale,
                       k_scale, true);
}

dsa_status_t dsa_indexer_scores_fp8_paged(const dsa_config_t *cfg, const uint8_t *q_idx8, const float *q_scale,
                                          const float *w, const uint8_t *k8_pool, const float *k_scale_pool,
                                          const dsa_pages_t *pages, const int32_t *q_pos, int B, int Q, int T,
                                          float *scores, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  if (!q_idx8 || !q_scale || !w || !k8_pool || !k_scale_pool || !q_pos || !scores) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx8) || !aligned16(q_scale) || !aligned16(w) || !aligned16(k8_pool) ||
      !aligned16(k_scale_pool) || !aligned16(q_pos) || !aligned16(scores))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  return launch_indexer(*dev, q_idx8, w, k8_pool, q_pos, B, Q, T, scores, reinterpret_cast<cudaStream_t>(stream),
                        nullptr, pages, q_scale, k_scale_pool);
}

dsa_status_t dsa_sparse_mla_attn_fp8_paged(const dsa_config_t *cfg, const dsa_bf16_t *q, const uint8_t *kv8_pool,
                                           const dsa_pages_t *pages, const int32_t *idx, int B, int Q, int T,
                                           dsa_bf16_t *out, float *lse, void *ws, size_t ws_bytes,
                                           dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  if (!q || !kv8_pool || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv8_pool) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (ws && !aligned16(ws)))
    return DSA_ERR_ALIGNMENT;
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  const Layout L = layout(B, Q, T, 1, cfg->topk, dev->sms);
  if (attn_shape(static_cast<long long>(B) * Q, cfg->topk, dev->sms).nsplit > 1 &&
      (ws == nullptr || ws_bytes < L.total))
    return DSA_ERR_WORKSPACE;
  const dsa_bf16_t *qs[1] = {q};
  const void *kvs[1] = {kv8_pool};
  dsa_bf16_t *outs[1] = {out};
  float *lses[1] = {lse};
  return launch_attention(*dev, L, static_cast<uint8_t *>(ws), qs, kvs, outs, lses, 1, idx, B * Q, Q, T, cfg->topk,
                          cfg->sm_scale, reinterpret_cast<cudaStream_t>(stream), pages, true);
}

dsa_status_t dsa_indexshare_group_forward_fp8_paged(const dsa_config_t *cfg, const uint8_t *q_idx8,
                                                    const float *q_scale, const float *w, const uint8_t *k8_pool,
                                                    const float *k_scale_pool, const int32_t *q_pos,
                                                    const dsa_bf16_t *const *q, const dsa_bf16_t *const *kv_pools,
                                                    int n_layers, const dsa_pages_t *pages, int B, int Q, int T,
                                                    dsa_bf16_t *const *out, int32_t *idx_out, void *ws,
                                                    size_t ws_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  if (!q_scale || !k_scale_pool) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_scale) || !aligned16(k_scale_pool)) return DSA_ERR_ALIGNMENT;
  return group_forward(cfg, q_idx8, w, k8_pool, q_pos, q, reinterpret_cast<const void *const *>(kv_pools), n_layers,
                       B, Q, T, out, idx_out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), pages, q_scale,
                       k_scale_pool);
}

dsa_status_t dsa_indexshare_group_forward_fp8kv_paged(const dsa_config_t *cfg, const uint8_t *q_idx8,
                                                      const float *q_scale, const float *w, const uint8_t *k8_pool,
                                                      const float *k_scale_pool, const int32_t *q_pos,
                                                      const dsa_bf16_t *const *q, const uint8_t *const *kv8_pools,
                                                      int n_layers, const dsa_pages_t *pages, int B, int Q, int T,
                                                      dsa_bf16_t *const *out, int32_t *idx_out, void *ws,
                                                      size_t ws_bytes, dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  DSA_TRY(check_pages(pages, B, T));
  if (!q_scale || !k_scale_pool) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_scale) || !aligned16(k_scale_pool)) return DSA_ERR_ALIGNMENT;
  return group_forward(cfg, q_idx8, w, k8_pool, q_pos, q, reinterpret_cast<const void *const *>(kv8_pools), n_layers,
                       B, Q, T, out, idx_out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), pages, q_scale,
                       k_scale_pool, true);
}
}  // extern "C"

// ---------------------------------------------------------------------------
// Attention without a caller workspace: the split-k partials live in a fixed
// array compiled into the library.  In host code `g_noalloc_partials` names a
// host-side stand-in, not device memory: its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kNoAllocMaxRows = 64;                          // B * Q per call
constexpr size_t kPartialTileBytes = size_t(kHeads) * kLora * 4;  // one (row, split) partial O
constexpr size_t kPartialMlBytes = size_t(kHeads) * 2 * 4;        // its (max, sum) per head
constexpr int kNoAllocTiles = static_cast<int>(kNoAllocScratchBytes / (kPartialTileBytes + kPartialMlBytes));

static __device__ __align__(256) unsigned char g_noalloc_partials[kNoAllocScratchBytes];

void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up once).
bool noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_partials) != cudaSuccess || ptr == nullptr) return false;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return true;
}

}  // namespace

extern "C" {

dsa_status_t dsa_sparse_mla_attn_noalloc(const dsa_config_t *cfg, const dsa_bf16_t *q, const dsa_bf16_t *kv,
                                         const int32_t *idx, int B, int Q, int T, dsa_bf16_t *out, float *lse,
                                         dsa_stream_t stream) {
  DSA_TRY(check_config(cfg));
  if (empty_call(B, Q, T)) return DSA_OK;
  DSA_TRY(check_sizes(B, Q, T));
  if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)))
    return DSA_ERR_ALIGNMENT;
  const int rows = B * Q;
  if (rows > kNoAllocMaxRows) return DSA_ERR_WORKSPACE;  // beyond what the static scratch holds
  DeviceState *dev = nullptr;
  if (!device_state(&dev)) return DSA_ERR_CUDA;
  void *scratch = nullptr;
  if (!noalloc_scratch(&scratch)) return DSA_ERR_CUDA;
  // the usual split of the index slots, with no more (row, split) partials
  // than the array holds; rows <= 64 always leaves at least one split
  AttnShape a = attn_shape(rows, cfg->topk, dev->sms);
  const int max_splits = kNoAllocTiles / rows;
  if (a.nsplit > max_splits) {
    const int nblocks = (cfg->topk + dsa::mla::kKeys - 1) / dsa::mla::kKeys;
    a.bps = (nblocks + max_splits - 1) / max_splits;
    a.nsplit = (nblocks + a.bps - 1) / a.bps;
  }
  dsa::attn::Params p;
  std::memset(&p, 0, sizeof(p));
  p.q[0] = reinterpret_cast<const __nv_bfloat16 *>(q);
  p.kv[0] = reinterpret_cast<const __nv_bfloat16 *>(kv);
  p.out[0] = reinterpret_cast<__nv_bfloat16 *>(out);
  p.lse[0] = lse;
  p.idx = idx;
  p.n_layers = 1;
  p.Q = Q;
  p.T = T;
  p.K = cfg->topk;
  p.rows = rows;
  p.nsplit = a.nsplit;
  p.blocks_per_split = a.bps;
  // every (row, split) partial is fully written before the combine reads it,
  // so nothing in the array has to be cleared between calls
  p.part_o = static_cast<float *>(scratch);
  p.part_ml = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + kNoAllocTiles * kPartialTileBytes);
  p.scale_log2 = cfg->sm_scale * 1.4426950408889634f;
  return enqueue_attention(p, B, reinterpret_cast<cudaStream_t>(stream));
}

const char *dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_ALIGNMENT: return "DSA_ERR_ALIGNMENT";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
  }
  return "DSA_ERR_UNKNOWN";
}

dsa_status_t dsa_set_wait_limit_ns(unsigned long long limit_ns) {
  const unsigned long long v = limit_ns == 0 ? dsa::kWaitLimitNs : limit_ns;
  return cudaMemcpyToSymbol(dsa::g_wait_limit_ns, &v, sizeof(v)) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t dsa_get_device_error(dsa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  unsigned word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, dsa::g_error_word, sizeof(word)) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpyToSymbol(dsa::g_error_word, &zero, sizeof(zero)) != cudaSuccess) return DSA_ERR_CUDA;
  if (word & dsa::kErrTimeout) return DSA_ERR_TIMEOUT;
  if (word & dsa::kErrDeviceCheck) return DSA_ERR_DEVICE_CHECK;
  return DSA_OK;
}

}  // extern "C"
