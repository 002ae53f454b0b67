// Top-k selection of indexer scores: per row keep the min(k, L) positions
// s < L = pos+1 with the largest scores, ties to the lower position, written in
// ascending position order and padded with -1 ("GLM-5.2 Explained: 1M Token
// Context AI Agent Model", §2.1: the indexer keeps the top-K positions;
// index_topk = 2048 in the GLM-5.2 config).
//
// Radix select, no sort.  Each fp32 score maps to an order-preserving 32-bit
// key; three histogram passes (11 + 11 + 10 bits) find the exact k-th largest
// key tau and how many keys equal to tau are taken (`need`).  A final pass
// writes, in position order, every position with key > tau plus the first
// `need` positions with key == tau.  All counts are integers, so the result
// does not depend on thread scheduling.
//
// Two launch shapes:
//   * many rows (prefill): one block per row runs every pass over its row;
//   * few long rows (decode): each row is cut into chunks, one block per
//     (chunk, row); the histograms are summed in global memory, every block
//     re-derives tau from them, and a per-chunk count pass gives each chunk
//     its output offset.  No block ever waits on another: passes are
//     separate launches in stream order.
#pragma once

#include "common.cuh"

namespace dsa {
namespace topk {

constexpr int kThreads = 512;
constexpr int kMaxBins = 2048;
constexpr int kPasses = 3;

__device__ __forceinline__ int pass_shift(int p) { return p == 0 ? 21 : (p == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t pass_digit_mask(int p) { return p == 2 ? 0x3FFu : 0x7FFu; }
__device__ __forceinline__ int pass_bins(int p) { return p == 2 ? 1024 : 2048; }
// Bits above this pass's digit: the prefix fixed by earlier passes.
__device__ __forceinline__ uint32_t pass_high_mask(int p) {
  return p == 0 ? 0u : (p == 1 ? 0xFFE00000u : 0xFFFFFC00u);
}

__device__ __forceinline__ int visible_length(const int32_t *q_pos, int row, int T) {
  const int pos = __ldg(q_pos + row);
  if (pos < 0 || pos >= T) raise_error(kErrDeviceCheck);
  const int L = pos + 1;
  return L < 0 ? 0 : (L > T ? T : L);
}

struct Scratch {
  uint32_t warp_a[kThreads / 32];
  uint32_t warp_b[kThreads / 32];
  uint32_t result[4];
};

// Given a histogram (nbins <= 2048 bins, in shared memory) and 1 <= need <=
// total count, finds the bin b such that count(bins > b) < need <= count(bins
// >= b).  Writes b to sc->result[0] and need - count(bins > b) to result[1].
// Called by every thread of the block; ends with the result visible to all.
__device__ void find_threshold_bin(const uint32_t *hist, int nbins, uint32_t need, Scratch *sc) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = nbins / kThreads;  // 2 or 4 bins per thread
  uint32_t h[4] = {0, 0, 0, 0};
  uint32_t ts = 0;
  for (int i = 0; i < per; ++i) {
    h[i] = hist[t * per + i];
    ts += h[i];
  }
  // suffix sum over threads (>= t) via warp shuffles, then over warps
  uint32_t v = ts;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t n = __shfl_down_sync(0xffffffffu, v, off);
    if (lane + off < 32) v += n;
  }
  if (lane == 0) sc->warp_a[warp] = v;
  __syncthreads();
  uint32_t above_warps = 0;
  for (int w = warp + 1; w < kThreads / 32; ++w) above_warps += sc->warp_a[w];
  uint32_t cum = v + above_warps - ts;  // count in bins of threads > t
  for (int i = per - 1; i >= 0; --i) {
    if (cum < need && need <= cum + h[i]) {
      sc->result[0] = static_cast<uint32_t>(t * per + i);
      sc->result[1] = need - cum;
    }
    cum += h[i];
  }
  __syncthreads();
}

// Block-wide exclusive prefix of a 0/1 flag in thread order; also returns the
// block total.  Uses sc->warp_b; ends with a __syncthreads.
__device__ __forceinline__ uint32_t block_prefix(bool flag, uint32_t *total, Scratch *sc) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  const uint32_t in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) sc->warp_b[warp] = __popc(bal);
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const uint32_t c = sc->warp_b[w];
    before += (w < warp) ? c : 0u;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return before + in_warp;
}

// Ordered write of the selection for positions [start, end) of one row.
// `out_base` is the number of selected positions before `start`, `eq_base` the
// number of keys equal to tau before `start`.
__device__ void write_selected(const float *srow, int start, int end, uint32_t tau, uint32_t need,
                               uint32_t out_base, uint32_t eq_base, int32_t *out, Scratch *sc) {
  for (int t0 = start; t0 < end; t0 += kThreads) {
    const int i = t0 + threadIdx.x;
    const bool in = i < end;
    const uint32_t key = in ? score_key(__ldg(srow + i)) : 0u;
    const bool gt = in && key > tau;
    const bool eq = in && key == tau;
    uint32_t eq_tot, sel_tot;
    const uint32_t eq_rank = eq_base + block_prefix(eq, &eq_tot, sc);
    const bool sel = gt || (eq && eq_rank < need);
    const uint32_t slot = out_base + block_prefix(sel, &sel_tot, sc);
    if (sel) out[slot] = i;
    out_base += sel_tot;
    eq_base += eq_tot;
  }
}

// --------------------------------------------------------------------------
// One block per row: every pass over the row inside one block.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const float *__restrict__ scores,
                                                            const int32_t *__restrict__ q_pos, int T, int K,
                                                            int32_t *__restrict__ idx) {
  __shared__ uint32_t hist[kMaxBins];
  __shared__ Scratch sc;
  const int row = blockIdx.x;
  const int L = visible_length(q_pos, row, T);
  const float *srow = scores + (size_t)row * T;
  int32_t *out = idx + (size_t)row * K;
  if (L <= K) {
    for (int i = threadIdx.x; i < K; i += kThreads) out[i] = i < L ? i : -1;
    return;
  }
  uint32_t prefix = 0, need = static_cast<uint32_t>(K);
  for (int p = 0; p < kPasses; ++p) {
    const int nb = pass_bins(p), sh = pass_shift(p);
    const uint32_t hm = pass_high_mask(p), dm = pass_digit_mask(p);
    for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < L; i += kThreads) {
      const uint32_t key = score_key(__ldg(srow + i));
      if ((key & hm) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    find_threshold_bin(hist, nb, need, &sc);
    prefix |= sc.result[0] << sh;
    need = sc.result[1];
    __syncthreads();
  }
  write_selected(srow, 0, L, prefix, need, 0, 0, out, &sc);
}

// --------------------------------------------------------------------------
// Few long rows: (chunk, row) blocks.  ghist [kPasses][rows][kMaxBins] must be
// zero before pass 0; counts [rows][nchunk][2] = (#key > tau, #key == tau).
// --------------------------------------------------------------------------
struct ChunkParams {
  const float *scores;
  const int32_t *q_pos;
  int T, K, rows, chunk, nchunk;
  uint32_t *ghist;
  uint32_t *counts;
  int32_t *idx;
};

// Re-derives (prefix, need) from the global histograms of passes < npass.
__device__ void derive_prefix(const ChunkParams &p, int row, int npass, uint32_t *hist, Scratch *sc,
                              uint32_t *prefix_out, uint32_t *need_out) {
  uint32_t prefix = 0, need = static_cast<uint32_t>(p.K);
  for (int q = 0; q < npass; ++q) {
    const int nb = pass_bins(q);
    const uint32_t *g = p.ghist + ((size_t)q * p.rows + row) * kMaxBins;
    for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = g[i];
    __syncthreads();
    find_threshold_bin(hist, nb, need, sc);
    prefix |= sc->result[0] << pass_shift(q);
    need = sc->result[1];
    __syncthreads();
  }
  *prefix_out = prefix;
  *need_out = need;
}

template <int PASS>
__global__ void __launch_bounds__(kThreads) topk_chunk_hist_kernel(const ChunkParams p) {
  __shared__ uint32_t hist[kMaxBins];
  __shared__ Scratch sc;
  const int row = blockIdx.y, c = blockIdx.x;
  const int L = visible_length(p.q_pos, row, p.T);
  const int start = c * p.chunk;
  if (L <= p.K || start >= L) return;
  const int end = min(start + p.chunk, L);
  uint32_t prefix, need;
  derive_prefix(p, row, PASS, hist, &sc, &prefix, &need);
  const int nb = pass_bins(PASS), sh = pass_shift(PASS);
  const uint32_t hm = pass_high_mask(PASS), dm = pass_digit_mask(PASS);
  for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
  __syncthreads();
  const float *srow = p.scores + (size_t)row * p.T;
  for (int i = start + threadIdx.x; i < end; i += kThreads) {
    const uint32_t key = score_key(__ldg(srow + i));
    if ((key & hm) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
  }
  __syncthreads();
  uint32_t *g = p.ghist + ((size_t)PASS * p.rows + row) * kMaxBins;
  for (int i = threadIdx.x; i < nb; i += kThreads)
    if (hist[i]) atomicAdd(g + i, hist[i]);
}

__global__ void __launch_bounds__(kThreads) topk_chunk_count_kernel(const ChunkParams p) {
  __shared__ uint32_t hist[kMaxBins];
  __shared__ Scratch sc;
  const int row = blockIdx.y, c = blockIdx.x;
  const int L = visible_length(p.q_pos, row, p.T);
  const int start = c * p.chunk;
  if (L <= p.K) return;
  uint32_t tau, need;
  derive_prefix(p, row, kPasses, hist, &sc, &tau, &need);
  uint32_t gt = 0, eq = 0;
  const int end = min(start + p.chunk, L);
  const float *srow = p.scores + (size_t)row * p.T;
  for (int i = start + threadIdx.x; i < end; i += kThreads) {
    const uint32_t key = score_key(__ldg(srow + i));
    gt += key > tau;
    eq += key == tau;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, off);
    eq += __shfl_xor_sync(0xffffffffu, eq, off);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sc.warp_a[warp] = gt;
    sc.warp_b[warp] = eq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t G = 0, E = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      G += sc.warp_a[w];
      E += sc.warp_b[w];
    }
    uint32_t *dst = p.counts + ((size_t)row * p.nchunk + c) * 2;
    dst[0] = G;
    dst[1] = E;
  }
}

__global__ void __launch_bounds__(kThreads) topk_chunk_write_kernel(const ChunkParams p) {
  __shared__ uint32_t hist[kMaxBins];
  __shared__ Scratch sc;
  const int row = blockIdx.y, c = blockIdx.x;
  const int L = visible_length(p.q_pos, row, p.T);
  int32_t *out = p.idx + (size_t)row * p.K;
  if (L <= p.K) {
    if (c == 0)
      for (int i = threadIdx.x; i < p.K; i += kThreads) out[i] = i < L ? i : -1;
    return;
  }
  const int start = c * p.chunk;
  if (start >= L) return;
  uint32_t tau, need;
  derive_prefix(p, row, kPasses, hist, &sc, &tau, &need);
  // selections before this chunk: every key > tau, plus the first `need` keys == tau
  uint32_t gt_before = 0, eq_before = 0;
  for (int cc = threadIdx.x; cc < c; cc += kThreads) {
    const uint32_t *src = p.counts + ((size_t)row * p.nchunk + cc) * 2;
    gt_before += src[0];
    eq_before += src[1];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gt_before += __shfl_xor_sync(0xffffffffu, gt_before, off);
    eq_before += __shfl_xor_sync(0xffffffffu, eq_before, off);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sc.warp_a[warp] = gt_before;
    sc.warp_b[warp] = eq_before;
  }
  __syncthreads();
  uint32_t G = 0, E = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    G += sc.warp_a[w];
    E += sc.warp_b[w];
  }
  __syncthreads();
  const uint32_t out_base = G + (E < need ? E : need);
  const int end = min(start + p.chunk, L);
  write_selected(p.scores + (size_t)row * p.T, start, end, tau, need, out_base, E, out, &sc);
}

}  // namespace topk
}  // namespace dsa
