// Top-k selection of indexer scores: per row keep the min(k, L) positions
// s < L = pos+1 with the largest scores, ties to the lower position, written in
// ascending position order and padded with -1 ("GLM-5.2 Explained: 1M Token
// Context AI Agent Model", §2.1: the indexer keeps the top-K positions;
// index_topk = 2048 in the GLM-5.2 config).
//
// Radix select, no full sort of the row.  Each fp32 score maps to an
// order-preserving 32-bit key; (key, position) then maps to a unique 64-bit
// composite (key << 32 | ~position), whose descending order is exactly
// "score desc, position asc".  The k largest composites are the selection.
//
//   1. histogram of the top 11 key bits (digit 0) over the row -> the bin b0
//      holding the k-th largest key;
//   2. pass 1 over the row: every position with digit 0 > b0 is a candidate;
//      positions in bin b0 feed a histogram of the next 11 bits (digit 1);
//   3. pass 2 over the row: positions in bin b0 whose digit 1 is >= b1 (the
//      sub-bin holding the k-th key) are candidates too;
//   4. radix select over the ~k candidates' composites gives the exact k-th
//      composite tau; the k positions with composite >= tau are sorted
//      ascending (bitonic, in shared memory) and written.
// Every count is an integer and the final order comes from a sort, so the
// result does not depend on thread scheduling.
//
// Two launch shapes:
//   * many rows (prefill): one block per row does every step in shared memory;
//   * few long rows (decode): (chunk, row) blocks do steps 1-3 and append
//     candidates to a global buffer (one atomic per block), then one block per
//     row does step 4.  Step 1 may come fused from the indexer.  Passes are
//     separate launches in stream order; no block waits on another.
// If a row's candidates overflow the shared-memory buffer (e.g. thousands of
// exactly equal scores), the one-block-per-row path falls back to three
// exact radix passes over the row and an ordered write.
#pragma once

#include "common.cuh"

namespace dsa {
namespace topk {

constexpr int kThreads = 512;
constexpr int kBins = 2048;          // 11-bit digits
constexpr int kShift0 = 21;          // digit 0: key bits 31..21
constexpr int kShift1 = 10;          // digit 1: key bits 20..10
constexpr int kSortN = 2048;         // bitonic sort size (>= the largest k)
constexpr int kSmemCand = 11776;     // composites held in shared memory (92 KB: two blocks per SM)
constexpr int kBlockCand = 2048;     // candidates a chunk block stages before its one global append
constexpr int kUnroll = 8;

// dynamic shared memory of the select and row kernels
constexpr int kSelectSmem = kSmemCand * 8 + kBins * 4 + kSortN * 4;

__device__ __forceinline__ int visible_length(const int32_t *q_pos, int row, int T) {
  const int pos = __ldg(q_pos + row);
  if (pos < 0 || pos >= T) raise_error(kErrDeviceCheck);
  const int L = pos + 1;
  return L < 0 ? 0 : (L > T ? T : L);
}

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t pos) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~pos);
}
__device__ __forceinline__ int32_t composite_pos(uint64_t v) { return static_cast<int32_t>(~static_cast<uint32_t>(v)); }

struct Scratch {
  uint32_t warp_a[kThreads / 32];
  uint32_t warp_b[kThreads / 32];
  uint32_t result[4];
  uint32_t count;
  uint32_t base;
};

// Given a histogram of kBins bins in shared memory and 1 <= need <= total
// count, finds the bin b with count(bins > b) < need <= count(bins >= b).
// Writes b to sc->result[0], need - count(bins > b) to result[1] and the bin's
// own count to result[2].  Called by every thread; ends with the result visible.
__device__ void find_threshold_bin(const uint32_t *hist, uint32_t need, Scratch *sc) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr int per = kBins / kThreads;  // 4 bins per thread
  uint32_t h[per];
  uint32_t ts = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    h[i] = hist[t * per + i];
    ts += h[i];
  }
  uint32_t v = ts;  // suffix sum over the lanes of this warp at or after this lane
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t n = __shfl_down_sync(0xffffffffu, v, off);
    if (lane + off < 32) v += n;
  }
  if (lane == 0) sc->warp_a[warp] = v;
  __syncthreads();
  uint32_t above_warps = 0;
  for (int w = warp + 1; w < kThreads / 32; ++w) above_warps += sc->warp_a[w];
  uint32_t cum = v + above_warps - ts;  // count in the bins of later threads
#pragma unroll
  for (int i = per - 1; i >= 0; --i) {
    if (cum < need && need <= cum + h[i]) {
      sc->result[0] = static_cast<uint32_t>(t * per + i);
      sc->result[1] = need - cum;
      sc->result[2] = h[i];
    }
    cum += h[i];
  }
  __syncthreads();
}

// Block-wide exclusive prefix of a 0/1 flag in thread order, plus the total.
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

// Where candidates go: a shared-memory list of `cap` entries whose counter is
// sc->count; entries beyond it go straight to a global list (`gdst`, counter
// `gcount`, capacity `gcap`) when one is given, else they are only counted.
struct Sink {
  uint64_t *list;
  uint32_t cap;
  uint64_t *gdst;
  uint32_t *gcount;
  uint32_t gcap;
};

// Warp-aggregated append of `v` for every lane with take == true.  Every lane
// of the warp must call it.
__device__ __forceinline__ void sink_append(const Sink &s, Scratch *sc, bool take, uint64_t v) {
  const int lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, take);
  if (bal == 0) return;
  const int leader = __ffs(bal) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(&sc->count, static_cast<uint32_t>(__popc(bal)));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (!take) return;
  const uint32_t slot = base + __popc(bal & ((1u << lane) - 1u));
  if (slot < s.cap) {
    s.list[slot] = v;
  } else if (s.gdst != nullptr) {
    const uint32_t g = atomicAdd(s.gcount, 1u);
    if (g < s.gcap) s.gdst[g] = v;
  }
}

// Histogram of digit 0 of the row's keys over [start, end).
__device__ void hist_digit0(const float *srow, int start, int end, uint32_t *hist) {
  for (int base = start; base < end; base += kThreads * kUnroll) {
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      v[u] = i < end ? __ldg(srow + i) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      if (i < end) atomicAdd(&hist[score_key(v[u]) >> kShift0], 1u);
    }
  }
}

// Pass 1 over [start, end): digit 0 > b0 (>= b0 when the whole bin b0 is
// taken) -> candidate; digit 0 == b0 -> hist1[digit 1] (when hist1 is given).
// Pass 2 (pass2 == true): digit 0 == b0 and digit 1 >= b1 -> candidate.
__device__ void scan_row(const float *srow, int start, int end, bool pass2, uint32_t b0, bool whole_b0, uint32_t b1,
                         uint32_t *hist1, const Sink &sink, Scratch *sc) {
  for (int base = start; base < end; base += kThreads * kUnroll) {  // warp-uniform trip count
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      v[u] = i < end ? __ldg(srow + i) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      const uint32_t key = score_key(v[u]);
      const uint32_t d0 = key >> kShift0;
      bool take;
      if (!pass2) {
        take = i < end && (d0 > b0 || (whole_b0 && d0 == b0));
        if (hist1 != nullptr && i < end && d0 == b0) atomicAdd(&hist1[(key >> kShift1) & (kBins - 1)], 1u);
      } else {
        take = i < end && d0 == b0 && ((key >> kShift1) & (kBins - 1)) >= b1;
      }
      sink_append(sink, sc, take, composite(key, static_cast<uint32_t>(i)));
    }
  }
}

// Exact k-th largest composite among src[0..n) (1 <= k <= n): radix passes of
// 11-bit digits from the top, stopping as soon as the threshold bin is taken
// whole.  Every composite >= the returned value is selected: exactly k.
__device__ uint64_t select_threshold(const uint64_t *src, uint32_t n, uint32_t k, uint32_t *hist, Scratch *sc) {
  uint64_t prefix = 0, known = 0;
  uint32_t need = k;
  for (int shift = 53;; shift -= 11) {
    const int sh = shift < 0 ? 0 : shift;
    const int width = shift < 0 ? 11 + shift : 11;
    const uint64_t dmask = (1ull << width) - 1ull;
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
      const uint64_t v = src[i];
      if ((v & known) == prefix) atomicAdd(&hist[static_cast<uint32_t>((v >> sh) & dmask)], 1u);
    }
    __syncthreads();
    find_threshold_bin(hist, need, sc);
    const uint32_t bin = sc->result[0];
    const uint32_t rem = sc->result[1], cnt = sc->result[2];
    __syncthreads();
    prefix |= static_cast<uint64_t>(bin) << sh;
    known |= dmask << sh;
    if (rem == cnt || sh == 0) return prefix;  // the whole bin is taken: every lower bit may be zero
    need = rem;
  }
}

// Writes the k selected positions (composite >= tau among src[0..n)) in
// ascending order: gathered into `sortbuf`, bitonic-sorted, stored to out.
__device__ void write_sorted(const uint64_t *src, uint32_t n, uint64_t tau, int k, int32_t *sortbuf, int32_t *out,
                             Scratch *sc) {
  if (threadIdx.x == 0) sc->base = 0;
  for (int i = threadIdx.x; i < kSortN; i += kThreads) sortbuf[i] = 0x7FFFFFFF;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
    const uint64_t v = src[i];
    if (v >= tau) {
      const uint32_t slot = atomicAdd(&sc->base, 1u);
      if (slot < kSortN) sortbuf[slot] = composite_pos(v);
    }
  }
  __syncthreads();
  for (int size = 2; size <= kSortN; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < kSortN / 2; t += kThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const int32_t a = sortbuf[lo], b = sortbuf[hi];
        if ((a > b) == up) {
          sortbuf[lo] = b;
          sortbuf[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < k; i += kThreads) out[i] = sortbuf[i];
}

// Three exact radix passes over the row and an ordered write; used when the
// candidates do not fit in shared memory.
__device__ void row_select_multipass(const float *srow, int L, int K, int32_t *out, uint32_t *hist, Scratch *sc) {
  uint32_t prefix = 0, need = static_cast<uint32_t>(K);
  for (int p = 0; p < 3; ++p) {
    const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
    const uint32_t hm = p == 0 ? 0u : (p == 1 ? 0xFFE00000u : 0xFFFFFC00u);
    const uint32_t dm = p == 2 ? 0x3FFu : 0x7FFu;
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < L; i += kThreads) {
      const uint32_t key = score_key(__ldg(srow + i));
      if ((key & hm) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    find_threshold_bin(hist, need, sc);
    prefix |= sc->result[0] << sh;
    need = sc->result[1];
    __syncthreads();
  }
  const uint32_t tau = prefix;
  uint32_t out_base = 0, eq_base = 0;
  for (int t0 = 0; t0 < L; t0 += kThreads) {
    const int i = t0 + threadIdx.x;
    const bool in = i < L;
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

__device__ __forceinline__ bool write_short_row(int L, int K, int32_t *out) {
  if (L > K) return false;
  for (int i = threadIdx.x; i < K; i += kThreads) out[i] = i < L ? i : -1;
  return true;
}

struct SmemViews {
  uint64_t *cand;
  uint32_t *hist;
  int32_t *sortbuf;
};

__device__ __forceinline__ SmemViews smem_views(uint8_t *smem) {
  SmemViews s;
  s.cand = reinterpret_cast<uint64_t *>(smem);
  s.hist = reinterpret_cast<uint32_t *>(smem + kSmemCand * 8);
  s.sortbuf = reinterpret_cast<int32_t *>(smem + kSmemCand * 8 + kBins * 4);
  return s;
}

// --------------------------------------------------------------------------
// Many rows: one block per row does every step in shared memory.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const float *__restrict__ scores,
                                                            const int32_t *__restrict__ q_pos, int T, int K,
                                                            int32_t *__restrict__ idx) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ Scratch sc;
  const SmemViews s = smem_views(smem);
  const int row = blockIdx.x;
  const int L = visible_length(q_pos, row, T);
  const float *srow = scores + (size_t)row * T;
  int32_t *out = idx + (size_t)row * K;
  if (write_short_row(L, K, out)) return;
  uint32_t *hist1 = reinterpret_cast<uint32_t *>(s.sortbuf);  // the sort buffer is free until the end
  for (int i = threadIdx.x; i < kBins; i += kThreads) {
    s.hist[i] = 0;
    hist1[i] = 0;
  }
  if (threadIdx.x == 0) sc.count = 0;
  __syncthreads();
  hist_digit0(srow, 0, L, s.hist);
  __syncthreads();
  find_threshold_bin(s.hist, static_cast<uint32_t>(K), &sc);
  const uint32_t b0 = sc.result[0], need1 = sc.result[1];
  const bool whole = sc.result[1] == sc.result[2];
  const Sink sink{s.cand, kSmemCand, nullptr, nullptr, 0};
  scan_row(srow, 0, L, false, b0, whole, 0, whole ? nullptr : hist1, sink, &sc);
  __syncthreads();
  if (!whole) {
    find_threshold_bin(hist1, need1, &sc);
    const uint32_t b1 = sc.result[0];
    scan_row(srow, 0, L, true, b0, false, b1, nullptr, sink, &sc);
    __syncthreads();
  }
  const uint32_t n = sc.count;
  __syncthreads();
  if (n > static_cast<uint32_t>(kSmemCand)) {
    row_select_multipass(srow, L, K, out, s.hist, &sc);
    return;
  }
  const uint64_t tau = select_threshold(s.cand, n, static_cast<uint32_t>(K), s.hist, &sc);
  write_sorted(s.cand, n, tau, K, s.sortbuf, out, &sc);
}

// --------------------------------------------------------------------------
// Few long rows: (chunk, row) blocks.  ghist [rows][2][kBins] (digit 0, then
// digit 1 within bin b0) and gcount [rows] must be zero before step 1;
// cand [rows][T] holds the composites.
// --------------------------------------------------------------------------
struct ChunkParams {
  const float *scores;
  const int32_t *q_pos;
  int T, K, rows, chunk, nchunk;
  uint32_t *ghist;
  uint32_t *gcount;
  uint64_t *cand;
  int32_t *idx;
};

__global__ void __launch_bounds__(kThreads) topk_chunk_hist_kernel(const ChunkParams p) {
  __shared__ uint32_t hist[kBins];
  const int row = blockIdx.y, c = blockIdx.x;
  const int L = visible_length(p.q_pos, row, p.T);
  const int start = c * p.chunk;
  if (L <= p.K || start >= L) return;
  const int end = min(start + p.chunk, L);
  for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
  __syncthreads();
  hist_digit0(p.scores + (size_t)row * p.T, start, end, hist);
  __syncthreads();
  uint32_t *g = p.ghist + (size_t)row * 2 * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (hist[i]) atomicAdd(g + i, hist[i]);
}

// PASS 1: candidates above bin b0 and the digit-1 histogram of bin b0.
// PASS 2: candidates in bin b0 at or above sub-bin b1.
template <int PASS>
__global__ void __launch_bounds__(kThreads) topk_chunk_scan_kernel(const ChunkParams p) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint64_t staged[kBlockCand];
  __shared__ Scratch sc;
  const int row = blockIdx.y, c = blockIdx.x;
  const int L = visible_length(p.q_pos, row, p.T);
  const int start = c * p.chunk;
  if (L <= p.K || start >= L) return;
  const int end = min(start + p.chunk, L);
  const uint32_t *g0 = p.ghist + (size_t)row * 2 * kBins;
  uint32_t *g1 = p.ghist + (size_t)row * 2 * kBins + kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = g0[i];
  if (threadIdx.x == 0) sc.count = 0;
  __syncthreads();
  find_threshold_bin(hist, static_cast<uint32_t>(p.K), &sc);
  const uint32_t b0 = sc.result[0], need1 = sc.result[1];
  const bool whole = sc.result[1] == sc.result[2];
  if (PASS == 2 && whole) return;  // pass 1 already took bin b0 whole
  uint32_t b1 = 0;
  if (PASS == 1) {
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
  } else {
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = g1[i];
    __syncthreads();
    find_threshold_bin(hist, need1, &sc);
    b1 = sc.result[0];
  }
  __syncthreads();
  uint64_t *gdst = p.cand + (size_t)row * p.T;
  const Sink sink{staged, kBlockCand, gdst, p.gcount + row, static_cast<uint32_t>(p.T)};
  scan_row(p.scores + (size_t)row * p.T, start, end, PASS == 2, b0, whole, b1,
           (PASS == 1 && !whole) ? hist : nullptr, sink, &sc);
  __syncthreads();
  // one global append for the staged candidates of this block
  const uint32_t n = sc.count < static_cast<uint32_t>(kBlockCand) ? sc.count : static_cast<uint32_t>(kBlockCand);
  if (threadIdx.x == 0) sc.base = n ? atomicAdd(p.gcount + row, n) : 0u;
  if (PASS == 1 && !whole)
    for (int i = threadIdx.x; i < kBins; i += kThreads)
      if (hist[i]) atomicAdd(g1 + i, hist[i]);
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n; i += kThreads)
    if (sc.base + i < static_cast<uint32_t>(p.T)) gdst[sc.base + i] = staged[i];
}

__global__ void __launch_bounds__(kThreads) topk_chunk_select_kernel(const ChunkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ Scratch sc;
  const SmemViews s = smem_views(smem);
  const int row = blockIdx.x;
  const int L = visible_length(p.q_pos, row, p.T);
  int32_t *out = p.idx + (size_t)row * p.K;
  if (write_short_row(L, p.K, out)) return;
  uint32_t n = p.gcount[row];  // <= L: each visible position is appended at most once
  if (n > static_cast<uint32_t>(L)) {  // a corrupted counter: report it, never read past the row
    if (threadIdx.x == 0) raise_error(kErrDeviceCheck);
    n = static_cast<uint32_t>(L);
  }
  const uint64_t *gc = p.cand + (size_t)row * p.T;
  const uint64_t *src = gc;
  if (n <= static_cast<uint32_t>(kSmemCand)) {
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) s.cand[i] = gc[i];
    __syncthreads();
    src = s.cand;
  }
  const uint64_t tau = select_threshold(src, n, static_cast<uint32_t>(p.K), s.hist, &sc);
  write_sorted(src, n, tau, p.K, s.sortbuf, out, &sc);
}

}  // namespace topk
}  // namespace dsa
