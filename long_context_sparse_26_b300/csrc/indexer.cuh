// Lightning Indexer scores on the 5th-generation tensor cores.
//
// S[b,t,s] = sum_j w[b,t,j] * ReLU(q_I[b,t,j,:] . k_I[b,s,:]) for s <= pos(b,t)
// ("GLM-5.2 Explained: 1M Token Context AI Agent Model", §2.1, relevance score
// I_{t,s} = w . sigma(q_t^T h_s), read with sigma = ReLU per indexer head).
//
// One MMA tile puts 128 cached keys on M and the 64 heads of QG query tokens on
// N (N = 64*QG), K = the 128 indexer dims.  The fp32 tile lands in tensor
// memory with one key per TMEM lane, so the ReLU and the weighted head sum run
// inside one thread: no shuffles, no shared-memory round trip.
//
// Warp roles (one block per SM, persistent over a contiguous range of
// (sequence, query group, key tile) units):
//   warp 0     TMA producer: key tiles (two 64-dim halves, 128-byte swizzle)
//              into a ring of stages; the query-group operand once per group.
//   warp 1     allocates tensor memory and issues tcgen05.mma (one thread).
//   warps 2..  epilogue: tcgen05.ld of their 32 TMEM lanes, ReLU, weighted
//              head sum, one coalesced fp32 store per key and query.  Four
//              warps (one per TMEM lane quarter) for 1 or 2 queries per
//              group; eight for 4 queries (two per quarter, two queries each),
//              so that every scheduler interleaves two epilogue warps; eight
//              for one FP8 query too, whose units are two key tiles (two
//              warps per quarter, one tile each).
// Key tiles entirely after every query's position in the group are not
// loaded; the epilogue writes -inf there.
//
// With one query per sequence (decode), the epilogue can also count each
// visible score's top 13 key bits into a per-row histogram (the first step of
// the top-k selection), so the count costs no extra pass over the scores:
// the epilogue warps share one 8192-bin shared-memory histogram and add it
// to the global one when the block's sequence changes.  The flush is fenced
// on both sides by an mbarrier every epilogue warp arrives on (a bounded
// wait, so a block that gives up never strands a warp).  With several
// queries per group the same rounds guard the group's head weights, which
// the epilogue warps share.  (Counting there too was measured: those
// epilogues set the kernel's pace, and the count cost more than the
// top-k's histogram pass it saves.)
#pragma once

#include "common.cuh"

namespace dsa {
namespace indexer {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kTileKeys = 128;                     // UMMA M
// A key tile is 128 keys x 128 dims.  bf16: two 64-dim panels of 128-byte
// rows (16 KB each); FP8 (E4M3): one panel, a 128-dim row being 128 bytes.
// A unit of work (one pipeline stage, one accumulator slot) is kSub tiles.
// HIST (one query per group): the epilogue counts the top-k's digit-0
// histograms; a separate instantiation, so that calls without them pay
// nothing.
template <int QG, bool F8 = false, bool HIST = false>
struct Cfg {
  static constexpr int N = QG * kHeads;                 // UMMA N: 64, 128 or 256
  static constexpr int kPanels = F8 ? 1 : 2;            // 128-byte panels per row
  static constexpr int kPanelDims = F8 ? 128 : 64;      // dims per panel
  // FP8 decode: 256-key units, so that the single MMA-issuing thread's fixed
  // cost per unit (two barrier waits, two commits, the loop) is paid once per
  // 32 KB of keys, as it is for bf16; the two tiles of a unit go to two
  // epilogue warps per lane quarter
  static constexpr int kSub = (F8 && QG == 1) ? 2 : 1;
  static constexpr int kUnitKeys = kSub * kTileKeys;
  static constexpr int kPanelBytes = kUnitKeys * 128;   // one panel of a unit
  static constexpr int kABytes = kPanels * kPanelBytes; // per stage: 32 KB
  static constexpr int kHalfBBytes = N * 128;
  static constexpr int kBBytes = kPanels * kHalfBBytes;
  // (4 queries, bf16: two stages, measured faster than three or four; the
  // 256-column tile keeps the epilogue the slower side)
  static constexpr int kStages = F8 ? (QG == 1 ? 5 : 8) : (QG == 4 ? 2 : 5);
  // with 4 queries the two warps of a quarter split the queries
  static constexpr int kEpiWarps = (QG == 4 || kSub == 2) ? 8 : 4;
  static constexpr int kQPW = QG * 4 * kSub / kEpiWarps;  // queries per epilogue warp
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static_assert(!HIST || QG == 1, "histograms are counted for one query per group");
  static constexpr int kHistBytes = HIST ? 8192 * 4 : 0;  // the block's digit-0 histogram
  // FP8: each epilogue warp prefetches its keys' scales kScaleDepth units
  // ahead with cp.async, so the load latency never sits between a tile's
  // accumulator and its release
  static constexpr int kScaleDepth = 8;
  static constexpr int kScaleBytes = F8 ? kEpiWarps * kScaleDepth * 32 * 4 : 0;
  static constexpr int kAcc = QG == 4 ? 2 : 4;          // accumulator buffers in TMEM
  static constexpr int kTmemCols = (kAcc * kSub * N <= 256) ? 256 : 512;
  // head weights: one query, a copy per epilogue warp (in registers after
  // the load); several, one copy of the group's weights that the warps share
  static constexpr bool kWarpWeights = QG == 1;
  static constexpr int kWBytes = kWarpWeights ? kEpiWarps * kQPW * kHeads * 4 : QG * kHeads * 4;
  static constexpr int kSmall = 256 + kWBytes;            // barriers + flags, then the weights
  static constexpr int kSmemBytes = 1024 + kStages * kABytes + kBBytes + kSmall + kHistBytes + kScaleBytes;
  static constexpr int kKSteps = F8 ? kDim / 32 : kDim / 16;  // MMA instructions per tile
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  static_assert(kAcc * kSub * N <= kTmemCols, "accumulators must fit the allocation");
  static_assert((2 * kStages + 2 * kAcc + 4) * 8 + 8 <= 256, "barriers and flags fit their area");
};

struct Params {
  const float *w;        // [B, Q, 64]
  const int32_t *q_pos;  // [B, Q]
  float *scores;         // [B, Q, T]
  int B, Q, T;
  int ngroups;           // ceil(Q / QG)
  int ntiles;            // ceil(T / keys per unit): units of one (sequence, query group)
  long long units;       // B * ngroups * ntiles
  int stream_keys;       // 1: every key tile is read once (evict-first in L2)
  uint32_t *ghist;       // HIST only (Q == 1): [B][8192], each row's digit-0 histogram (added to)
  // paged key cache (block_table null: keys are [B, T, 128] contiguous):
  // position s of sequence b is row block_table[b][s / page_size] * page_size
  // + s % page_size of the [pages * page_size, 128] pool; page_size % 64 == 0
  const int32_t *block_table;  // [B, max_pages]
  int page_size, max_pages, num_pages;
  // FP8 caches only: row (b,s) of the key cache stands for k8 * k_scale[b*T+s]
  // (paged: the scales form a [pages, page_size] pool beside the code pool)
  // and head row (b,t,j) of the queries for q8 * q_scale[(b*Q+t)*64+j]
  const float *k_scale;
  const float *q_scale;
};

constexpr int kHistBins = 8192;          // digit 0 of the top-k: key bits 31..19
constexpr int kHistShift = 19;
constexpr int kHistRowStride = 8192;  // per-row words of the global histograms

// One round on `bar` (one arrival per epilogue warp): every warp's shared-
// memory reads and writes before it are visible to every warp after it.
// False if the block gave up.
__device__ __forceinline__ bool epi_round(int lane, uint64_t *bar, uint32_t &bar_phase, volatile int *abort) {
  __syncwarp();
  int ok = 1;
  if (lane == 0) {
    mbar_arrive(bar);
    ok = mbar_wait_bounded(bar, bar_phase, abort) ? 1 : 0;
  }
  bar_phase ^= 1u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Adds the block's histogram to row `row` of the global ones and clears it;
// epilogue warp e of NW takes every NW-th run of 32 bins.  Called between two
// rounds (no warp counts meanwhile).
template <int NW>
__device__ __forceinline__ void flush_hist(uint32_t *hist, uint32_t *ghist, size_t row, int e, int lane) {
  for (int i = e * 32 + lane; i < kHistBins; i += NW * 32) {
    const uint32_t c = hist[i];
    if (c == 0u) continue;
    hist[i] = 0u;
    atomicAdd(ghist + row * kHistRowStride + i, c);
  }
}

// Largest visible position of a query group (-1 if none), clamped to [-1, T-1].
template <int QG>
__device__ __forceinline__ int group_max_pos(const Params &p, int b, int q0) {
  int m = -1;
#pragma unroll
  for (int i = 0; i < QG; ++i) {
    if (q0 + i < p.Q) {
      int pos = __ldg(p.q_pos + (size_t)b * p.Q + q0 + i);
      pos = pos < 0 ? -1 : (pos >= p.T ? p.T - 1 : pos);
      m = pos > m ? pos : m;
    }
  }
  return m;
}

// Walks a block's units in order without a 64-bit division per unit: unit u
// is key tile `tile` of query group `g` of sequence `b`, seg = b * ngroups + g.
struct UnitCursor {
  long long u, seg;
  int tile, b, g;
  __device__ __forceinline__ UnitCursor(long long u0, const Params &p) : u(u0) {
    seg = u0 / p.ntiles;
    tile = static_cast<int>(u0 - seg * p.ntiles);
    b = static_cast<int>(seg / p.ngroups);
    g = static_cast<int>(seg - (long long)b * p.ngroups);
  }
  __device__ __forceinline__ void next(const Params &p) {
    ++u;
    if (++tile == p.ntiles) {
      tile = 0;
      ++seg;
      if (++g == p.ngroups) {
        g = 0;
        ++b;
      }
    }
  }
};

// PGS: FP8 key scales in a paged pool (located through the block table);
// a separate instantiation, so the contiguous FP8 epilogue pays nothing for it.
// HIST: p.ghist is non-null and receives the digit-0 histograms.
template <int QG, bool F8 = false, bool PGS = false, bool HIST = false>
__global__ void __launch_bounds__(Cfg<QG, F8, HIST>::kThreads, 1)
    indexer_scores_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                          const Params p) {
  using C = Cfg<QG, F8, HIST>;
  constexpr int kPanelBytes = C::kPanelBytes;
  constexpr int kABytes = C::kABytes;
  constexpr int kUnitKeys = C::kUnitKeys;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = base;                                   // [kStages][panels][kUnitKeys rows][128 B]
  uint8_t *sB = base + C::kStages * kABytes;            // [panels][N rows][128 B]
  uint8_t *small = sB + C::kBBytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(small);
  uint64_t *empty = full + C::kStages;
  uint64_t *tfull = empty + C::kStages;
  uint64_t *tempty = tfull + C::kAcc;
  uint64_t *bfull = tempty + C::kAcc;
  uint64_t *bfree = bfull + 1;
  uint64_t *mma_done = bfree + 1;
  uint64_t *hist_bar = mma_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(hist_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // one query: [epilogue warps][64], each warp's own copy of the head
  // weights; several: [QG][64], the group's weights shared by the warps
  float *sw_all = reinterpret_cast<float *>(small + 256);
  uint32_t *hist = reinterpret_cast<uint32_t *>(small + C::kSmall);  // HIST: [8192]
  // FP8: [epilogue warps][kScaleDepth][32] key scales in flight
  float *scale_ring = reinterpret_cast<float *>(small + C::kSmall + C::kHistBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const long long u_begin = p.units * blockIdx.x / gridDim.x;
  const long long u_end = p.units * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::kAcc; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], C::kEpiWarps);
    }
    mbar_init(bfull, 1);
    mbar_init(bfree, 1);
    mbar_init(mma_done, 1);
    mbar_init(hist_bar, C::kEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  if constexpr (HIST)
    for (int i = threadIdx.x; i < C::kHistBytes / 4; i += blockDim.x) hist[i] = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      long long cur_seg = -1;
      int seg_max = -1;
      uint32_t b_loads = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      for (UnitCursor c(u_begin, p); c.u < u_end && !*abort_flag; c.next(p)) {
        const long long seg = c.seg;
        const int tile = c.tile, b = c.b, q0 = c.g * QG;
        if (seg != cur_seg) seg_max = group_max_pos<QG>(p, b, q0);
        if (tile * kUnitKeys > seg_max) continue;  // fully masked unit: no load
        if (seg != cur_seg) {
          if (b_loads > 0 && !mbar_wait_bounded(bfree, (b_loads - 1) & 1u, abort_flag)) break;
          mbar_arrive_expect_tx(bfull, C::kBBytes);
          const int yq = (b * p.Q + q0) * kHeads;
#pragma unroll
          for (int h = 0; h < C::kPanels; ++h) tma_load_2d(sB + h * C::kHalfBBytes, &tmap_q, h * 64, yq, bfull);
          ++b_loads;
          cur_seg = seg;
        }
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&full[stage], kABytes);
        const int yk = b * p.T + tile * kUnitKeys;
        uint8_t *dst = sA + stage * kABytes;
        if (p.block_table != nullptr) {
          // 64-row boxes per panel, each located through the block table
          // (rows past T read page 0: the epilogue masks them; a page outside
          // the pool reads as zeros, TMA bounds every box)
#pragma unroll
          for (int r = 0; r < kUnitKeys / 64; ++r) {
            const int lrow = tile * kUnitKeys + 64 * r;
            const int page = lrow / p.page_size;
            int phys = lrow < p.T ? __ldg(p.block_table + (size_t)b * p.max_pages + page) : 0;
            if (phys < 0 || phys >= p.num_pages) {
              raise_error(kErrDeviceCheck);
              phys = 0;
            }
            const int y = phys * p.page_size + (lrow - page * p.page_size);
#pragma unroll
            for (int h = 0; h < C::kPanels; ++h)
              tma_load_2d_hint(dst + h * kPanelBytes + r * 64 * 128, &tmap_k, h * 64, y, &full[stage], policy);
          }
        } else {
          // 128-row boxes (the tensor map's), kSub per panel
#pragma unroll
          for (int t = 0; t < C::kSub; ++t)
#pragma unroll
            for (int h = 0; h < C::kPanels; ++h) {
              uint8_t *box = dst + h * kPanelBytes + t * kTileKeys * 128;
              if (p.stream_keys)
                tma_load_2d_hint(box, &tmap_k, h * 64, yk + t * kTileKeys, &full[stage], policy);
              else
                tma_load_2d(box, &tmap_k, h * 64, yk + t * kTileKeys, &full[stage]);
            }
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Every copy this block issued has landed before the block may exit.
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait_drain(&full[s], (issued_parity >> s) & 1u, kWaitLimitNs);
      if (b_loads > 0) mbar_wait_drain(bfull, (b_loads - 1) & 1u, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = F8 ? tc_idesc_e4m3(kTileKeys, C::N) : tc_idesc_bf16(kTileKeys, C::N);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      long long cur_seg = -1;
      int seg_max = -1;
      uint32_t b_waits = 0;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (UnitCursor c(u_begin, p); c.u < u_end && !*abort_flag; c.next(p)) {
        const long long seg = c.seg;
        const int tile = c.tile, b = c.b, q0 = c.g * QG;
        if (seg != cur_seg) seg_max = group_max_pos<QG>(p, b, q0);
        if (tile * kUnitKeys > seg_max) continue;
        if (seg != cur_seg) {
          if (b_waits > 0) tc_commit(bfree);  // previous group's operand is free once its MMAs finish
          if (!mbar_wait_bounded(bfull, b_waits & 1u, abort_flag)) break;
          ++b_waits;
          cur_seg = seg;
        }
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag)) break;
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) break;
        tc_fence_after();
        const uint32_t a_stage = a0 + stage * kABytes;
#pragma unroll
        for (int t = 0; t < C::kSub; ++t) {
          // tile t of the unit: its 128 rows into accumulator columns
          // (acc * kSub + t) * N
          const uint32_t d = tmem_base + static_cast<uint32_t>((acc * C::kSub + t) * C::N);
#pragma unroll
          for (int kk = 0; kk < C::kKSteps; ++kk) {
            // each K step is 32 bytes of a 128-byte swizzled row: 16 bf16 or 32 E4M3
            const uint32_t koff = (kk & 3) * 32u;
            const uint64_t ad = tc_desc_sw128(a_stage + (kk >> 2) * kPanelBytes + t * kTileKeys * 128 + koff);
            const uint64_t bd = tc_desc_sw128(b0 + (kk >> 2) * C::kHalfBBytes + koff);
            if constexpr (F8)
              tc_mma_f8(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
            else
              tc_mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(&empty[stage]);
        tc_commit(&tfull[acc]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++acc == C::kAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued by this thread are complete before tensor memory is freed.
      tc_commit(mma_done);
      mbar_wait_drain(mma_done, 0, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int QPW = C::kQPW;
    const int e = warp - 2;                        // epilogue warp index
    const int quarter = warp & 3;                  // TMEM lanes this warp may read
    // the two warps of a lane quarter split a unit's tiles (kSub = 2) or
    // the group's queries (4 queries)
    const int sub = C::kSub > 1 ? (e >> 2) : 0;               // tile of the unit this warp reads
    const int qb = C::kSub > 1 ? 0 : (e >> 2) * QPW;          // first query (within the group) of this warp
    const int key_off = sub * kTileKeys + quarter * 32 + lane;  // this lane's key within a unit
    float *sw = C::kWarpWeights ? sw_all + e * QPW * kHeads : sw_all + qb * kHeads;
    constexpr bool do_hist = HIST;
    uint32_t hist_phase = 0;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    long long cur_seg = -1;
    int seg_max = -1;
    int posv[QPW];
    float2 wreg[QG == 1 ? kHeads / 2 : 1];  // one query: its head weights live in registers
    int b = 0, q0 = 0;
    constexpr int kSD = C::kScaleDepth;
    const uint32_t ks_slot0 = smem_u32(scale_ring + e * kSD * 32 + lane);
    // FP8: one commit group per unit, issued kSD units ahead by a second
    // cursor (units past the range or keys past T copy nothing; the group is
    // still committed)
    UnitCursor pc(u_begin, p);
    auto prefetch_scale = [&]() {
      if (pc.u < u_end) {
        const int kk = pc.tile * kUnitKeys + key_off;
        if (kk < p.T) {
          // the key's scale: [B, T] contiguous, or a pool [pages, page_size]
          // beside the code pool, located through the same block table (a
          // page outside the pool reads page 0, as the codes do; the
          // producer reports it)
          size_t si = (size_t)pc.b * p.T + kk;
          if constexpr (PGS) {
            const int page = kk / p.page_size;
            int phys = __ldg(p.block_table + (size_t)pc.b * p.max_pages + page);
            phys = (phys < 0 || phys >= p.num_pages) ? 0 : phys;
            si = (size_t)phys * p.page_size + (kk - page * p.page_size);
          }
          cp_async_4(ks_slot0 + static_cast<uint32_t>((pc.u - u_begin) & (kSD - 1)) * 128u, p.k_scale + si);
        }
      }
      cp_async_commit();
      pc.next(p);
    };
    if constexpr (F8)
      for (int d = 0; d < kSD; ++d) prefetch_scale();
    for (UnitCursor c(u_begin, p); c.u < u_end; c.next(p)) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const long long u = c.u, seg = c.seg;
      const int tile = c.tile;
      if (seg != cur_seg) {
        // every warp is done with the previous group (its counts and, for
        // several queries, the shared weights) before anyone flushes or
        // reloads; for one query the rounds are needed only around a flush
        const bool rounds = QG > 1 || (do_hist && cur_seg >= 0);
        if (rounds && !epi_round(lane, hist_bar, hist_phase, abort_flag)) break;
        if (do_hist && cur_seg >= 0) flush_hist<C::kEpiWarps>(hist, p.ghist, b, e, lane);
        b = c.b;
        q0 = c.g * QG;
        seg_max = group_max_pos<QG>(p, b, q0);
        __syncwarp();  // the warp is done with the previous group's weights
        // the warp's own copy, or the group's QG x 64 weights loaded by the
        // warps between them
        constexpr bool kWW = C::kWarpWeights;
        const int w_first = kWW ? lane : e * 32 + lane;
        const int w_step = kWW ? 32 : C::kEpiWarps * 32;
        const int w_count = kWW ? QPW * kHeads : QG * kHeads;
        const int w_q0 = kWW ? q0 + qb : q0;
        float *w_dst = kWW ? sw : sw_all;
        for (int i = w_first; i < w_count; i += w_step) {
          const int q = w_q0 + i / kHeads;
          const size_t wi = ((size_t)b * p.Q + q) * kHeads + (i % kHeads);
          // FP8: the query head's scale folds into its weight (scales are
          // positive, so they pass through the ReLU)
          w_dst[i] = q < p.Q ? __ldg(p.w + wi) * (F8 ? __ldg(p.q_scale + wi) : 1.0f) : 0.0f;
        }
        if (rounds && !epi_round(lane, hist_bar, hist_phase, abort_flag)) break;
#pragma unroll
        for (int i = 0; i < QPW; ++i) {
          const int q = q0 + qb + i;
          int pos = (q < p.Q) ? __ldg(p.q_pos + (size_t)b * p.Q + q) : -1;
          if (q < p.Q && (pos < 0 || pos >= p.T) && lane == 0 && tile == 0) raise_error(kErrDeviceCheck);
          posv[i] = pos < 0 ? -1 : (pos >= p.T ? p.T - 1 : pos);
        }
        __syncwarp();
        if constexpr (QG == 1) {
#pragma unroll
          for (int j = 0; j < kHeads / 2; ++j) wreg[j] = reinterpret_cast<const float2 *>(sw)[j];
        }
        cur_seg = seg;
      }
      const int key = tile * kUnitKeys + key_off;
      const bool real = tile * kUnitKeys <= seg_max;
      if (real) {
        // One lane polls; the verdict is shared so the whole warp either
        // proceeds to the warp-collective TMEM loads or leaves together.
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
      }
      float kscale = 1.0f;
      if constexpr (F8) {
        cp_async_wait<kSD - 1>();  // this unit's group has landed
        kscale = scale_ring[(e * kSD + ((u - u_begin) & (kSD - 1))) * 32 + lane];
      }
#pragma unroll
      for (int i = 0; i < QPW; ++i) {
        if (q0 + qb + i >= p.Q) break;
        float s = 0.0f;
        if (real) {
          // both 32-column halves of the query's 64 heads, one wait
          const uint32_t taddr =
              tmem_base + lane_addr + static_cast<uint32_t>((acc * C::kSub + sub) * C::N + (qb + i) * kHeads);
          const float4 *w4 = reinterpret_cast<const float4 *>(sw + i * kHeads);
          if constexpr (QG == 1) {
            // decode: each 32-column half is loaded and reduced in turn, two
            // heads per paired FMA against the weights held in registers
            // (the epilogue's instruction count sets the pace for FP8 keys)
            float v[32];
            float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tmem_ld_32x32b_x32(taddr + h * 32, v);
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                a0 = ffma2(make_float2(fmaxf(v[j + 0], 0.0f), fmaxf(v[j + 1], 0.0f)), wreg[(h * 32 + j) >> 1], a0);
                a1 = ffma2(make_float2(fmaxf(v[j + 2], 0.0f), fmaxf(v[j + 3], 0.0f)), wreg[((h * 32 + j) >> 1) + 1], a1);
              }
            }
            s = (a0.x + a0.y) + (a1.x + a1.y);
          } else {
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32_nowait(taddr, v0);
            tmem_ld_32x32b_x32_nowait(taddr + 32, v1);
            tmem_wait_ld();
            // four independent chains of paired FMAs (two heads each)
            float2 a[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              const float4 wv = w4[j >> 2];
              const uint32_t *v = j < 32 ? v0 + j : v1 + (j - 32);
              const int c = (j >> 2) & 1;
              a[2 * c] = ffma2(make_float2(fmaxf(__uint_as_float(v[0]), 0.0f), fmaxf(__uint_as_float(v[1]), 0.0f)),
                               make_float2(wv.x, wv.y), a[2 * c]);
              a[2 * c + 1] = ffma2(make_float2(fmaxf(__uint_as_float(v[2]), 0.0f), fmaxf(__uint_as_float(v[3]), 0.0f)),
                                   make_float2(wv.z, wv.w), a[2 * c + 1]);
            }
            s = ((a[0].x + a[0].y) + (a[1].x + a[1].y)) + ((a[2].x + a[2].y) + (a[3].x + a[3].y));
          }
        }
        if (F8 && real && key < p.T) s *= kscale;
        if (key < p.T) {
          float *row = p.scores + ((size_t)b * p.Q + q0 + qb + i) * (size_t)p.T;
          const bool vis = real && key <= posv[i];
          row[key] = vis ? s : -INFINITY;
          // (measured: this inline count beats one deferred past the store)
          if constexpr (HIST)
            if (vis) atomicAdd(&hist[score_key(s) >> kHistShift], 1u);
        }
      }
      if (real) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        if (++acc == C::kAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // the slot just read is refilled (the read above has been consumed)
      if constexpr (F8) prefetch_scale();
    }
    if constexpr (F8) asm volatile("cp.async.wait_all;" ::: "memory");
    if (do_hist && cur_seg >= 0 && !*abort_flag && epi_round(lane, hist_bar, hist_phase, abort_flag))
      flush_hist<C::kEpiWarps>(hist, p.ghist, b, e, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace indexer
}  // namespace dsa
