// Sparse absorbed-MLA attention on the 5th-generation tensor cores.
//
// For one query token and one layer: z[h, j] = sm_scale * q[h, :] . kv[idx[j], :]
// over 576-dim cached rows (512 compressed-KV dims, then 64 rotated RoPE dims),
// p = softmax_j(z), O[h, :] = sum_j p[h, j] * kv[idx[j], :512]: the value is the
// leading kv_lora_rank dims of the same row ("GLM-5.2 Explained: 1M Token
// Context AI Agent Model", §2.1: K/V are loaded only for the selected
// positions; §1.1: MLA is kept; kv_lora_rank = 512 in the GLM-5.2 config of
// "GLM-5.2核心技术解析：IndexShare架构与MTP层优化详解"; 64 heads).
//
// Block = (layer, split, query row): it walks kKeys-key windows of its slice
// of the index set through a ring of two window slots.  A slot is nine
// 64-dim panels x 64 rows x 128 B in the 128-byte-swizzled layout the tensor
// cores read, and it moves in five panel groups: group g < 4 is panels 2g and
// 2g+1 (dims 128g..128g+127), group 4 the RoPE panel 8.  Per window:
//   gather  the selected latent rows, group by group, by 16-byte cp.async
//           copies from the producer warps (unused slots zero-filled); a
//           group of the next window is gathered as soon as the window two
//           back has released it, so gathers overlap the tail of GEMM 2;
//   GEMM 1  S[64 heads, kKeys] = Q . K^T  tcgen05, M = 64, N = kKeys, K = 576
//           (Q: nine TMA-loaded panels, resident for the whole block),
//           consumed group by group as the groups land, so the MMAs overlap
//           the rest of the gather;
//   softmax two threads per head (one per 32 keys) read the head's S row from
//           tensor memory: masked, scaled (log2 e folded in), exponentiated
//           against a per-head reference max, summed, and written as bf16
//           P^T rows into the window's RoPE panel (dead once GEMM 1 has read
//           it);
//   GEMM 2  O^T[512 dims, 64 heads] += V^T . P^T  tcgen05, M = 128 (4 chunks of
//           128 dims), N = 64, K = kKeys, from a thread of its own; V^T is read
//           from the gathered panels as an MN-major operand (no transpose
//           pass); chunk c releases group c of the slot as it completes, the
//           last chunk also group 4 (which held P).
// The reference max only moves when a head's tile max exceeds it by more than
// 2^8 (log2 units); then the block rescales that head's O^T column and its
// running sum before that window's GEMM 2.  Anything in between stays within
// fp32 range, and the final O / l is the same for every choice of reference.
//
// Warp roles (one block per SM):
//   producers  9 warps (bf16 rows) or 5 (FP8 rows): rows w, w + P, ... of
//              every window; warp 0 also loads the query panels by TMA;
//   GEMM 1     two warps, one issuing thread each, on alternate panel groups
//              into two partial S tiles (the first also allocates tensor
//              memory); GEMM 2 a third: one thread issues these small MMAs at
//              about half the rate the tensor pipe takes them, two or three
//              keep it fed;
//   last 4     softmax and O^T rescale; warp w owns TMEM lanes
//              32*(w%4)..+31: heads 16*(w%4)..+15 of S (an M = 64 result
//              sits in lanes 0-15 of each 32-lane quarter; both half-warps
//              read them, 32 columns each) and dims 128c + 32*(w%4)..+31 of
//              O^T chunk c.
// Tensor memory: O^T in columns 0-255 (chunk c at 64c); the two S partials in
// two window buffers of kKeys columns each, from 256 and from 384.
// Every warp of the block writes the result, one 128-dim chunk of O^T for
// its lane quarter, straight from tensor memory (lane = dim, so each head's
// stores from a warp are 32 consecutive dims): bf16 and normalised when the
// block's (layer, row) is one split, else the unnormalised fp32 partial plus
// (reference max, sum) per head for the combine kernel.
#pragma once

#include "common.cuh"
#include "sparse_mla.cuh"

namespace dsa {
namespace mla {

using attn::kMaxLayers;
using attn::Params;

constexpr int kH = 64;
constexpr int kDv = 512;
constexpr int kKeys = 64;                            // keys per window (GEMM 1 N, GEMM 2 K)
constexpr int kWindows = 2;                          // window slots in the ring
constexpr int kRingRows = kWindows * kKeys;          // 128
constexpr int kPanels = 9;                           // 576 dims / 64
constexpr int kGroups = 5;                           // panel groups of a window slot
constexpr int kPanelBytes = kRingRows * 128;         // one 64-dim panel of the ring: 16 KB
constexpr int kRingBytes = kPanels * kPanelBytes;    // 147456
constexpr int kQBytes = kPanels * kH * 128;          // 73728
// Warp roles: the producers, then the three MMA-issuing warps, then four
// softmax warps.  bf16 rows: nine producer warps (random 1152-byte rows are
// gathered faster the more warps issue the copies: 2.9 TB/s from five warps,
// 4.6 TB/s from nine, measured on a B300); FP8 rows: five (their
// dequantisation needs the registers of a 384-thread block).
template <bool F8KV>
struct Roles {
  static constexpr int kProducerWarps = F8KV ? 5 : 9;
  static constexpr int kMmaWarp = kProducerWarps;           // tensor-memory allocation, GEMM 1 on groups 0, 2, 4
  static constexpr int kMma1bWarp = kProducerWarps + 1;     // GEMM 1 on groups 1, 3
  static constexpr int kGemm2Warp = kProducerWarps + 2;     // GEMM 2 issue
  static constexpr int kSoftmaxWarp0 = kProducerWarps + 3;  // four softmax warps, one per TMEM lane quarter
  static constexpr int kThreads = 32 * (kProducerWarps + 3 + 4);
  static constexpr int kRowsPerWarp = (kKeys + kProducerWarps - 1) / kProducerWarps;  // rows of a window per producer warp
  static constexpr int kPatA = (kRowsPerWarp + 1) / 2;      // copy instructions of a two-panel group (two rows each)
  static constexpr int kPatB = (kRowsPerWarp + 3) / 4;      // copy instructions of the RoPE panel (four rows each)
  static_assert(kSoftmaxWarp0 % 4 == 0, "softmax warp w reads TMEM lane quarter w % 4");
};
constexpr int kMaxProducerWarps = 9;
// FP8 latent rows are gathered and converted in stages of 32 rows, two per window
constexpr int kStageRows = 32;
constexpr int kStages = kRingRows / kStageRows;      // 4
constexpr int kWinStages = kKeys / kStageRows;       // 2
constexpr int kHalves = kKeys / 32;                  // 32-column TMEM loads per S row
constexpr int kTmemCols = 512;
constexpr int kOCol = 0;
constexpr int kSCol = 256;                           // S partial of groups 0, 2, 4; two window buffers
constexpr int kSColB = 384;                          // S partial of groups 1, 3; two window buffers
constexpr int kSmallBytes = 4096;
constexpr int kSmemBytes = 1024 + kQBytes + kRingBytes + kSmallBytes;
static_assert(kSmemBytes <= 232448, "shared memory per block");
static_assert(kRingBytes >= kH * kDv * 4, "the epilogue stages an fp32 partial in the gather ring");
static_assert(kKeys % kStageRows == 0 && kKeys % 32 == 0 && kKeys == 64, "windows of 64 keys");
static_assert(kSColB + 2 * kKeys <= kTmemCols && kSCol + 2 * kKeys <= kSColB, "S partials fit the allocation");
constexpr float kRescaleLog2 = 8.0f;                 // rescale when the max grows by > 2^8

struct Maps {
  CUtensorMap q[kMaxLayers];   // [rows*64, 576] bf16, box 64 x 64, 128-byte swizzle
};

// Instruction descriptor, kind::f16, fp32 accumulate, bf16 operands.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn_major ? (1u << 15) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory descriptor of a 128-byte-swizzled operand.  K-major: rows of
// 128 B (64 K-elements), 8-row groups `sbo` bytes apart.  MN-major: 64
// MN-elements per 128-byte row, the next 64 MN-elements `lbo` bytes on, K rows
// 128 B apart in 8-row groups `sbo` bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The mbarrier receives one arrival (no pending-count increment) once every
// cp.async this thread issued before has landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Thread-block clusters: a barrier over every thread of every CTA of the
// cluster (arrive with release, wait with acquire), and loads from another
// CTA's shared memory at the address a local one maps to.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by the MUFU approximation (ex2.approx.ftz.f32: 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Lanes 0-15 of the warp's quarter, twice: threads 0-15 get lane t, columns
// [taddr, taddr + 32); threads 16-31 get lane t - 16, columns [taddr + 32,
// taddr + 64) (16x32bx2 shape, half-split offset 32 columns).  Not waited.
__device__ __forceinline__ void tmem_ld_16x32bx2_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], 32;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 8 columns, load (waited) and store.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Warp-uniform bounded wait: lane 0 polls, the verdict goes to every lane.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Raw content of index slot `slot` of a row (-1 past k).  The load is only
// issued here; nothing reads the value until checked_pos, tiles later.
__device__ __forceinline__ int slot_raw(const int32_t *irow, int slot, int K) {
  return slot < K ? __ldg(irow + slot) : -1;
}
// The position a raw slot names, or -1 when unused or out of range (an
// out-of-range index is reported when `report`).
__device__ __forceinline__ int checked_pos(int raw, int T, bool report) {
  if (raw < -1 || raw >= T) {
    if (report) raise_error(kErrDeviceCheck);
    return -1;
  }
  return raw;
}

constexpr int kMaxClusterSplits = 8;

struct Small {
  alignas(16) float xa[2][kH];    // per-head rescale factors (1/l for the epilogue)
  alignas(16) float cml[kH][2];   // cluster launch: this split's (reference max, sum) per head
  alignas(16) float cw[kH][kMaxClusterSplits];  // cluster launch: each split's weight in the merge, per head
  float cinv[kH];                 // cluster launch: 1 / the merged sum, per head
  uint64_t full[kWindows][kGroups];   // a group of a window slot has landed (producer arrivals)
  uint64_t empty[kWindows][kGroups];  // a group of a window slot is free (GEMM 2 commits)
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full;                // every softmax warp has written its P rows and its flags
  uint64_t p_free;                // GEMM 2 of the window has completed
  uint64_t resc_done;             // every softmax warp has rescaled its O^T lanes
  uint64_t q_full;
  uint64_t mma_done;
  uint64_t mma1b_done;
  uint64_t mma2_done;
  uint64_t staged[kMaxProducerWarps][kStages];  // FP8 latent rows: a warp's copies of a stage have landed
  uint32_t tmem_slot;
  int abort;
  int status[2][4];               // per softmax warp, per window parity: 1 = ok
  int need[2][4];                 // per softmax warp: a head of it moves its reference max
};
static_assert(sizeof(Small) <= kSmallBytes, "small shared region");

// 16 E4M3 codes times their scale, rounded to bf16, packed in dim order.
__device__ __forceinline__ void dequant16(const uint4 &code, float scale, uint32_t (&out)[8]) {
  const uint32_t w[4] = {code.x, code.y, code.z, code.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu);
      const __half2 v = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));  // low byte -> .x
      const float2 f = __half22float2(v);
      out[2 * i + h] = pack_bf16x2(f.x * scale, f.y * scale);
    }
  }
}

template <bool F8KV>
__global__ void __launch_bounds__(Roles<F8KV>::kThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
  using R = Roles<F8KV>;
  constexpr int kProducerWarps = R::kProducerWarps, kMmaWarp = R::kMmaWarp, kMma1bWarp = R::kMma1bWarp;
  constexpr int kGemm2Warp = R::kGemm2Warp, kSoftmaxWarp0 = R::kSoftmaxWarp0;
  constexpr int kRowsPerWarp = R::kRowsPerWarp, kPatA = R::kPatA, kPatB = R::kPatB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = base;                                  // [9 panels][64 heads][128 B]
  uint8_t *sK = sQ + kQBytes;                          // [9 panels][128 ring rows][128 B]
  Small *sm = reinterpret_cast<Small *>(sK + kRingBytes);
  volatile int *abort_flag = &sm->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // this block's (layer, row) unit, its split and the windows per split;
  // unit u is layer u % n_layers of row u / n_layers.  Units from tail_base
  // on (the last, partial wave of a launch with one split per unit) take
  // tail_nsplit splits.  `tile` indexes the block's fp32 partial.
  const int nl = p.n_layers;
  int layer_, split_, row_, bps_, nsplit_;
  size_t tile_;
  if (p.cluster) {
    // the splits of a unit are consecutive blocks (one cluster); tile unused
    split_ = blockIdx.x % p.nsplit;
    const int u = blockIdx.x / p.nsplit;
    layer_ = u % nl;
    row_ = u / nl;
    bps_ = p.blocks_per_split;
    nsplit_ = p.nsplit;
    tile_ = 0;
  } else if (p.tail_nsplit > 0 && static_cast<int>(blockIdx.x) >= p.tail_base) {
    const int t = static_cast<int>(blockIdx.x) - p.tail_base, tu = t / p.tail_nsplit;
    const int u = p.tail_base + tu;
    split_ = t - tu * p.tail_nsplit;
    layer_ = u % nl;
    row_ = u / nl;
    bps_ = p.tail_bps;
    nsplit_ = p.tail_nsplit;
    tile_ = (size_t)tu * p.tail_nsplit + split_;
  } else {
    layer_ = blockIdx.x % nl;
    const int rest = blockIdx.x / nl;
    split_ = rest % p.nsplit;
    row_ = rest / p.nsplit;
    bps_ = p.blocks_per_split;
    nsplit_ = p.nsplit;
    tile_ = ((size_t)layer_ * p.rows + row_) * p.nsplit + split_;
  }
  const int layer = layer_, split = split_, row = row_, unit_splits = nsplit_;
  const size_t tile = tile_;
  const int b = row / p.Q;
  const int slot0 = split * bps_ * kKeys;
  int nblk = bps_;
  {
    const int remaining = (p.K - slot0 + kKeys - 1) / kKeys;
    nblk = remaining < nblk ? remaining : nblk;
    if (nblk < 0) nblk = 0;
  }
  const int32_t *irow = p.idx + (size_t)row * p.K;

  if (threadIdx.x == 0) {
    for (int w = 0; w < kWindows; ++w)
      for (int g = 0; g < kGroups; ++g) {
        mbar_init(&sm->full[w][g], 32 * kProducerWarps);
        mbar_init(&sm->empty[w][g], 1);
      }
    for (int i = 0; i < kStages; ++i)
      for (int w = 0; w < kProducerWarps; ++w) mbar_init(&sm->staged[w][i], 32);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm->s_full[i], 2);  // both GEMM 1 issuers commit
      mbar_init(&sm->s_empty[i], 4);
    }
    mbar_init(&sm->p_full, 4);
    mbar_init(&sm->p_free, 1);
    mbar_init(&sm->resc_done, 4);
    mbar_init(&sm->q_full, 1);
    mbar_init(&sm->mma_done, 1);
    mbar_init(&sm->mma1b_done, 1);
    mbar_init(&sm->mma2_done, 1);
    sm->abort = 0;
    fence_mbar_init();
    // the query panels are an input of this call, not of the kernel before:
    // they load while that kernel may still be running (dependent launch)
    if (nblk > 0) {
      prefetch_tensormap(&maps.q[layer]);
      mbar_arrive_expect_tx(&sm->q_full, kQBytes);
      for (int pp = 0; pp < kPanels; ++pp)
        tma_load_2d(sQ + pp * kH * 128, &maps.q[layer], pp * 64, row * kH, &sm->q_full);
    }
  }
  if (warp == kMmaWarp) tmem_alloc(&sm->tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_slot;
  // launched as a dependent of the kernel that writes the index set (the
  // top-k select): nothing below reads idx before that kernel has completed
  // and its writes are visible (a no-op without such a dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------ producers
    const bool q_issued = warp == 0 && nblk > 0;  // thread 0 issued the query panels
    const bool paged = p.block_table != nullptr;
    constexpr size_t kRowBytes = F8KV ? attn::kF8RowBytes : (kDv + 64) * 2;
    const uint8_t *kvb = reinterpret_cast<const uint8_t *>(p.kv[layer]) + (paged ? 0 : (size_t)b * p.T * kRowBytes);
    // row of kvb holding position pos (-1: none); the block-table load is
    // issued a window before the row is used
    auto row_of = [&](int pos) -> int {
      if (pos < 0 || !paged) return pos;
      const int page = pos / p.page_size;
      const int phys = __ldg(p.block_table + (size_t)b * p.max_pages + page);
      if (phys < 0 || phys >= p.num_pages) {
        if (warp == 0) raise_error(kErrDeviceCheck);
        return -1;
      }
      return phys * p.page_size + (pos - page * p.page_size);
    };
    const uint32_t k0 = smem_u32(sK);
    if constexpr (!F8KV) {
      // lane l holds index slots l and l + 32 of a window: the raw slots two
      // windows ahead, their cache rows one window ahead
      auto slot_of = [&](int jj, int half) -> int {
        return jj < nblk ? slot_raw(irow, slot0 + jj * kKeys + half * 32 + lane, p.K) : -1;
      };
      int raw1_lo = slot_of(1, 0), raw1_hi = slot_of(1, 1);
      int raw2_lo = slot_of(2, 0), raw2_hi = slot_of(2, 1);
      int nxt_lo = row_of(checked_pos(slot_of(0, 0), p.T, warp == 0));
      int nxt_hi = row_of(checked_pos(slot_of(0, 1), p.T, warp == 0));
      bool stop = false;
      for (int jj = 0; jj < nblk && !stop; ++jj) {
        const int cur_lo = nxt_lo, cur_hi = nxt_hi;
        nxt_lo = row_of(checked_pos(raw1_lo, p.T, warp == 0));
        nxt_hi = row_of(checked_pos(raw1_hi, p.T, warp == 0));
        raw1_lo = raw2_lo;
        raw1_hi = raw2_hi;
        raw2_lo = slot_of(jj + 3, 0);
        raw2_hi = slot_of(jj + 3, 1);
        const int w = jj % kWindows;
        const uint32_t ph = static_cast<uint32_t>(jj / kWindows) & 1u;
        // this warp owns window rows warp + 5k.  Copy pattern A (a two-panel
        // group, 16 chunks a row) covers two rows an instruction, lane l
        // taking row k = 2i + l/16; pattern B (the RoPE panel, 8 chunks a
        // row) four rows, k = 4i + l/8.  Per lane: the cache row of each
        // instruction and its ring row (-1: no such row in the window)
        int posA[kPatA], ringA[kPatA], posB[kPatB], ringB[kPatB];
#pragma unroll
        for (int i = 0; i < kPatA; ++i) {
          const int k = 2 * i + (lane >> 4);
          const int r = warp + kProducerWarps * k;
          const int vlo = __shfl_sync(0xffffffffu, cur_lo, r & 31);
          const int vhi = __shfl_sync(0xffffffffu, cur_hi, r & 31);
          posA[i] = r < 32 ? vlo : vhi;
          ringA[i] = (k < kRowsPerWarp && r < kKeys) ? w * kKeys + r : -1;
        }
#pragma unroll
        for (int i = 0; i < kPatB; ++i) {
          const int k = 4 * i + (lane >> 3);
          const int r = warp + kProducerWarps * k;
          const int vlo = __shfl_sync(0xffffffffu, cur_lo, r & 31);
          const int vhi = __shfl_sync(0xffffffffu, cur_hi, r & 31);
          posB[i] = r < 32 ? vlo : vhi;
          ringB[i] = (k < kRowsPerWarp && r < kKeys) ? w * kKeys + r : -1;
        }
        for (int gi = 0; gi < kGroups; ++gi) {
          if (!warp_wait(&sm->empty[w][gi], ph ^ 1u, abort_flag)) {
            stop = true;
            break;
          }
          if (gi < kGroups - 1) {
            // panels 2gi and 2gi + 1: bytes 256 gi .. 256 gi + 255 of the row
            const int c = lane & 15;
            const uint32_t pbase = k0 + (2 * gi + (c >> 3)) * kPanelBytes;
#pragma unroll
            for (int i = 0; i < kPatA; ++i) {
              if (ringA[i] >= 0) {
                const int pos = posA[i];
                const uint8_t *src = kvb + (size_t)(pos < 0 ? 0 : pos) * kRowBytes + gi * 256 + c * 16;
                cp_async_16(pbase + ringA[i] * 128 + (((c & 7) ^ (ringA[i] & 7)) << 4), src, pos < 0 ? 0u : 16u);
              }
            }
          } else {
            // panel 8 (RoPE): bytes 1024 .. 1151 of the row
            const int c = lane & 7;
            const uint32_t pbase = k0 + 8 * kPanelBytes;
#pragma unroll
            for (int i = 0; i < kPatB; ++i) {
              if (ringB[i] >= 0) {
                const int pos = posB[i];
                const uint8_t *src = kvb + (size_t)(pos < 0 ? 0 : pos) * kRowBytes + 1024 + c * 16;
                cp_async_16(pbase + ringB[i] * 128 + ((c ^ (ringB[i] & 7)) << 4), src, pos < 0 ? 0u : 16u);
              }
            }
          }
          cp_async_mbar_arrive(&sm->full[w][gi]);
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
      // FP8 latent rows, dequantised in shared memory, in stages of 32 rows
      // (stage i holds index slots 32i..32i+31 in ring rows 32 (i % 4) ..:
      // window i / 2 in slot (i / 2) % 2).  A warp owns rows warp, warp + 5,
      // ... of every stage.  Each 656-byte row first lands by cp.async in its
      // own ring lines (41 16-byte chunks: chunk c in panel c / 8, slot c % 8,
      // unswizzled), tracked by the warp's own mbarrier per stage; then the
      // warp reads its rows back, syncs, and writes the bf16 row over the same
      // lines in the swizzled operand layout.  Only the owning warp touches a
      // row's lines, so a warp sync orders the reads before the writes.  The
      // warp interleaves issuing copies (once every group of the window's
      // slot is free) with converting stages whose copies landed, so several
      // stages stay in flight; a window's groups are released to GEMM 1 once
      // both of its stages are converted.
      constexpr int kRPW = (kStageRows + kProducerWarps - 1) / kProducerWarps;  // rows per warp and stage
      const int nstage = nblk * kWinStages;
      auto load_slot = [&](int g) -> int { return g < nstage ? slot_raw(irow, slot0 + g * kStageRows + lane, p.K) : -1; };
      // rows of stage i (per lane: slot i*32 + lane), slot loads one issue ahead
      int raw_cur = load_slot(0), raw_next = load_slot(1);
      auto issue = [&](int i) {
        const int rows_i = row_of(checked_pos(raw_cur, p.T, warp == 0));
        raw_cur = raw_next;
        raw_next = load_slot(i + 2);
        const uint32_t sbase = k0 + (i % kStages) * kStageRows * 128;
#pragma unroll
        for (int j = 0; j < kRPW; ++j) {
          const int r = warp + kProducerWarps * j;
          if (r < kStageRows) {
            const int pos = __shfl_sync(0xffffffffu, rows_i, r);
            const uint8_t *src = kvb + (size_t)(pos < 0 ? 0 : pos) * kRowBytes;
            const uint32_t nbytes = pos < 0 ? 0u : 16u;  // unused slot: a zero row
            const uint32_t rbase = sbase + r * 128;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c = lane + 32 * cc;  // chunk of the 656-byte row
              if (c < attn::kF8RowBytes / 16) cp_async_16(rbase + (c >> 3) * kPanelBytes + (c & 7) * 16, src + c * 16, nbytes);
            }
          }
        }
        cp_async_mbar_arrive(&sm->staged[warp][i % kStages]);
      };
      auto convert = [&](int i) {
        const uint32_t sbase = k0 + (i % kStages) * kStageRows * 128;
        uint4 code[kRPW], rope[kRPW];
        float scale[kRPW];
#pragma unroll
        for (int j = 0; j < kRPW; ++j) {
          const int r = warp + kProducerWarps * j;
          if (r < kStageRows) {
            const uint32_t rbase = sbase + r * 128;
            // code chunk lane; scale chunk 32 (panel 4, slot 0); RoPE chunks 33..40
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(code[j].x), "=r"(code[j].y), "=r"(code[j].z), "=r"(code[j].w)
                         : "r"(rbase + (lane >> 3) * kPanelBytes + (lane & 7) * 16));
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(scale[j]) : "r"(rbase + 4 * kPanelBytes + 4 * (lane >> 3)));
            const int rc = 33 + (lane & 7);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(rope[j].x), "=r"(rope[j].y), "=r"(rope[j].z), "=r"(rope[j].w)
                         : "r"(rbase + (rc >> 3) * kPanelBytes + (rc & 7) * 16));
          }
        }
        __syncwarp();  // every lane has read its rows' staged bytes
#pragma unroll
        for (int j = 0; j < kRPW; ++j) {
          const int r = warp + kProducerWarps * j;
          if (r < kStageRows) {
            const uint32_t rbase = sbase + r * 128;  // ring row s*32 + r; (s*32 + r) % 8 == r % 8
            uint32_t v[8];
            dequant16(code[j], scale[j], v);
            // dims 16*lane..+15: panel lane/4, 16-byte chunks 2*(lane%4) and +1
            const uint32_t pb = rbase + (lane >> 2) * kPanelBytes;
            const int c0 = 2 * (lane & 3);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pb + (((c0 ^ r) & 7) << 4)), "r"(v[0]),
                         "r"(v[1]), "r"(v[2]), "r"(v[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pb + ((((c0 + 1) ^ r) & 7) << 4)),
                         "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                         : "memory");
            if (lane < 8)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rbase + 8 * kPanelBytes +
                                                                             (((lane ^ r) & 7) << 4)),
                           "r"(rope[j].x), "r"(rope[j].y), "r"(rope[j].z), "r"(rope[j].w)
                           : "memory");
          }
        }
        fence_proxy_async_smem();
        if (i % kWinStages == kWinStages - 1)
          for (int g = 0; g < kGroups; ++g) mbar_arrive(&sm->full[(i / kWinStages) % kWindows][g]);
      };
      int issued = 0, conv = 0;
      unsigned long long t_idle = 0;
      while (conv < nstage) {
        bool prog = false;
        if (issued < nstage) {
          int ok = 1;
          if (issued % kWinStages == 0) {
            // the first stage of a window waits for every group of its slot
            const int wv = issued / kWinStages;
            const uint32_t ph = static_cast<uint32_t>(wv / kWindows) & 1u;
            if (lane == 0)
              for (int g = 0; g < kGroups; ++g) ok &= mbar_try_wait(&sm->empty[wv % kWindows][g], ph ^ 1u) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
          }
          if (ok) {
            issue(issued);
            ++issued;
            prog = true;
          }
        }
        if (conv < issued) {
          const uint32_t ph = static_cast<uint32_t>(conv / kStages) & 1u;
          int ok = lane == 0 ? (mbar_try_wait(&sm->staged[warp][conv % kStages], ph) ? 1 : 0) : 0;
          if (__shfl_sync(0xffffffffu, ok, 0)) {
            convert(conv);
            ++conv;
            prog = true;
          }
        }
        if (prog) {
          t_idle = 0;
        } else {
          int stop = 0;
          if (lane == 0) {
            const unsigned long long now = global_timer_ns();
            if (t_idle == 0) {
              t_idle = now;
            } else if (*abort_flag) {
              stop = 1;
            } else if (now - t_idle > wait_limit_ns()) {
              raise_error(kErrTimeout);
              *abort_flag = 1;
              stop = 1;
            }
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
    if (q_issued && lane == 0) mbar_wait_drain(&sm->q_full, 0, kWaitLimitNs);
  } else if (warp == kMmaWarp || warp == kMma1bWarp) {
    // ------------------------------------------------------------ GEMM 1 issuers
    // Two threads share GEMM 1 (one thread issues these small MMAs at about
    // half the rate the tensor pipe takes them): the MMA warp on groups 0, 2
    // and 4 into the S partial at kSCol, the next warp on groups 1 and 3 into
    // the one at kSColB; the softmax adds the two.
    const bool part_a = warp == kMmaWarp;
    if (lane == 0 && nblk > 0) {
      constexpr uint32_t id1 = idesc(64, kKeys, false, false);
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK);
      bool ok = mbar_wait_bounded(&sm->q_full, 0, abort_flag);
      // GEMM 1 of each window in order, once its S buffer is free, group by
      // group as the groups land
      for (int g1 = 0; ok && g1 < nblk; ++g1) {
        const int w = g1 % kWindows;  // window slot in the ring
        const int sb = g1 & 1;        // S buffer
        const uint32_t ph = static_cast<uint32_t>(g1 / kWindows) & 1u;
        ok = mbar_wait_bounded(&sm->s_empty[sb], (static_cast<uint32_t>(g1 >> 1) & 1u) ^ 1u, abort_flag);
        const uint32_t d = tmem_base + (part_a ? kSCol : kSColB) + sb * kKeys;
        const uint32_t ks = k0 + w * kKeys * 128;  // the window's rows in every panel
        bool first = true;
        for (int gi = part_a ? 0 : 1; ok && gi < kGroups; gi += 2) {
          ok = mbar_wait_bounded(&sm->full[w][gi], ph, abort_flag);
          if (!ok) break;
          fence_proxy_async_smem();  // the gathered rows were written through the generic proxy
          tc_fence_after();
          const int np = gi < kGroups - 1 ? 2 : 1;
          for (int pi = 0; pi < np; ++pi) {
            const int pp = gi < kGroups - 1 ? 2 * gi + pi : 8;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t qoff = pp * (kH * 128) + kk * 32;
              const uint32_t koff = pp * kPanelBytes + kk * 32;
              tc_mma_bf16(d, desc_sw128(q0 + qoff, 16, 1024), desc_sw128(ks + koff, 16, 1024), id1,
                          first ? 0u : 1u);
              first = false;
            }
          }
        }
        if (!ok) break;
        tc_commit(&sm->s_full[sb]);
      }
      uint64_t *done = part_a ? &sm->mma_done : &sm->mma1b_done;
      tc_commit(done);
      mbar_wait_drain(done, 0, kWaitLimitNs);
    }
  } else if (warp == kGemm2Warp) {
    // ------------------------------------------------------------ GEMM 2 issuer
    // GEMM 2 of window j once every softmax warp has written its P rows (and,
    // when a head's reference max moved, rescaled its O^T lanes):
    // O^T[512 dims, 64 heads] += V^T . P^T, chunk by chunk, each chunk's
    // commit releasing the panel group it read; the last also releases the
    // RoPE panel that held P
    if (lane == 0 && nblk > 0) {
      constexpr uint32_t id2 = idesc(128, 64, true, false);
      int issued = 0;
      uint32_t nresc = 0;
      for (int j = 0; j < nblk; ++j) {
        if (!mbar_wait_bounded(&sm->p_full, static_cast<uint32_t>(j) & 1u, abort_flag)) break;
        const volatile int *nd = sm->need[j & 1];
        const bool any = (nd[0] | nd[1] | nd[2] | nd[3]) != 0;
        if (any && j > 0) {
          if (!mbar_wait_bounded(&sm->resc_done, nresc & 1u, abort_flag)) break;
          ++nresc;
        }
        tc_fence_after();
        const int w = j % kWindows;
        const uint32_t ks = smem_u32(sK) + w * kKeys * 128;
        const uint32_t p0 = smem_u32(sK) + 8 * kPanelBytes + w * kKeys * 128;  // P^T
#pragma unroll
        for (int c = 0; c < kDv / 128; ++c) {
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint64_t ad = desc_sw128(ks + 2 * c * kPanelBytes + kk * 16 * 128, kPanelBytes, 1024);
            const uint64_t bd = desc_sw128(p0 + kk * 32, 16, 1024);
            tc_mma_bf16(tmem_base + kOCol + c * 64, ad, bd, id2, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&sm->empty[w][c]);
        }
        tc_commit(&sm->empty[w][kGroups - 1]);
        tc_commit(&sm->p_free);
        ++issued;
      }
      // every GEMM 2 issued is complete before tensor memory is freed
      if (issued > 0) {
        tc_commit(&sm->mma2_done);
        mbar_wait_drain(&sm->mma2_done, 0, kWaitLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;                         // TMEM lane quarter of this warp
    const int w4 = warp - kSoftmaxWarp0;             // index among the softmax warps
    // the two half-warps share the 16 heads of the quarter: lane l takes head
    // 16 q4 + l % 16 and keys 32 (l / 16) .. +31 of every window
    const int hh = lane >> 4;
    const int head = q4 * 16 + (lane & 15);
    const bool owner = lane < 16;                    // writes the head's per-head results
    const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
    float m_ref = -INFINITY, l = 0.0f;
    bool all_ok = true;
    bool late_fail = false;     // a wait failed after this window's status exchange
    // validity of window j's keys (bit k of word h = key 32h + k), from the
    // index set itself; slots are loaded two windows ahead, checked when used
    auto load_slot = [&](int j, int h) -> int {
      return j < nblk ? slot_raw(irow, slot0 + j * kKeys + h * 32 + lane, p.K) : -1;
    };
    int n1[kHalves], n2[kHalves];
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
      n1[h] = load_slot(0, h);
      n2[h] = load_slot(1, h);
    }
    for (int j = 0; j < nblk; ++j) {
      const int sb = j & 1;
      uint32_t mask[kHalves];
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        mask[h] = __ballot_sync(0xffffffffu, checked_pos(n1[h], p.T, false) >= 0);
        n1[h] = n2[h];
        n2[h] = load_slot(j + 2, h);
      }
      bool ok = warp_wait(&sm->s_full[sb], static_cast<uint32_t>(j >> 1) & 1u, abort_flag);
      uint32_t sv[32];  // this lane's 32 raw scores (the two partials added), then scaled, masked logits
      float mt = -INFINITY;
      if (ok) {
        tc_fence_after();
        uint32_t t[32];
        tmem_ld_16x32bx2_x32(tmem_base + lane_addr + kSCol + sb * kKeys, sv);
        tmem_ld_16x32bx2_x32(tmem_base + lane_addr + kSColB + sb * kKeys, t);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->s_empty[sb]);
        const uint32_t mk = hh ? mask[1] : mask[0];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float v = ((mk >> k) & 1u) ? (__uint_as_float(sv[k]) + __uint_as_float(t[k])) * p.scale_log2
                                           : -INFINITY;
          sv[k] = __float_as_uint(v);
          mt = fmaxf(mt, v);
        }
      }
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));  // the head's window max (both half-warps)
      if (late_fail) ok = false;
      const bool need = ok && mt > m_ref + kRescaleLog2;
      const float m_new = need ? mt : m_ref;
      const float alpha = need ? fast_exp2(m_ref - m_new) : 1.0f;
      float rs = 0.0f;  // this lane's share of the head's window sum
      if (ok) {
        // this window's probabilities against the (possibly moved) reference,
        // as bf16 P^T row `head` in the window's RoPE panel (panel 8 of its
        // ring slot): GEMM 1 of this window, its only other reader, has
        // completed, and the panel is not refilled before GEMM 2 of this
        // window has read it
        const float ref = m_new == -INFINITY ? 0.0f : m_new;
        uint8_t *prow = sK + 8 * kPanelBytes + (j % kWindows) * kKeys * 128 + head * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = 4 * hh + cc;  // 16-byte chunk of the row: keys 8c .. 8c + 7
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = fast_exp2(__uint_as_float(sv[8 * cc + 2 * e]) - ref);
            const float bq = fast_exp2(__uint_as_float(sv[8 * cc + 2 * e + 1]) - ref);
            rs += a + bq;
            pk[e] = pack_bf16x2(a, bq);
          }
          *reinterpret_cast<uint4 *>(prow + ((c ^ (head & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      if (owner) sm->xa[j & 1][head] = alpha;
      fence_proxy_async_smem();
      tc_fence_before();
      const unsigned any_need = __ballot_sync(0xffffffffu, need);
      if (lane == 0) {
        sm->need[j & 1][w4] = any_need ? 1 : 0;
        sm->status[j & 1][w4] = ok ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->p_full);
      named_bar_sync(1, 128);
      all_ok = sm->status[j & 1][0] && sm->status[j & 1][1] && sm->status[j & 1][2] && sm->status[j & 1][3];
      if (!all_ok) break;
      const bool rescale = sm->need[j & 1][0] || sm->need[j & 1][1] || sm->need[j & 1][2] || sm->need[j & 1][3];
      if (rescale && j > 0) {
        // O^T column h *= alpha[h] on this warp's 32 lanes of every chunk,
        // once the previous window's GEMM 2 has completed and before this
        // window's is issued (rare: 8 columns at a time keeps the registers
        // of the hot path free).  A failed wait skips the rescale and fails
        // this warp at the next window's exchange (or at the epilogue's)
        if (!warp_wait(&sm->p_free, static_cast<uint32_t>(j - 1) & 1u, abort_flag)) {
          late_fail = true;
        } else {
          tc_fence_after();
#pragma unroll 1
          for (int g = 0; g < (kDv / 128) * (kH / 8); ++g) {
            const int c = g / (kH / 8), h0 = (g % (kH / 8)) * 8;
            const uint32_t taddr = tmem_base + lane_addr + kOCol + c * 64 + h0;
            uint32_t r[8];
            tmem_ld8(taddr, r);
#pragma unroll
            for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * sm->xa[j & 1][h0 + i]);
            tmem_st8(taddr, r);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->resc_done);
      }
      if (need) {
        m_ref = m_new;
        l *= alpha;
      }
      l += rs;
    }

    // ---- epilogue: O^T / l per head, staged in the idle gather buffers
    l += __shfl_xor_sync(0xffffffffu, l, 16);  // the head's sum: both half-warps' shares
    bool ok = all_ok && !late_fail;
    if (nblk > 0 && ok) ok = warp_wait(&sm->p_free, static_cast<uint32_t>(nblk - 1) & 1u, abort_flag);
    float *inv_l = sm->xa[0];
    named_bar_sync(1, 128);  // every warp is past its last read of xa
    if (owner) inv_l[head] = l > 0.0f ? 1.0f / l : 0.0f;
    if (lane == 0) sm->status[0][w4] = ok ? 1 : 0;
    named_bar_sync(1, 128);
    ok = sm->status[0][0] && sm->status[0][1] && sm->status[0][2] && sm->status[0][3];
    // After the last GEMM 2 every MMA into O^T is complete; on an abort it
    // may not be, so its tensor memory is not read.
    const bool one = unit_splits == 1;
    if (owner && p.cluster) {
      sm->cml[head][0] = ok ? m_ref : -INFINITY;
      sm->cml[head][1] = ok ? l : 0.0f;
    } else if (owner) {
      if (one) {
        if (p.lse[layer] != nullptr) {
          const float ln2 = 0.69314718055994531f;
          p.lse[layer][(size_t)row * kH + head] = (ok && l > 0.0f) ? (m_ref + log2f(l)) * ln2 : -INFINITY;
        }
      } else {
        float *pm = p.part_ml + (tile * kH) * 2;
        pm[head * 2 + 0] = ok ? m_ref : -INFINITY;
        pm[head * 2 + 1] = ok ? l : 0.0f;
      }
    }
  }

  // ---- the block's result, stored by every warp: once the softmax warps
  // have published 1/l and the block's status (and, when it is ok, the last
  // GEMM 2 has completed), warp w takes the 128-dim chunks w / 4, w / 4 +
  // (warps / 4), ... of O^T for its TMEM lane quarter w % 4, straight from
  // tensor memory to global memory: lane = dim, so for each head a warp's
  // stores cover 32 consecutive dims (coalesced).  After an abort the
  // tensor memory is not read (an MMA may still be writing it): zeros.
  tc_fence_before();
  __syncthreads();
  {
    const bool ok = sm->status[0][0] && sm->status[0][1] && sm->status[0][2] && sm->status[0][3];
    const bool one = unit_splits == 1;
    if (ok && nblk > 0) {
      tc_fence_after();
      const float *inv_l = sm->xa[0];
      const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
      // a cluster launch stages the partial in this block's idle ring
      // (every copy and MMA into it has completed) for the merge below
      float *po = one ? nullptr : (p.cluster ? reinterpret_cast<float *>(sK) : p.part_o + (tile * kH) * kDv);
      __nv_bfloat16 *bo = one ? p.out[layer] + (size_t)row * kH * kDv : nullptr;
#pragma unroll 1
      for (int c = warp >> 2; c < kDv / 128; c += R::kThreads / 128) {
        const int d = c * 128 + (warp & 3) * 32 + lane;
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32_nowait(tmem_base + lane_addr + kOCol + c * 64, r0);
        tmem_ld_32x32b_x32_nowait(tmem_base + lane_addr + kOCol + c * 64 + 32, r1);
        tmem_wait_ld();
        if (one) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            bo[i * kDv + d] = __float2bfloat16_rn(__uint_as_float(r0[i]) * inv_l[i]);
            bo[(32 + i) * kDv + d] = __float2bfloat16_rn(__uint_as_float(r1[i]) * inv_l[32 + i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            po[i * kDv + d] = __uint_as_float(r0[i]);
            po[(32 + i) * kDv + d] = __uint_as_float(r1[i]);
          }
        }
      }
    } else {
      uint4 *dst = one ? reinterpret_cast<uint4 *>(p.out[layer] + (size_t)row * kH * kDv)
                       : (p.cluster ? reinterpret_cast<uint4 *>(sK)
                                    : reinterpret_cast<uint4 *>(p.part_o + (tile * kH) * kDv));
      const int n16 = one ? kH * kDv * 2 / 16 : kH * kDv * 4 / 16;
      for (int i = threadIdx.x; i < n16; i += R::kThreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // ---- cluster launch: the unit's splits merge among themselves.  Every
  // CTA's partial O (staged above as [head][dim] fp32 in its ring) and its
  // (max, sum) per head are visible cluster-wide after the first barrier;
  // CTA `split` then merges dims [split * D, split * D + D), D = 512 / nsplit,
  // exactly as the combine kernel does, and the second barrier keeps every
  // CTA's shared memory alive until the others have read it.
  if (p.cluster) {
    const int ns = p.nsplit;
    cluster_sync_all();
    if (threadIdx.x < kH) {
      const int h = threadIdx.x;
      const uint32_t ml_local = smem_u32(&sm->cml[h][0]);
      float ms[kMaxClusterSplits], ls[kMaxClusterSplits];
      float M = -INFINITY;
      for (int s2 = 0; s2 < ns; ++s2) {
        const float2 v = ld_cluster_f2(cluster_map(ml_local, s2));
        ms[s2] = v.x;
        ls[s2] = v.y;
        M = fmaxf(M, v.x);
      }
      const float ref = M == -INFINITY ? 0.0f : M;
      float den = 0.0f;
      for (int s2 = 0; s2 < ns; ++s2) {
        const float f = exp2f(ms[s2] - ref);
        sm->cw[h][s2] = f;
        den += f * ls[s2];
      }
      sm->cinv[h] = den > 0.0f ? 1.0f / den : 0.0f;
      if (split == 0 && p.lse[layer] != nullptr)
        p.lse[layer][(size_t)row * kH + h] = den > 0.0f ? (M + log2f(den)) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();
    const int D = kDv / ns, q4n = D / 4;
    const uint32_t stage = smem_u32(sK);
    __nv_bfloat16 *orow = p.out[layer] + (size_t)row * kH * kDv;
    for (int it = threadIdx.x; it < kH * q4n; it += R::kThreads) {
      const int h = it / q4n, d = split * D + (it - h * q4n) * 4;
      const uint32_t off = stage + static_cast<uint32_t>((h * kDv + d) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s2 = 0; s2 < ns; ++s2) {
        const float f = sm->cw[h][s2];
        const float4 v = ld_cluster_f4(cluster_map(off, s2));
        acc.x += f * v.x;
        acc.y += f * v.y;
        acc.z += f * v.z;
        acc.w += f * v.w;
      }
      const float inv = sm->cinv[h];
      uint2 packed;
      packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2 *>(orow + (size_t)h * kDv + d) = packed;
    }
    cluster_sync_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace mla
}  // namespace dsa
