// Sparse absorbed-MLA attention over the rows an index set names.
//
// For one query token and one layer: z[h, j] = sm_scale * q[h, :] . kv[idx[j], :]
// over the 576-dim rows (512 compressed-KV dims + 64 rotated RoPE dims),
// p = softmax_j(z), O[h, :] = sum_j p[h, j] * kv[idx[j], :512]: the value is the
// leading kv_lora_rank dims of the same row ("GLM-5.2 Explained: 1M Token
// Context AI Agent Model", §2.1: K/V are loaded only for the selected
// positions; §1.1: MLA; kv_lora_rank = 512 in the GLM-5.2 config; 64 heads).
//
// Block = (layer, split, query row).  256 threads = 8 warps.  The block keeps
// the 64x576 query tile in shared memory and streams 64-row blocks of gathered
// latent rows (16-byte cp.async gathers, double-buffered, XOR-swizzled
// 16-byte chunks so ldmatrix is conflict-free).  Per block of 64 rows:
//   S = Q K^T      warp (wm, wn): heads 16*wm.., rows 32*wn..      (mma.sync)
//   online softmax in fp32 (exp2 with log2(e) folded into the scale);
//   P (bf16) goes through shared memory;
//   O += P V       warp (wm, wn): heads 16*wm.., dims 256*wn..     (mma.sync)
// A split over the index slots writes an unnormalised fp32 partial plus its
// (max, sum); the combine kernel merges the splits.  With one split the block
// normalises and writes bf16 directly.
#pragma once

#include "common.cuh"

namespace dsa {
namespace attn {

constexpr int kH = 64;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kBlk = 64;                       // gathered rows per block step
constexpr int kThreads = 256;
constexpr int kRowBytes = kDqk * 2;            // 1152
constexpr int kChunks = kRowBytes / 16;        // 72 chunks of 16 B per row
constexpr int kTileBytes = 64 * kRowBytes;     // 73728
constexpr int kPBytes = kH * kBlk * 2;         // 8192
constexpr int kMaxLayers = 8;
constexpr int kSmemBytes = 3 * kTileBytes + kPBytes + 2 * kBlk * 4 + 2 * kH * 4 + 2 * kH * 4;
static_assert(kSmemBytes <= 232448, "shared memory per block");

struct Params {
  const __nv_bfloat16 *q[kMaxLayers];   // [B*Q, 64, 576] per layer
  const __nv_bfloat16 *kv[kMaxLayers];  // [B, T, 576] per layer
  __nv_bfloat16 *out[kMaxLayers];       // [B*Q, 64, 512] per layer
  float *lse[kMaxLayers];               // [B*Q, 64] per layer, or null
  const int32_t *idx;                   // [B*Q, K], shared by every layer
  int n_layers, Q, T, K;
  int rows;                             // B*Q
  int nsplit, blocks_per_split;
  float *part_o;                        // [n_layers*rows, nsplit, 64, 512]
  float *part_ml;                       // [n_layers*rows, nsplit, 64, 2]
  float scale_log2;                     // sm_scale * log2(e)
};

// Byte offset of 16-byte chunk c of row r in a swizzled tile with 1152-byte rows.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return static_cast<uint32_t>(r * kRowBytes + (((c & ~7) | ((c ^ r) & 7)) << 4));
}
// Same for the 64x64 bf16 P tile (128-byte rows).
__device__ __forceinline__ uint32_t p_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sQ = smem;
  uint8_t *sK = smem + kTileBytes;                        // two stages
  uint8_t *sP = smem + 3 * kTileBytes;
  int *sValid = reinterpret_cast<int *>(sP + kPBytes);    // [2][64]
  float *sRedMax = reinterpret_cast<float *>(sValid + 2 * kBlk);  // [2][64]
  float *sRedSum = sRedMax + 2 * kH;                      // [2][64]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp & 3, wn = warp >> 2;
  const int g = lane >> 2, t4 = lane & 3;

  // block -> (layer, split, row); the layer varies fastest so that blocks that
  // gather the same rows (draft steps over one cache) run side by side.
  const int nl = p.n_layers;
  const int layer = blockIdx.x % nl;
  const int rest = blockIdx.x / nl;
  const int split = rest % p.nsplit;
  const int row = rest / p.nsplit;
  const int b = row / p.Q;

  const __nv_bfloat16 *qrow = p.q[layer] + (size_t)row * kH * kDqk;
  const __nv_bfloat16 *kvb = p.kv[layer] + (size_t)b * p.T * kDqk;
  const int32_t *irow = p.idx + (size_t)row * p.K;
  const int slot0 = split * p.blocks_per_split * kBlk;
  int nblk = p.blocks_per_split;
  {
    const int remaining = (p.K - slot0 + kBlk - 1) / kBlk;
    nblk = remaining < nblk ? remaining : nblk;
    if (nblk < 0) nblk = 0;
  }

  const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sPa = smem_u32(sP);

  // query tile
  for (int i = tid; i < kH * kChunks; i += kThreads) {
    const int r = i / kChunks, c = i - r * kChunks;
    cp_async_16(sQa + tile_off(r, c), reinterpret_cast<const uint8_t *>(qrow) + (size_t)r * kRowBytes + c * 16, 16);
  }
  cp_async_commit();

  auto load_block = [&](int j, int stage) {
    const int sbase = slot0 + j * kBlk;
    const uint32_t dst = sKa + stage * kTileBytes;
    for (int i = tid; i < kBlk * kChunks; i += kThreads) {
      const int r = i / kChunks, c = i - r * kChunks;
      const int slot = sbase + r;
      int pos = slot < p.K ? __ldg(irow + slot) : -1;
      if (pos < -1 || pos >= p.T) {
        if (c == 0) raise_error(kErrDeviceCheck);
        pos = -1;
      }
      const uint8_t *src = reinterpret_cast<const uint8_t *>(kvb) + (size_t)(pos < 0 ? 0 : pos) * kRowBytes + c * 16;
      cp_async_16(dst + tile_off(r, c), src, pos < 0 ? 0u : 16u);
      if (c == 0) sValid[stage * kBlk + r] = pos >= 0;
    }
    cp_async_commit();
  };

  float o[32][4];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 units) for heads g and g+8
  float l0 = 0.0f, l1 = 0.0f;            // this thread's partial sums

  const int hA = wm * 16;  // first head of this warp
  if (nblk > 0) load_block(0, 0);
  for (int j = 0; j < nblk; ++j) {
    const int stage = j & 1;
    if (j + 1 < nblk) {
      load_block(j + 1, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t kst = sKa + stage * kTileBytes;

    // ---- S = Q K^T for heads hA.., rows 32*wn..
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
#pragma unroll 4
    for (int ks = 0; ks < kDqk / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sQa + tile_off(hA + (lane & 7) + (((lane >> 3) & 1) << 3), ks * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + tile_off(wn * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)), b0,
                b1, b2, b3);
        mma_bf16_16816(s[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    // ---- scale, mask, block max
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int kk = wn * 32 + nt * 8 + 2 * t4;
      const bool v0 = sValid[stage * kBlk + kk] != 0, v1 = sValid[stage * kBlk + kk + 1] != 0;
      s[nt][0] = v0 ? s[nt][0] * p.scale_log2 : -INFINITY;
      s[nt][1] = v1 ? s[nt][1] * p.scale_log2 : -INFINITY;
      s[nt][2] = v0 ? s[nt][2] * p.scale_log2 : -INFINITY;
      s[nt][3] = v1 ? s[nt][3] * p.scale_log2 : -INFINITY;
      bm0 = fmaxf(bm0, fmaxf(s[nt][0], s[nt][1]));
      bm1 = fmaxf(bm1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
    }
    if (t4 == 0) {
      sRedMax[wn * kH + hA + g] = bm0;
      sRedMax[wn * kH + hA + g + 8] = bm1;
    }
    __syncthreads();
    bm0 = fmaxf(sRedMax[hA + g], sRedMax[kH + hA + g]);
    bm1 = fmaxf(sRedMax[hA + g + 8], sRedMax[kH + hA + g + 8]);
    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
    const float ref0 = mn0 == -INFINITY ? 0.0f : mn0;  // nothing valid yet: keep everything at 0
    const float ref1 = mn1 == -INFINITY ? 0.0f : mn1;
    const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = exp2f(s[nt][0] - ref0), p1 = exp2f(s[nt][1] - ref0);
      const float p2 = exp2f(s[nt][2] - ref1), p3 = exp2f(s[nt][3] - ref1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      const int c = wn * 4 + nt;  // 16-byte chunk of the P row (8 keys)
      *reinterpret_cast<uint32_t *>(sP + p_off(hA + g, c) + t4 * 4) = pack_bf16x2(p0, p1);
      *reinterpret_cast<uint32_t *>(sP + p_off(hA + g + 8, c) + t4 * 4) = pack_bf16x2(p2, p3);
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
    __syncthreads();

    // ---- O += P V for heads hA.., dims 256*wn..
#pragma unroll
    for (int ks = 0; ks < kBlk / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sPa + p_off(hA + (lane & 7) + (((lane >> 3) & 1) << 3), ks * 2 + (lane >> 4)), a0, a1, a2, a3);
      const int vrow = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int dp = 0; dp < 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(kst + tile_off(vrow, wn * 32 + dp * 2 + (lane >> 4)), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();  // stage and P are free for the next block
  }

  // ---- row sums over both key halves
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  if (t4 == 0) {
    sRedSum[wn * kH + hA + g] = l0;
    sRedSum[wn * kH + hA + g + 8] = l1;
  }
  __syncthreads();
  const float L0 = sRedSum[hA + g] + sRedSum[kH + hA + g];
  const float L1 = sRedSum[hA + g + 8] + sRedSum[kH + hA + g + 8];
  const int dbase = wn * 256 + 2 * t4;
  const size_t rowL = (size_t)layer * p.rows + row;

  if (p.nsplit == 1) {
    const float inv0 = L0 > 0.0f ? 1.0f / L0 : 0.0f;
    const float inv1 = L1 > 0.0f ? 1.0f / L1 : 0.0f;
    __nv_bfloat16 *orow = p.out[layer] + (size_t)row * kH * kDv;
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      const int d = dbase + nt * 8;
      *reinterpret_cast<uint32_t *>(orow + (size_t)(hA + g) * kDv + d) = pack_bf16x2(o[nt][0] * inv0, o[nt][1] * inv0);
      *reinterpret_cast<uint32_t *>(orow + (size_t)(hA + g + 8) * kDv + d) =
          pack_bf16x2(o[nt][2] * inv1, o[nt][3] * inv1);
    }
    if (p.lse[layer] != nullptr && wn == 0 && t4 == 0) {
      float *lrow = p.lse[layer] + (size_t)row * kH;
      const float ln2 = 0.69314718055994531f;
      lrow[hA + g] = L0 > 0.0f ? (m0 + log2f(L0)) * ln2 : -INFINITY;
      lrow[hA + g + 8] = L1 > 0.0f ? (m1 + log2f(L1)) * ln2 : -INFINITY;
    }
  } else {
    float *po = p.part_o + ((rowL * p.nsplit + split) * kH) * kDv;
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      const int d = dbase + nt * 8;
      *reinterpret_cast<float2 *>(po + (size_t)(hA + g) * kDv + d) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2 *>(po + (size_t)(hA + g + 8) * kDv + d) = make_float2(o[nt][2], o[nt][3]);
    }
    if (wn == 0 && t4 == 0) {
      float *pm = p.part_ml + ((rowL * p.nsplit + split) * kH) * 2;
      pm[(hA + g) * 2 + 0] = m0;
      pm[(hA + g) * 2 + 1] = L0;
      pm[(hA + g + 8) * 2 + 0] = m1;
      pm[(hA + g + 8) * 2 + 1] = L1;
    }
  }
}

// Merges the splits of one (layer, row, head): O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s, lse = (M + log2(sum)) * ln 2.  128 threads x 4 dims.
__global__ void __launch_bounds__(128) combine_kernel(const Params p) {
  const int head = blockIdx.x;
  const size_t rowL = blockIdx.y;
  const int layer = static_cast<int>(rowL / p.rows);
  const int row = static_cast<int>(rowL - (size_t)layer * p.rows);
  const float *pm = p.part_ml + (rowL * p.nsplit * kH) * 2;
  float M = -INFINITY;
  for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, pm[((size_t)s * kH + head) * 2]);
  const float ref = M == -INFINITY ? 0.0f : M;
  float den = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int d = threadIdx.x * 4;
  for (int s = 0; s < p.nsplit; ++s) {
    const float ms = pm[((size_t)s * kH + head) * 2], ls = pm[((size_t)s * kH + head) * 2 + 1];
    const float f = exp2f(ms - ref);
    den += f * ls;
    const float4 v = *reinterpret_cast<const float4 *>(p.part_o + ((rowL * p.nsplit + s) * kH + head) * kDv + d);
    acc.x += f * v.x;
    acc.y += f * v.y;
    acc.z += f * v.z;
    acc.w += f * v.w;
  }
  const float inv = den > 0.0f ? 1.0f / den : 0.0f;
  __nv_bfloat16 *orow = p.out[layer] + ((size_t)row * kH + head) * kDv + d;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(orow) = packed;
  if (threadIdx.x == 0 && p.lse[layer] != nullptr)
    p.lse[layer][(size_t)row * kH + head] = den > 0.0f ? (M + log2f(den)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace attn
}  // namespace dsa
