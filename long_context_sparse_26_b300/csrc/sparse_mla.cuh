// Shared parameters of the sparse MLA attention launch, and the kernel that
// merges split-k partial results.
//
// The attention of one query token over the rows an index set names
// ("GLM-5.2 Explained: 1M Token Context AI Agent Model", §2.1: K/V are loaded
// only for the selected positions) may be split over several blocks, each
// taking a contiguous slice of the index slots.  Each split leaves an
// unnormalised fp32 partial O_s[64 heads, 512 dims] and, per head, the
// reference max m_s (log2 units) its exponentials were taken against and its
// sum l_s.  combine_kernel merges them exactly:
//   O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s,
//   lse = (M + log2(sum_s 2^(m_s - M) l_s)) * ln 2.
#pragma once

#include "common.cuh"

namespace dsa {
namespace attn {

constexpr int kH = 64;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kMaxLayers = 8;
// FP8 latent row: the 512 compressed-KV dims as E4M3 codes, one fp32 scale
// per 128-dim group, then the 64 RoPE dims kept in bf16
constexpr int kF8Codes = 512;
constexpr int kF8ScaleOff = 512;                  // 4 x fp32
constexpr int kF8RopeOff = 528;                   // 64 x bf16
constexpr int kF8RowBytes = 656;

struct Params {
  const __nv_bfloat16 *q[kMaxLayers];   // [B*Q, 64, 576] per layer
  const void *kv[kMaxLayers];           // [B, T, 576] bf16 per layer, or [B, T, 656] bytes (FP8 rows)
  __nv_bfloat16 *out[kMaxLayers];       // [B*Q, 64, 512] per layer
  float *lse[kMaxLayers];               // [B*Q, 64] per layer, or null
  const int32_t *idx;                   // [B*Q, K], shared by every layer
  int n_layers, Q, T, K;
  int rows;                             // B*Q
  int nsplit, blocks_per_split;
  // units (layer u % n_layers, row u / n_layers) from tail_base on take
  // tail_nsplit splits of tail_bps windows instead (tail_nsplit 0: none;
  // then nsplit is 1); their partials are tiles (u - tail_base) * tail_nsplit + split
  int tail_base, tail_nsplit, tail_bps;
  // 1: the nsplit splits of each unit are one thread-block cluster (blocks
  // u * nsplit .. u * nsplit + nsplit - 1 for unit u), which merges them
  // itself through distributed shared memory: no partials, no combine
  int cluster;
  float *part_o;                        // [n_layers*rows, nsplit, 64, 512], or the tail units' tiles
  float *part_ml;                       // [n_layers*rows, nsplit, 64, 2], likewise
  float scale_log2;                     // sm_scale * log2(e)
  // paged latent caches (block_table null: kv[l] is [B, T, 576] contiguous):
  // position s of sequence b is row block_table[b][s / page_size] * page_size
  // + s % page_size of kv[l] viewed as a [num_pages * page_size, 576] pool
  const int32_t *block_table;           // [B, max_pages], shared by every layer
  int page_size, max_pages, num_pages;
  int kv_fp8;                           // 1: kv[l] holds FP8 latent rows of kF8RowBytes
};

// Merges the splits of one (layer, row, head): O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s, lse = (M + log2(sum)) * ln 2.  128 threads x 4 dims.
// blockIdx.y: the (layer, row) of the launch, or the tail unit.
__global__ void __launch_bounds__(128) combine_kernel(const Params p) {
  // launched as a dependent of the attention kernel: its partials are
  // complete and visible once this returns
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int head = blockIdx.x;
  int layer, row, ns;
  size_t tile0;  // the unit's first partial tile
  if (p.tail_nsplit > 0) {
    const int u = p.tail_base + static_cast<int>(blockIdx.y);
    layer = u % p.n_layers;
    row = u / p.n_layers;
    ns = p.tail_nsplit;
    tile0 = (size_t)blockIdx.y * ns;
  } else {
    const size_t rowL = blockIdx.y;
    layer = static_cast<int>(rowL / p.rows);
    row = static_cast<int>(rowL - (size_t)layer * p.rows);
    ns = p.nsplit;
    tile0 = rowL * ns;
  }
  const float *pm = p.part_ml + (tile0 * kH) * 2;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, pm[((size_t)s * kH + head) * 2]);
  const float ref = M == -INFINITY ? 0.0f : M;
  float den = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int d = threadIdx.x * 4;
  for (int s = 0; s < ns; ++s) {
    const float ms = pm[((size_t)s * kH + head) * 2], ls = pm[((size_t)s * kH + head) * 2 + 1];
    const float f = exp2f(ms - ref);
    den += f * ls;
    const float4 v = *reinterpret_cast<const float4 *>(p.part_o + ((tile0 + s) * kH + head) * kDv + d);
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
