/*
 * dsa.h — C ABI of libdsa: DSA sparse attention with IndexShare on B300 (sm_103a).
 *
 * The method (GLM-5.2's DSA with IndexShare):
 *   - A Lightning Indexer scores every cached position s for each query token t
 *     ("GLM-5.2 Explained: 1M Token Context AI Agent Model", §2.1, the relevance
 *     score I_{t,s} = w . sigma(q_t^T h_s)).  This library reads it in DSA's
 *     multi-head form  S[t,s] = sum_j w[t,j] * ReLU(q_I[t,j,:] . k_I[s,:])  with
 *     64 indexer heads of dim 128, causal (s <= pos(t)).
 *   - The top index_topk = 2048 positions are kept ("GLM-5.2核心技术解析：
 *     IndexShare架构与MTP层优化详解", section "IndexShare的工作原理", config keys).
 *   - Softmax attention of absorbed MLA runs over those rows only: 64 heads, key =
 *     the 576-dim cached row (512 compressed-KV dims, kv_lora_rank, then 64
 *     rotated RoPE dims), value = its first 512 dims.
 *   - IndexShare: the indexer and top-k run in the first layer of each group of
 *     index_topk_freq = 4 sparse layers; the other 3 reuse the index set
 *     ("GLM-5.2 技术报告解读", training-strategy table, IndexShare row).
 *   - With index_share_for_mtp_iteration, MTP draft steps after step 0 reuse its
 *     top-k and attend to the target model's cache only ("GLM-5.2 技术报告解读",
 *     section "MTP层改进"; "GLM-5.2 Explained", §2.2.1).
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers unless stated; the caller owns every buffer.
 *     The library allocates no device memory: scratch comes from a caller
 *     workspace of at least dsa_workspace_bytes() bytes.
 *   - Tensors are dense, row-major (C order) in the shapes given, and every
 *     pointer is 16-byte aligned (else DSA_ERR_ALIGNMENT).
 *   - bf16 tensors are passed as uint16_t bit patterns (dsa_bf16_t).
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and returns.  Argument errors are reported before
 *     anything is enqueued.  A failed launch returns DSA_ERR_CUDA.  Checks made on
 *     the device (an index outside [-1, T), a position outside [0, T), a wait
 *     that ran out of time) are recorded in a device error word that
 *     dsa_get_device_error() reads.
 *   - Index buffers hold int32 positions in [0, T) in ascending order, padded
 *     with -1 when fewer than topk positions are visible.
 *   - The fixed shape constants (64x128 indexer, 64 heads, 576/512 dims) are
 *     compiled in; a config with other values returns DSA_ERR_UNSUPPORTED.
 *   - A call with no query rows (B or Q, or S for MTP drafting, equal to 0 and
 *     no size negative) has nothing to do: it returns DSA_OK at once and
 *     reads no pointer.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dsa_bf16_t;               /* bf16 bit pattern */
typedef struct CUstream_st *dsa_stream_t;  /* same handle as cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive or too large size */
  DSA_ERR_UNSUPPORTED = 2,   /* config constant other than the compiled shapes */
  DSA_ERR_ALIGNMENT = 3,     /* a pointer not 16-byte aligned */
  DSA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
  DSA_ERR_CUDA = 5,          /* a CUDA runtime/driver call or launch failed */
  DSA_ERR_DEVICE_CHECK = 6,  /* a device-side argument check failed */
  DSA_ERR_TIMEOUT = 7        /* a device-side wait gave up */
} dsa_status_t;

/* Model constants (GLM-5.2 config keys: index_topk, index_topk_freq,
 * index_share_for_mtp_iteration, kv_lora_rank; 64 attention heads). */
typedef struct {
  int n_idx_heads;          /* indexer heads: 64 */
  int idx_dim;              /* indexer head dim: 128 */
  int topk;                 /* index_topk: 2048 (1..2048 accepted) */
  int topk_freq;            /* index_topk_freq: 4 layers per IndexShare group */
  int kv_lora_rank;         /* 512: value dims = leading latent dims */
  int rope_dim;             /* 64: trailing rotated key-only dims */
  int n_heads;              /* 64 attention heads */
  float sm_scale;           /* softmax scale, 1/sqrt(576) */
  int index_share_for_mtp;  /* 1: MTP draft steps reuse the step-0 index set */
} dsa_config_t;

/* Fills *cfg with the GLM-5.2 values above. */
void dsa_config_default(dsa_config_t *cfg);

/* Workspace bytes needed by any call below on B sequences x Q query tokens
 * with context T and n_layers attention layers per call (a group: n_layers =
 * topk_freq; MTP drafting: Q = 1, n_layers = the number of draft steps).
 * Returns 0 only for invalid arguments (a small nonzero size for an empty
 * call). */
size_t dsa_workspace_bytes(const dsa_config_t *cfg, int B, int Q, int T, int n_layers);

/* Indexer scores (step a1).
 *   q_idx  [B, Q, 64, 128] bf16   indexer queries
 *   w      [B, Q, 64]      fp32   per-token, per-head weights
 *   k_idx  [B, T, 128]     bf16   indexer key cache
 *   q_pos  [B, Q]          int32  position of each query token, in [0, T)
 *   scores [B, Q, T]       fp32   out: S[b,t,s] for s <= q_pos[b,t], -inf after
 * Runs on the tensor cores (tcgen05, TMA-fed key tiles). */
dsa_status_t dsa_indexer_scores(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                const dsa_bf16_t *k_idx, const int32_t *q_pos, int B, int Q, int T,
                                float *scores, dsa_stream_t stream);

/* Top-k selection (step a2).
 *   scores [B, Q, T] fp32, q_pos [B, Q] int32  ->  idx [B, Q, topk] int32
 * Row (b,t) keeps the min(topk, q_pos+1) positions s <= q_pos with the largest
 * scores, ties to the lower position, written in ascending position order and
 * padded with -1.  Scores must be finite.  Deterministic (radix select, no
 * sort).  Uses the workspace. */
dsa_status_t dsa_topk_select(const dsa_config_t *cfg, const float *scores, const int32_t *q_pos,
                             int B, int Q, int T, int32_t *idx, void *ws, size_t ws_bytes,
                             dsa_stream_t stream);

/* Sparse MLA attention, one layer (step a3).
 *   q   [B, Q, 64, 576] bf16   absorbed queries (512 latent + 64 RoPE dims)
 *   kv  [B, T, 576]     bf16   latent cache of this layer
 *   idx [B, Q, topk]    int32  positions to attend to (-1 = unused slot)
 *   out [B, Q, 64, 512] bf16   softmax(sm_scale * q . K^T) . K[:, :512]
 *   lse [B, Q, 64]      fp32   optional (NULL allowed): natural-log sum-exp of
 *                              the scaled logits (-inf when a row has no index)
 * A row with no valid index writes zeros.  Uses the workspace. */
dsa_status_t dsa_sparse_mla_attn(const dsa_config_t *cfg, const dsa_bf16_t *q, const dsa_bf16_t *kv,
                                 const int32_t *idx, int B, int Q, int T, dsa_bf16_t *out, float *lse,
                                 void *ws, size_t ws_bytes, dsa_stream_t stream);

/* One IndexShare group (steps a1 + a2 once, then a3 for every layer).
 *   q_idx, w, k_idx, q_pos   as for dsa_indexer_scores
 *   q[l]   [B, Q, 64, 576] bf16, kv[l] [B, T, 576] bf16, out[l] [B, Q, 64, 512]
 *          bf16 for l < n_layers (HOST arrays of n_layers device pointers;
 *          1 <= n_layers <= 8)
 *   idx_out [B, Q, topk] int32: optional (NULL allowed) copy of the shared set
 * The index set is computed once and read by all n_layers layers.  When the
 * stream reaches the end of the call, the workspace begins with the group's
 * indexer scores, [B, Q, T] fp32 exactly as dsa_indexer_scores writes them
 * (the same holds for the _paged and _fp8 group entry points below). */
dsa_status_t dsa_indexshare_group_forward(const dsa_config_t *cfg, const dsa_bf16_t *q_idx,
                                          const float *w, const dsa_bf16_t *k_idx,
                                          const int32_t *q_pos, const dsa_bf16_t *const *q,
                                          const dsa_bf16_t *const *kv, int n_layers, int B, int Q,
                                          int T, dsa_bf16_t *const *out, int32_t *idx_out, void *ws,
                                          size_t ws_bytes, dsa_stream_t stream);

/* Sparse MLA attention of n_layers layers over ONE shared index set (the
 * reuse half of step a4: the layers of an IndexShare group after the first
 * attend over the index set the first one selected).  One launch covers every
 * layer.
 *   q[l] [B, Q, 64, 576] bf16, kv[l] [B, T, 576] bf16, out[l] [B, Q, 64, 512]
 *        bf16 for l < n_layers (HOST arrays of device pointers; 1..8 layers)
 *   idx  [B, Q, topk] int32, as for dsa_sparse_mla_attn
 * Layer l's output equals dsa_sparse_mla_attn on (q[l], kv[l], idx) up to
 * the rounding of a different split of the key range.  Uses the workspace
 * (dsa_workspace_bytes with the same n_layers). */
dsa_status_t dsa_sparse_mla_attn_shared(const dsa_config_t *cfg, const dsa_bf16_t *const *q,
                                        const dsa_bf16_t *const *kv, int n_layers, const int32_t *idx, int B,
                                        int Q, int T, dsa_bf16_t *const *out, void *ws, size_t ws_bytes,
                                        dsa_stream_t stream);

/* MTP draft attention with index reuse (step a6).
 *   idx0    [B, 1, topk]    int32  the step-0 index set (from the indexer and
 *                                  top-k at the target's last position)
 *   q_steps [S, B, 64, 576] bf16   one query per draft step
 *   kv      [B, T, 576]     bf16   the target model's cache (no draft KV)
 *   out     [S, B, 64, 512] bf16
 * Every draft step attends to the rows idx0 names; 1 <= S <= 8.  The steps'
 * queries are all given up front; calling with S = 1 once per step gives the
 * same result. */
dsa_status_t dsa_mtp_draft_attn(const dsa_config_t *cfg, const int32_t *idx0,
                                const dsa_bf16_t *q_steps, const dsa_bf16_t *kv, int S, int B, int T,
                                dsa_bf16_t *out, void *ws, size_t ws_bytes, dsa_stream_t stream);

/* Sparse MLA attention without any caller workspace (same arguments and
 * result as dsa_sparse_mla_attn, minus ws/ws_bytes).  The pages have no
 * counterpart: this is for callers that cannot allocate device memory at the
 * point of the call -- e.g. code running where cudaMalloc is forbidden or
 * unsafe (inside a framework's memory pool or an allocator callback, or a
 * host that reserved all device memory up front) -- and so cannot provide
 * the split-k scratch that dsa_sparse_mla_attn takes from its workspace.
 * The scratch is instead a fixed 16 MiB array compiled into the library,
 * which every GPU that loads the library keeps until the process exits.
 *   - At most 64 query rows (B * Q <= 64) per call; larger calls return
 *     DSA_ERR_WORKSPACE before anything is enqueued.  The key range is split
 *     over fewer blocks than dsa_sparse_mla_attn may use when the rows'
 *     partial results would not fit, so outputs agree with it to rounding.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array and nothing in it needs to
 *     start at zero; calls whose work overlaps on the GPU (different streams,
 *     no ordering between them) race on it and must not be issued.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
dsa_status_t dsa_sparse_mla_attn_noalloc(const dsa_config_t *cfg, const dsa_bf16_t *q, const dsa_bf16_t *kv,
                                         const int32_t *idx, int B, int Q, int T, dsa_bf16_t *out, float *lse,
                                         dsa_stream_t stream);

/* Paged caches (the serving layout: fixed-size pages in a pool, one block
 * table per sequence).  Position s of sequence b is held in row
 *   block_table[b * max_pages + s / page_size] * page_size + s % page_size
 * of a pool viewed as [num_pages * page_size, row].  page_size is a multiple
 * of 64 (else DSA_ERR_UNSUPPORTED); max_pages * page_size >= T.  A page index
 * outside [0, num_pages) is reported through the device error word
 * (DSA_ERR_DEVICE_CHECK) and its rows read as zeros.  block_table is a DEVICE
 * pointer; the struct itself is read on the host at the call. */
typedef struct {
  const int32_t *block_table;  /* [B, max_pages] */
  int num_pages;
  int page_size;
  int max_pages;
} dsa_pages_t;

/* dsa_indexer_scores over a paged key cache k_pool [num_pages, page_size, 128]
 * bf16; everything else as there. */
dsa_status_t dsa_indexer_scores_paged(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                      const dsa_bf16_t *k_pool, const dsa_pages_t *pages, const int32_t *q_pos, int B,
                                      int Q, int T, float *scores, dsa_stream_t stream);

/* dsa_sparse_mla_attn over a paged latent cache kv_pool [num_pages, page_size,
 * 576] bf16; idx holds logical positions, as there. */
dsa_status_t dsa_sparse_mla_attn_paged(const dsa_config_t *cfg, const dsa_bf16_t *q, const dsa_bf16_t *kv_pool,
                                       const dsa_pages_t *pages, const int32_t *idx, int B, int Q, int T,
                                       dsa_bf16_t *out, float *lse, void *ws, size_t ws_bytes, dsa_stream_t stream);

/* dsa_indexshare_group_forward over a paged key cache k_pool and paged
 * latent caches kv_pools[l] (all sharing one block table, as the layers of a
 * model share their sequences' page layout). */
dsa_status_t dsa_indexshare_group_forward_paged(const dsa_config_t *cfg, const dsa_bf16_t *q_idx, const float *w,
                                                const dsa_bf16_t *k_pool, const int32_t *q_pos,
                                                const dsa_bf16_t *const *q, const dsa_bf16_t *const *kv_pools,
                                                int n_layers, const dsa_pages_t *pages, int B, int Q, int T,
                                                dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                                dsa_stream_t stream);

/* FP8 (E4M3) indexer caches, the "KV-cache FP8" storage of the pages: each
 * 128-dim key row k8[b,s,:] (bytes, E4M3) stands for k8[b,s,:] * k_scale[b,s]
 * and each query head row q8[b,t,j,:] for q8[b,t,j,:] * q_scale[b,t,j]; the
 * scales are positive fp32 (a positive scale passes through the ReLU, so
 * S[b,t,s] = k_scale[b,s] * sum_j w[b,t,j] q_scale[b,t,j] ReLU(q8 . k8)).
 *   q_idx8 [B, Q, 64, 128] u8, q_scale [B, Q, 64] fp32, k_idx8 [B, T, 128] u8,
 *   k_scale [B, T] fp32; everything else as for dsa_indexer_scores.  The
 *   products are exact in the tensor cores (kind::f8f6f4) and summed in fp32. */
dsa_status_t dsa_indexer_scores_fp8(const dsa_config_t *cfg, const uint8_t *q_idx8, const float *q_scale,
                                    const float *w, const uint8_t *k_idx8, const float *k_scale, const int32_t *q_pos,
                                    int B, int Q, int T, float *scores, dsa_stream_t stream);

/* dsa_indexshare_group_forward with FP8 indexer caches (as above); the
 * latent caches and attention stay bf16. */
dsa_status_t dsa_indexshare_group_forward_fp8(const dsa_config_t *cfg, const uint8_t *q_idx8, const float *q_scale,
                                              const float *w, const uint8_t *k_idx8, const float *k_scale,
                                              const int32_t *q_pos, const dsa_bf16_t *const *q,
                                              const dsa_bf16_t *const *kv, int n_layers, int B, int Q, int T,
                                              dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                              dsa_stream_t stream);

/* FP8 latent cache (the KV cache in FP8: "GLM-5.2 Explained: 1M Token Context
 * AI Agent Model", §3 and §5, Deployment Reference; the pages fix no row
 * format, so this is the library's reading, the one serving stacks use for
 * MLA caches).  Each cached position is one 656-byte row:
 *   bytes   0..511  the 512 compressed-KV dims as E4M3 codes,
 *   bytes 512..527  four fp32 scales, one per 128-dim group of those codes,
 *   bytes 528..655  the 64 RoPE dims, bf16 (kept at full width).
 * Row (b, s) stands for dims d < 512: code[d] * scale[d / 128], dims 512..575:
 * the RoPE values.  The kernel rounds each dequantised value to bf16 before
 * its bf16 tensor-core products (within the attention tolerance).  Code 0x7F /
 * 0xFF (E4M3 NaN) must not occur.
 * dsa_sparse_mla_attn with kv8 [B, T, 656] bytes (16-byte aligned); everything
 * else as there. */
dsa_status_t dsa_sparse_mla_attn_fp8(const dsa_config_t *cfg, const dsa_bf16_t *q, const uint8_t *kv8,
                                     const int32_t *idx, int B, int Q, int T, dsa_bf16_t *out, float *lse, void *ws,
                                     size_t ws_bytes, dsa_stream_t stream);

/* dsa_indexshare_group_forward_fp8 with FP8 latent caches too: kv8[l] is
 * [B, T, 656] bytes in the row format above. */
dsa_status_t dsa_indexshare_group_forward_fp8kv(const dsa_config_t *cfg, const uint8_t *q_idx8,
                                                const float *q_scale, const float *w, const uint8_t *k_idx8,
                                                const float *k_scale, const int32_t *q_pos, const dsa_bf16_t *const *q,
                                                const uint8_t *const *kv8, int n_layers, int B, int Q, int T,
                                                dsa_bf16_t *const *out, int32_t *idx_out, void *ws, size_t ws_bytes,
                                                dsa_stream_t stream);

/* FP8 caches in the paged layout (the pages' serving stack runs the FP8 KV
 * cache and PagedAttention together: "GLM-5.2 Explained: 1M Token Context AI
 * Agent Model", §5, Deployment Reference).  Every pool shares the one block
 * table of `pages` (the dsa_pages_t rules above):
 *   k8_pool      [num_pages, page_size, 128] u8   E4M3 indexer key codes
 *   k_scale_pool [num_pages, page_size]      fp32 their row scales
 *   kv8_pool(s)  [num_pages, page_size, 656] u8   FP8 latent rows (format above)
 *   kv_pools     [num_pages, page_size, 576] bf16 bf16 latent rows
 * Position s of sequence b reads row s % page_size of page
 * block_table[b * max_pages + s / page_size] in every pool; a page outside
 * [0, num_pages) is reported (DSA_ERR_DEVICE_CHECK) and reads page 0.
 * Results equal the contiguous FP8 entry points' on the caches the pools
 * stand for, bit for bit. */
dsa_status_t dsa_indexer_scores_fp8_paged(const dsa_config_t *cfg, const uint8_t *q_idx8, const float *q_scale,
                                          const float *w, const uint8_t *k8_pool, const float *k_scale_pool,
                                          const dsa_pages_t *pages, const int32_t *q_pos, int B, int Q, int T,
                                          float *scores, dsa_stream_t stream);

dsa_status_t dsa_sparse_mla_attn_fp8_paged(const dsa_config_t *cfg, const dsa_bf16_t *q, const uint8_t *kv8_pool,
                                           const dsa_pages_t *pages, const int32_t *idx, int B, int Q, int T,
                                           dsa_bf16_t *out, float *lse, void *ws, size_t ws_bytes,
                                           dsa_stream_t stream);

/* FP8 indexer caches, bf16 latent pools. */
dsa_status_t dsa_indexshare_group_forward_fp8_paged(const dsa_config_t *cfg, const uint8_t *q_idx8,
                                                    const float *q_scale, const float *w, const uint8_t *k8_pool,
                                                    const float *k_scale_pool, const int32_t *q_pos,
                                                    const dsa_bf16_t *const *q, const dsa_bf16_t *const *kv_pools,
                                                    int n_layers, const dsa_pages_t *pages, int B, int Q, int T,
                                                    dsa_bf16_t *const *out, int32_t *idx_out, void *ws,
                                                    size_t ws_bytes, dsa_stream_t stream);

/* FP8 indexer caches and FP8 latent pools. */
dsa_status_t dsa_indexshare_group_forward_fp8kv_paged(const dsa_config_t *cfg, const uint8_t *q_idx8,
                                                      const float *q_scale, const float *w, const uint8_t *k8_pool,
                                                      const float *k_scale_pool, const int32_t *q_pos,
                                                      const dsa_bf16_t *const *q, const uint8_t *const *kv8_pools,
                                                      int n_layers, const dsa_pages_t *pages, int B, int Q, int T,
                                                      dsa_bf16_t *const *out, int32_t *idx_out, void *ws,
                                                      size_t ws_bytes, dsa_stream_t stream);

/* Sets the time limit of the library's bounded device-side waits (an
 * mbarrier phase a kernel waits on: a tile landing, an MMA completing, a peer
 * warp's arrival), in nanoseconds of the GPU's global timer, for every kernel
 * enqueued on the current device after this call; 0 restores the default of
 * 2 s.  A kernel whose wait runs out records DSA_ERR_TIMEOUT in the device
 * error word, stops its block in step (copies and MMAs still in flight are
 * drained, tensor memory is freed after them), leaves its outputs
 * unspecified and returns; the context stays usable.  The drain waits at
 * block exit always keep the full 2 s limit.  The pages have no counterpart:
 * this is the library's failure-detection knob, so that a caller can make a
 * stuck dependency surface sooner than 2 s.
 * Synchronous with respect to the host (it writes a __device__ variable);
 * returns DSA_ERR_CUDA if that write fails. */
dsa_status_t dsa_set_wait_limit_ns(unsigned long long limit_ns);

/* Human-readable name of a status. */
const char *dsa_status_string(dsa_status_t status);

/* Synchronizes `stream`, then reads and clears the device error word:
 * DSA_OK, DSA_ERR_DEVICE_CHECK or DSA_ERR_TIMEOUT (DSA_ERR_CUDA if the
 * synchronization itself failed). */
dsa_status_t dsa_get_device_error(dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
