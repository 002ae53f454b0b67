"""CPU oracle for DSA sparse attention with IndexShare (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only the tests, the smoke check and the benchmark's CPU
baseline leg do.  It shares no code with the CUDA library.

The oracle is the plain definition of each step, written out in fp64:

* ``indexer_scores``: the Lightning Indexer score of every cached position for
  every query token ("GLM-5.2 Explained: 1M Token Context AI Agent Model",
  §2.1 "IndexShare: Cross-Layer Index Sharing for DSA Sparse Attention", the
  relevance score I_{t,s} = w . sigma(q_t^T h_s)).  The page names neither
  sigma nor the shape of w; this oracle reads it as DSA's multi-head form
  I[t, s] = sum_j w[t, j] * ReLU(q_I[t, j, :] . k_I[s, :]) with per-token,
  per-head weights w and no further scale.  Positions after the query's own
  position are masked (causal, the query's own position included).
* ``topk_select``: keep the top-k positions by score (same section: "selects
  the top-K high-relevance positions"), k = ``index_topk`` = 2048 ("GLM-5.2
  核心技术解析：IndexShare架构与MTP层优化详解", section "IndexShare的工作原理",
  config keys).  Ties go to the lower position.  The pages fix no order for
  the result; the oracle returns positions in ascending order and pads with -1
  when fewer than k positions are visible.  Implemented as one full stable
  sort of the visible row, no partial selection.
* ``sparse_mla_attn``: softmax attention over the gathered latent rows only
  ("GLM-5.2 Explained", §2.1: K and V are loaded only for the selected
  positions; §1.1: MLA is kept).  Absorbed MLA: each cached row is the 512-dim
  compressed KV (``kv_lora_rank`` = 512, "GLM-5.2核心技术解析", section "MTP在
  配置文件中的体现") followed by 64 rotated RoPE dims.  The key is the whole
  576-dim row, the value is its first 512 dims, 64 heads ("主要技术参数").
  Exact softmax: subtract the maximum, exponentiate, divide by the sum.
* ``indexshare_group_forward``: only the first layer of a group of
  ``index_topk_freq`` = 4 sparse layers runs the indexer and top-k; the other
  three reuse its index set ("GLM-5.2 技术报告解读", section "1. 预训练 Recipe",
  training-strategy table, IndexShare row; "GLM-5.2 Explained", §2.1, the
  reuse pseudocode).  The layers are independent given the index set.
* ``mtp_draft_attn``: with ``index_share_for_mtp_iteration`` set, only draft
  step 0 runs the indexer; later steps reuse its top-k, and attend only to the
  target model's cache, never to MTP-produced KV ("GLM-5.2 技术报告解读",
  section "MTP层改进"; "GLM-5.2 Explained", §2.2.1 "Index Sharing and KV Cache
  Reuse for MTP").
* ``gather_pages``: a paged cache (fixed-size pages in a pool, one block
  table per sequence: the page-table-managed KV cache of "GLM-5.2 Explained",
  §3 "System Optimization for 1M-Token Context Inference", and the
  PagedAttention deployment of §5 "Deployment Reference") read back as the
  contiguous cache it stands for: position s of sequence b is row
  s % page_size of page block_table[b, s // page_size].
* ``e4m3_to_f64``: exact value of FP8 E4M3 codes (the "KV-cache FP8" storage
  of "GLM-5.2 技术报告解读", section "2. 后训练 Pipeline", and the
  ``--kv-cache-dtype fp8`` of "GLM-5.2 Explained", §3), from the format
  definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
  subnormals at exponent 0, S.1111.111 is NaN and nothing is infinite.  An
  FP8 cache row stands for its decoded values times its fp32 scale; the
  oracle's indexer scores are those of the decoded, scaled rows.
* ``fp8_latent_to_f64``: the value of an FP8 latent cache row (the same
  FP8 KV cache, here for the MLA latent rows).  The pages fix no row layout;
  the reading taken is the one serving stacks use for MLA caches: 512
  compressed-KV dims as E4M3 codes with one fp32 scale per 128-dim group,
  followed by the 64 RoPE dims in bf16, 656 bytes per row.  Dim d < 512 is
  code[d] * scale[d // 128]; the RoPE dims are their bf16 values.  The
  oracle's attention over an FP8 cache is its attention over these values.
* ``indexer_flops``: the indexer's multiply-add count per query token, shared
  or per layer ("GLM-5.2 技术报告解读", training-strategy table: IndexShare
  removes the indexer dot products and top-k of 3 of every 4 layers).

Pins: every function here is checked by tests that do not reuse its code:
closed forms and hand-worked fixtures (tests/golden), brute force on tiny
inputs, dense attention as the k >= L special case, and invariants.  The one
figure left "parity unpinned" is the pages' 2.9x whole-model FLOP reduction at
1M context: it depends on the full model's FLOP mix, which the pages do not
give; only the indexer's exact 4x is pinned.
"""
from __future__ import annotations

import numpy as np

D_V_DEFAULT = 512


# ----------------------------------------------------------------------------
# bf16 helpers (bit patterns -> fp64, and round-to-nearest-even for reports)
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 value of bf16 bit patterns (uint16/int16 array)."""
    u32 = bits.astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even), returned as fp64."""
    f32 = np.asarray(x, dtype=np.float32)
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# a1: Lightning Indexer scores
# ----------------------------------------------------------------------------

def indexer_scores_row(q_idx: np.ndarray, w: np.ndarray, k_idx: np.ndarray, pos: int) -> np.ndarray:
    """Scores of one query token over one sequence's keys.

    q_idx [H_I, D_I], w [H_I], k_idx [T, D_I] (fp64).  Returns [T] fp64 with
    S[s] = sum_j w[j] * max(0, q_idx[j] . k_idx[s]) for s <= pos, and -inf for
    s > pos.
    """
    T = k_idx.shape[0]
    out = np.full(T, -np.inf, dtype=np.float64)
    L = min(pos + 1, T)
    if L <= 0:
        return out
    logits = q_idx @ k_idx[:L].T                 # [H_I, L], one dot product per (head, key)
    out[:L] = w @ np.maximum(logits, 0.0)        # ReLU per head, then the weighted head sum
    return out


def indexer_scores(q_idx: np.ndarray, w: np.ndarray, k_idx: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    """Scores [B, Q, T] for q_idx [B, Q, H_I, D_I], w [B, Q, H_I], k_idx [B, T, D_I], q_pos [B, Q]."""
    B, Q = q_pos.shape
    T = k_idx.shape[1]
    out = np.empty((B, Q, T), dtype=np.float64)
    for b in range(B):
        for t in range(Q):
            out[b, t] = indexer_scores_row(q_idx[b, t], w[b, t], k_idx[b], int(q_pos[b, t]))
    return out


# ----------------------------------------------------------------------------
# a2: top-k selection
# ----------------------------------------------------------------------------

def topk_select_row(scores: np.ndarray, pos: int, k: int) -> np.ndarray:
    """Top-k of one row: positions 0..pos, order (score desc, position asc).

    A full stable sort of the visible row by descending score keeps equal
    scores in ascending position order, so ties go to the lower position.
    The first min(k, L) positions are returned sorted ascending, padded with
    -1 to length k.
    """
    L = min(pos + 1, scores.shape[0])
    out = np.full(k, -1, dtype=np.int64)
    if L <= 0:
        return out
    visible = scores[:L]
    order = np.argsort(-visible, kind="stable")
    chosen = np.sort(order[:min(k, L)])
    out[:chosen.shape[0]] = chosen
    return out


def topk_select(scores: np.ndarray, q_pos: np.ndarray, k: int) -> np.ndarray:
    """idx [B, Q, k] int64 from scores [B, Q, T]."""
    B, Q = q_pos.shape
    out = np.empty((B, Q, k), dtype=np.int64)
    for b in range(B):
        for t in range(Q):
            out[b, t] = topk_select_row(scores[b, t], int(q_pos[b, t]), k)
    return out


# ----------------------------------------------------------------------------
# a3: sparse MLA attention over the selected rows
# ----------------------------------------------------------------------------

def sparse_mla_attn_row(q: np.ndarray, kv: np.ndarray, idx: np.ndarray, sm_scale: float,
                        d_v: int = D_V_DEFAULT):
    """Attention of one query token over the latent rows its indices name.

    q [H, D_qk], kv [T, D_qk] (or any array indexable by position), idx [k]
    with -1 for unused slots.  Returns (O [H, d_v], lse [H]) where
    z = sm_scale * q . K^T over the valid positions, p = softmax(z),
    O = p . K[:, :d_v] and lse = log(sum(exp(z))).  With no valid position,
    O = 0 and lse = -inf.
    """
    H = q.shape[0]
    valid = idx[idx >= 0]
    if valid.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    K = np.asarray(kv[valid], dtype=np.float64)  # gather [n, D_qk]
    z = sm_scale * (q @ K.T)                      # [H, n]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    O = p @ K[:, :d_v]                            # value = the first d_v (latent) dims
    lse = (m + np.log(l))[:, 0]
    return O, lse


def sparse_mla_attn(q: np.ndarray, kv: np.ndarray, idx: np.ndarray, sm_scale: float,
                    d_v: int = D_V_DEFAULT):
    """O [B, Q, H, d_v], lse [B, Q, H] for q [B, Q, H, D_qk], kv [B, T, D_qk], idx [B, Q, k]."""
    B, Q, H, _ = q.shape
    O = np.empty((B, Q, H, d_v))
    lse = np.empty((B, Q, H))
    for b in range(B):
        for t in range(Q):
            O[b, t], lse[b, t] = sparse_mla_attn_row(q[b, t], kv[b], idx[b, t], sm_scale, d_v)
    return O, lse


# ----------------------------------------------------------------------------
# a4 / a5: one IndexShare group, and the per-layer-indexer variant
# ----------------------------------------------------------------------------

def indexshare_group_forward(q_idx, w, k_idx, q_pos, qs, kvs, k: int, sm_scale: float,
                             d_v: int = D_V_DEFAULT):
    """One group: the indexer and top-k run once, every layer reuses the index set.

    Mirrors the reuse rule "compute the index set when none is held, else
    reuse the previous one" for the layers of one group.  Returns
    (idx [B, Q, k], [O_layer], [lse_layer]).
    """
    held = None
    outs, lses = [], []
    for q_l, kv_l in zip(qs, kvs):
        if held is None:
            held = topk_select(indexer_scores(q_idx, w, k_idx, q_pos), q_pos, k)
        O, lse = sparse_mla_attn(q_l, kv_l, held, sm_scale, d_v)
        outs.append(O)
        lses.append(lse)
    return held, outs, lses


def per_layer_indexer_forward(idx_qs, idx_ws, idx_ks, q_pos, qs, kvs, k: int, sm_scale: float,
                              d_v: int = D_V_DEFAULT):
    """Without IndexShare: every layer runs its own indexer and top-k."""
    idxs, outs = [], []
    for qi, wi, ki, q_l, kv_l in zip(idx_qs, idx_ws, idx_ks, qs, kvs):
        idx = topk_select(indexer_scores(qi, wi, ki, q_pos), q_pos, k)
        O, _ = sparse_mla_attn(q_l, kv_l, idx, sm_scale, d_v)
        idxs.append(idx)
        outs.append(O)
    return idxs, outs


# ----------------------------------------------------------------------------
# a6: MTP drafting with index reuse and KV share
# ----------------------------------------------------------------------------

def mtp_draft_attn(idx0: np.ndarray, q_steps: np.ndarray, kv: np.ndarray, sm_scale: float,
                   d_v: int = D_V_DEFAULT):
    """Draft steps that reuse the step-0 index set over the target's cache.

    idx0 [B, 1, k] (or [B, k]), q_steps [S, B, H, D_qk], kv [B, T, D_qk] is the
    target model's cache only: no draft-produced KV is appended, so no draft
    step attends to itself.  Returns O [S, B, H, d_v].
    """
    S, B, H, _ = q_steps.shape
    idx = idx0.reshape(B, -1)
    O = np.empty((S, B, H, d_v))
    for s in range(S):
        for b in range(B):
            O[s, b], _ = sparse_mla_attn_row(q_steps[s, b], kv[b], idx[b], sm_scale, d_v)
    return O


# ----------------------------------------------------------------------------
# Indexer work count (IndexShare saving)
# ----------------------------------------------------------------------------

def indexer_flops(T: int, n_layers: int, share: bool, n_heads: int = 64, head_dim: int = 128) -> int:
    """Indexer FLOPs per query token over a context of T keys for n_layers layers.

    Each visible key costs one head_dim dot product per indexer head (2 FLOP
    per multiply-add).  With IndexShare the indexer runs once per group of
    n_layers layers, otherwise once per layer.
    """
    per_pass = 2 * n_heads * head_dim * T
    return per_pass * (1 if share else n_layers)


# ----------------------------------------------------------------------------
# Paged caches
# ----------------------------------------------------------------------------

def gather_pages(pool: np.ndarray, block_table: np.ndarray, T: int) -> np.ndarray:
    """Contiguous [B, T, D] cache of a paged pool [num_pages, page_size, D]:
    row s of sequence b is pool[block_table[b, s // page_size], s % page_size]."""
    page_size = pool.shape[1]
    B = block_table.shape[0]
    s = np.arange(T)
    out = np.empty((B, T) + pool.shape[2:], dtype=pool.dtype)
    for b in range(B):
        out[b] = pool[block_table[b, s // page_size], s % page_size]
    return out


# ----------------------------------------------------------------------------
# FP8 (E4M3) storage
# ----------------------------------------------------------------------------

def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact fp64 value of E4M3 byte codes (NaN for the two NaN codes)."""
    c = np.asarray(codes).astype(np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = sign * np.ldexp(m / 8.0, -6)
    v = np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, v)


FP8_LATENT_ROW_BYTES = 656


def fp8_latent_to_f64(rows: np.ndarray) -> np.ndarray:
    """Values [..., 576] (fp64) of FP8 latent rows [..., 656] (uint8): bytes
    0..511 are E4M3 codes of dims 0..511, bytes 512..527 four little-endian
    fp32 scales (dims 128g..128g+127 use scale g), bytes 528..655 the 64 RoPE
    dims as little-endian bf16."""
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.uint8))
    if r.shape[-1] != FP8_LATENT_ROW_BYTES:
        raise ValueError("FP8 latent rows are 656 bytes")
    lead = r.shape[:-1]
    codes = e4m3_to_f64(r[..., :512]).reshape(*lead, 4, 128)
    scales = np.ascontiguousarray(r[..., 512:528]).view("<f4").astype(np.float64)  # [..., 4]
    nope = (codes * scales[..., None]).reshape(*lead, 512)
    rope = bf16_bits_to_f64(np.ascontiguousarray(r[..., 528:656]).view("<u2"))       # [..., 64]
    return np.concatenate([nope, rope], axis=-1)
