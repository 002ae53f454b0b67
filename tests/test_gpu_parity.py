"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Small seeded cases span several tiles and a ragged tail; edge cases cover
ties, short rows (-1 padding), masked positions and bad indices.  Tolerances
are in tests/parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_26_b300 import binding as dsa
from long_context_sparse_26_b300 import workloads as wl
from parity import check_attention, check_scores_row, check_topk_row, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCALE = wl.SM_SCALE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from long_context_sparse_26_b300.build import build_library
    build_library()
    dsa.lib()
    yield
    assert dsa.get_device_error() == 0


def _indexer_inputs(B, Q, T, first_pos, seed):
    q_idx = wl.indexer_queries(B, Q, seed, DEV)
    w = wl.head_weights(B, Q, seed, DEV)
    k_idx = wl.indexer_keys(B, T, seed, DEV)
    pos = torch.arange(first_pos, first_pos + Q, dtype=torch.int32, device=DEV).unsqueeze(0).repeat(B, 1)
    return q_idx, w, k_idx, pos.contiguous()


# --------------------------------------------------------------------------- a1: indexer scores

@pytest.mark.parametrize("B,Q,T,first", [
    (2, 1, 3000, 2999),      # decode, N=64, ragged last tile
    (1, 2, 1000, 998),       # two queries per group (N=128)
    (1, 4, 2500, 2496),      # four queries per group (N=256)
    (2, 5, 700, 300),        # ragged query group, masked tail tiles
    (1, 9, 4100, 4000),      # several groups, causal
    (3, 1, 128, 127),        # exactly one tile
])
def test_indexer_scores(B, Q, T, first):
    cfg = dsa.default_config()
    q_idx, w, k_idx, pos = _indexer_inputs(B, Q, T, first, seed=11 + T)
    scores = torch.full((B, Q, T), float("nan"), device=DEV)
    dsa.indexer_scores(cfg, q_idx, w, k_idx, pos, scores)
    torch.cuda.synchronize()
    ora = oracle.indexer_scores(f64(q_idx), f64(w), f64(k_idx), pos.cpu().numpy())
    g = scores.cpu().double().numpy()
    for b in range(B):
        for t in range(Q):
            check_scores_row(g[b, t], ora[b, t], int(pos[b, t]))


def test_indexer_signed_weights_and_exact_zero():
    """Negative head weights are allowed; keys orthogonal to every head give 0."""
    cfg = dsa.default_config()
    B, Q, T = 1, 1, 640
    q_idx, w, k_idx, pos = _indexer_inputs(B, Q, T, T - 1, seed=5)
    w = (w - 0.5 / 64).contiguous()
    k_idx[0, 100:140] = 0
    scores = torch.empty(B, Q, T, device=DEV)
    dsa.indexer_scores(cfg, q_idx, w, k_idx, pos, scores)
    ora = oracle.indexer_scores(f64(q_idx), f64(w), f64(k_idx), pos.cpu().numpy())
    g = scores.cpu().double().numpy()
    assert np.all(g[0, 0, 100:140] == 0.0)
    err = np.abs(g[0, 0] - ora[0, 0])
    assert err.max() <= 2e-3 * np.abs(ora[0, 0]).max()


# --------------------------------------------------------------------------- a2: top-k

def _topk_case(scores_np, pos_np, k):
    cfg = dsa.default_config(topk=k)
    B, Q, T = scores_np.shape
    scores = torch.from_numpy(scores_np.astype(np.float32)).to(DEV)
    pos = torch.from_numpy(pos_np.astype(np.int32)).to(DEV)
    idx = torch.full((B, Q, k), -7, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1)
    dsa.topk_select(cfg, scores, pos, idx, ws)
    torch.cuda.synchronize()
    # the oracle sorts the same fp32 values (exactly representable in fp64)
    ora = oracle.topk_select(scores_np.astype(np.float32).astype(np.float64), pos_np, k)
    return idx.cpu().numpy(), ora


@pytest.mark.parametrize("B,Q,T,k,kind", [
    (2, 1, 100_000, 2048, "normal"),     # few long rows: chunked path
    (1, 3, 70_001, 2048, "ints"),        # heavy exact ties
    (1, 2, 50_000, 2048, "equal"),       # every score equal: pure tie-break
    (1, 320, 5000, 2048, "normal"),      # many rows: one block per row
    (1, 320, 3000, 700, "ints"),
    (1, 300, 13000, 2048, "equal"),      # many rows, candidates overflow shared memory: fallback passes
    (1, 300, 40_000, 2048, "normal"),    # long rows: the plan from a sample, one pass
    (1, 300, 40_000, 2048, "unsampled"), # the winners mostly outside the sampled runs
    (1, 300, 40_000, 2048, "sampled"),   # the winners only inside the sampled runs: the sample misjudges, exact steps
    (1, 296, 33_000, 2048, "equal"),     # long rows of one value: too many candidates, exact steps
    (1, 300, 12_000, 700, "ints"),       # long rows for a small k, heavy ties
    (4, 1, 9000, 7, "normal"),           # tiny k
    (2, 2, 1500, 2048, "normal"),        # L < k: -1 padding
])
def test_topk_bit_exact(B, Q, T, k, kind):
    rng = np.random.default_rng(T + k)
    if kind in ("normal", "unsampled", "sampled"):
        s = rng.standard_normal((B, Q, T))
        # one run of 32 scores in every 8 is sampled by the long-row plan
        in_sample = (np.arange(T) // 32) % 8 == 0
        if kind == "unsampled":
            boost = ~in_sample & (rng.random(T) < 0.05)
            s[..., boost] += 6.0
        elif kind == "sampled":
            boost = in_sample & (rng.random(T) < 0.4)
            s[..., boost] += 6.0
    elif kind == "ints":
        s = rng.integers(0, 50, (B, Q, T)).astype(np.float64)
    else:
        s = np.full((B, Q, T), 0.25)
    s[..., ::97] = -s[..., ::97]            # negative scores too
    s[..., 5] = 0.0
    s[..., 6] = -0.0                       # -0 and +0 tie
    pos = rng.integers(max(0, T - 3000), T, (B, Q))
    pos[0, 0] = T - 1
    g, o = _topk_case(s, pos, k)
    assert np.array_equal(g, o)


def test_topk_short_and_empty_rows():
    s = np.random.default_rng(0).standard_normal((1, 4, 4096))
    pos = np.array([[0, 10, 2047, 2048]])
    g, o = _topk_case(s, pos, 2048)
    assert np.array_equal(g, o)
    assert list(g[0, 0, :2]) == [0, -1]


# --------------------------------------------------------------------------- a3: sparse attention

def _attn_inputs(B, Q, T, k, seed, pad=0):
    q = wl.mla_queries(B, Q, seed, 0, DEV)
    kv = wl.latent_cache(B, T, seed, 0, DEV)
    rng = np.random.default_rng(seed)
    idx = np.full((B, Q, k), -1, dtype=np.int32)
    for b in range(B):
        for t in range(Q):
            n = k - pad if k - pad <= T else T
            idx[b, t, :n] = np.sort(rng.choice(T, n, replace=False))
    return q, kv, torch.from_numpy(idx).to(DEV)


@pytest.mark.parametrize("B,Q,T,k,pad", [
    (1, 1, 5000, 2048, 0),       # one row: many splits
    (2, 2, 9000, 2048, 37),      # padding slots
    (3, 1, 3000, 100, 0),        # ragged last block
    (1, 1, 40, 2048, 0),         # fewer rows than slots
    (40, 8, 2500, 256, 0),       # many rows: single split, no combine
])
def test_sparse_attention(B, Q, T, k, pad):
    cfg = dsa.default_config(topk=k)
    q, kv, idx = _attn_inputs(B, Q, T, k, seed=B * 1000 + T, pad=pad)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1)
    dsa.sparse_mla_attn(cfg, q, kv, idx, out, lse, ws)
    torch.cuda.synchronize()
    O, LSE = oracle.sparse_mla_attn(f64(q), f64(kv), idx.cpu().numpy(), SCALE)
    check_attention(f64(out), O)
    assert np.abs(lse.cpu().double().numpy() - LSE).max() < 1e-3


@pytest.mark.parametrize("B", [16, 32, 64])
def test_attention_split_units(B):
    """Units with 8, 4 and 2 splits (16, 32, 64 rows of k = 2048 on 148 SMs):
    where every unit's splits fit the GPU at once as one thread-block cluster,
    the cluster merges them itself; every row against the oracle, lse
    included."""
    cfg = dsa.default_config()
    Q, T, k = 1, 3000, 2048
    q, kv, idx = _attn_inputs(B, Q, T, k, seed=B + 5, pad=3)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=DEV)
    dsa.sparse_mla_attn(cfg, q, kv, idx, out, lse, dsa.alloc_workspace(cfg, B, Q, T, 1))
    torch.cuda.synchronize()
    O, LSE = oracle.sparse_mla_attn(f64(q), f64(kv), idx.cpu().numpy(), SCALE)
    check_attention(f64(out), O)
    assert np.abs(lse.cpu().double().numpy() - LSE).max() < 1e-3


def test_attention_last_wave_split():
    """More (layer, row) units than SMs, with a partial last wave: the units of
    that wave are split and merged by the combine while the others run whole.
    Every row against the oracle, lse included (one layer), and every row of a
    two-layer shared launch shaped the same way."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = (sms + 4) // 4 * 4 + (4 if (sms + 4) % 4 else 0)  # a full wave and a few more, a multiple of 4
    T, k = 3000, 2048
    cfg = dsa.default_config(topk=k)
    # one layer: units = rows
    B, Q = 2, units // 2
    q, kv, idx = _attn_inputs(B, Q, T, k, seed=units, pad=0)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=DEV)
    dsa.sparse_mla_attn(cfg, q, kv, idx, out, lse, dsa.alloc_workspace(cfg, B, Q, T, 1))
    torch.cuda.synchronize()
    O, LSE = oracle.sparse_mla_attn(f64(q), f64(kv), idx.cpu().numpy(), SCALE)
    check_attention(f64(out), O)
    assert np.abs(lse.cpu().double().numpy() - LSE).max() < 1e-3
    # two layers over one index set: units = 2 x rows
    B2, Q2 = 2, units // 4
    _, _, idx2 = _attn_inputs(B2, Q2, T, k, seed=units + 1, pad=0)
    q2 = [wl.mla_queries(B2, Q2, 62, layer, DEV) for layer in range(2)]
    kv2 = [wl.latent_cache(B2, T, 62, layer, DEV) for layer in range(2)]
    outs = [torch.empty(B2, Q2, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    dsa.sparse_mla_attn_shared(cfg, q2, kv2, idx2, outs, dsa.alloc_workspace(cfg, B2, Q2, T, 2))
    torch.cuda.synchronize()
    for layer in range(2):
        O2, _ = oracle.sparse_mla_attn(f64(q2[layer]), f64(kv2[layer]), idx2.cpu().numpy(), SCALE)
        check_attention(f64(outs[layer]), O2)


def test_sparse_attention_shared_layers():
    """Three layers over one shared index set (with padding slots) in one
    launch, each against the oracle on its own cache."""
    cfg = dsa.default_config(topk=1000)
    B, Q, T, n = 2, 3, 7000, 3
    _, _, idx = _attn_inputs(B, Q, T, 1000, seed=61, pad=9)
    q = [wl.mla_queries(B, Q, 61, layer, DEV) for layer in range(n)]
    kv = [wl.latent_cache(B, T, 61, layer, DEV) for layer in range(n)]
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    dsa.sparse_mla_attn_shared(cfg, q, kv, idx, outs, dsa.alloc_workspace(cfg, B, Q, T, n))
    torch.cuda.synchronize()
    for layer in range(n):
        O, _ = oracle.sparse_mla_attn(f64(q[layer]), f64(kv[layer]), idx.cpu().numpy(), SCALE)
        check_attention(f64(outs[layer]), O)


def test_attention_one_hot_and_empty_rows():
    cfg = dsa.default_config(topk=64)
    B, Q, T = 1, 2, 300
    kv = wl.latent_cache(B, T, 3, 0, DEV)
    q = torch.zeros(B, Q, 64, 576, dtype=torch.bfloat16, device=DEV)
    q[0, 0] = (kv[0, 123].float() * 0.5).to(torch.bfloat16)   # logit at row 123 dominates
    idx = torch.full((B, Q, 64), -1, dtype=torch.int32, device=DEV)
    idx[0, 0, :5] = torch.tensor([3, 50, 123, 200, 299], dtype=torch.int32)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, device=DEV)
    dsa.sparse_mla_attn(cfg, q, kv, idx, out, lse, dsa.alloc_workspace(cfg, B, Q, T, 1))
    torch.cuda.synchronize()
    O, _ = oracle.sparse_mla_attn(f64(q), f64(kv), idx.cpu().numpy(), SCALE)
    check_attention(f64(out), O)
    assert torch.all(out[0, 1] == 0)                         # no valid index: zeros
    assert torch.all(torch.isneginf(lse[0, 1]))


def test_bad_index_is_reported_not_faulted():
    cfg = dsa.default_config(topk=64)
    B, Q, T = 1, 1, 100
    q, kv, idx = _attn_inputs(B, Q, T, 64, seed=1)
    idx[0, 0, 3] = T + 5
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    dsa.sparse_mla_attn(cfg, q, kv, idx, out, None, dsa.alloc_workspace(cfg, B, Q, T, 1))
    assert dsa.get_device_error() == 6
    assert dsa.get_device_error() == 0        # cleared by the read


# --------------------------------------------------------------------------- a4/a6: group and MTP

def _workspace_scores(ws, B, Q, T):
    """The group's own indexer scores: a group call leaves them, [B, Q, T] fp32,
    at the start of its workspace (include/dsa.h)."""
    return ws[: B * Q * T * 4].view(torch.float32).view(B, Q, T)


def _group_check(w_, B=None, T=None, rows=None, score_rows=(), repeat=False):
    """Runs one group through the ABI and checks sampled rows against the oracle:
    the index set (boundary ties allowed) and every layer's output; for the rows
    in `score_rows` also the group's own scores element by element.  With
    `repeat`, a second group call on the same inputs must give bit-identical
    indices and outputs."""
    cfg = dsa.default_config(topk=w_.topk)
    inp = wl.make_inputs(w_, DEV, B=B, T=T)
    B, Q, T = inp.q_idx.shape[0], inp.q_idx.shape[1], inp.k_idx.shape[1]
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(w_.n_layers)]
    idx = torch.empty(B, Q, w_.topk, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, w_.n_layers)
    dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs, idx, ws)
    torch.cuda.synchronize()
    rows = rows if rows is not None else [(b, t) for b in range(B) for t in range(Q)]
    g_idx = idx.cpu().numpy()
    g_scores = {bt: _workspace_scores(ws, B, Q, T)[bt[0], bt[1]].cpu().double().numpy() for bt in score_rows}
    ties = 0
    for (b, t) in rows:
        pos = int(inp.q_pos[b, t])
        S = oracle.indexer_scores_row(f64(inp.q_idx[b, t]), f64(inp.w[b, t]), f64(inp.k_idx[b]), pos)
        if (b, t) in g_scores:
            check_scores_row(g_scores[(b, t)], S, pos)
        o_idx = oracle.topk_select_row(S, pos, w_.topk)
        ties += check_topk_row(g_idx[b, t], o_idx, S, pos, w_.topk)
        del S
        for layer in range(w_.n_layers):
            # attention over the oracle's own index set, gathering only those rows
            valid = o_idx[o_idx >= 0]
            rows_kv = f64(inp.kv[layer][b, torch.from_numpy(valid).to(DEV)])
            O, _ = oracle.sparse_mla_attn_row(f64(inp.q[layer][b, t]), rows_kv, np.arange(valid.size), SCALE)
            if np.array_equal(g_idx[b, t], o_idx):
                check_attention(f64(outs[layer][b, t]), O)
            else:
                # boundary ties swap a few rows: compare with the oracle on the GPU's set
                gv = g_idx[b, t][g_idx[b, t] >= 0]
                rows_g = f64(inp.kv[layer][b, torch.from_numpy(gv).to(DEV)])
                Og, _ = oracle.sparse_mla_attn_row(f64(inp.q[layer][b, t]), rows_g, np.arange(gv.size), SCALE)
                check_attention(f64(outs[layer][b, t]), Og)
    assert not (set(score_rows) - set(rows)), "score rows must be among the sampled rows"
    if repeat:
        outs2 = [torch.empty_like(o) for o in outs]
        idx2 = torch.empty_like(idx)
        dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs2, idx2, ws)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx2), "the index set differs between two identical group calls"
        for a, b_ in zip(outs, outs2):
            assert torch.equal(a, b_), "the outputs differ between two identical group calls"
    del inp, ws, outs
    return ties


def test_group_tiny_decode():
    _group_check(wl.TINY)


def test_group_equals_four_independent_layers():
    """IndexShare on the GPU: the group call equals four single-layer calls fed
    the group's index set, bit for bit."""
    w_ = wl.TINY
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    B, Q, T = 1, 4, w_.T
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    idx = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 4)
    dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs, idx, ws)
    ws1 = dsa.alloc_workspace(cfg, B, Q, T, 4)
    for layer in range(4):
        single = torch.empty_like(outs[layer])
        dsa.sparse_mla_attn(cfg, inp.q[layer], inp.kv[layer], idx, single, None, ws1)
        # the group launch may split the slots differently: compare within rounding
        d = (single.float() - outs[layer].float()).abs().max().item()
        assert d <= 4e-3, d
    # the shared-index entry point (one launch over the four layers, the
    # launch the group makes) gives the group's outputs bit for bit
    shared = [torch.empty_like(o) for o in outs]
    dsa.sparse_mla_attn_shared(cfg, inp.q, inp.kv, idx, shared, ws1)
    torch.cuda.synchronize()
    for a, b in zip(shared, outs):
        assert torch.equal(a, b)
    # and the group's index set is the standalone indexer + top-k
    scores = torch.empty(B, Q, T, device=DEV)
    dsa.indexer_scores(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, scores)
    idx2 = torch.empty_like(idx)
    dsa.topk_select(cfg, scores, inp.q_pos, idx2, ws1)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)


def _digit0_hist(scores_row: np.ndarray, L: int) -> np.ndarray:
    """Counts of the top 13 bits of the order-preserving key of each fp32 score
    (sign folded, -0 as +0) over positions [0, L): the top-k's first digit."""
    bits = (scores_row[:L].astype(np.float32) + np.float32(0.0)).view(np.uint32)
    key = np.where(bits & np.uint32(0x80000000), ~bits, bits | np.uint32(0x80000000))
    return np.bincount((key >> np.uint32(19)).astype(np.int64), minlength=8192)


@pytest.mark.parametrize("B,T,pattern", [
    (3, 50_000, "none"),
    (2, 120_000, "dup"),     # exact ties made by duplicated keys
    (5, 9_000, "dup"),
    (2, 120_000, "hot"),     # a few scaled-up keys dominate the row
    (3, 9_000, "short"),     # rows barely longer than k among long ones
])
def test_group_decode_topk_bit_exact(B, T, pattern):
    """One query per sequence over a long context: the group's index set (whose
    first histogram is counted inside the indexer) equals the oracle's top-k of
    the very same fp32 scores, bit for bit."""
    cfg = dsa.default_config()
    q_idx, w, k_idx, pos = _indexer_inputs(B, 1, T, T - 1, seed=T + B)
    if pattern == "dup":   # copy a block of keys elsewhere: identical scores at different positions
        k_idx[:, T // 2:T // 2 + 3000] = k_idx[:, 1000:4000]
        k_idx[:, T - 500:] = k_idx[:, 200:700]
    elif pattern == "hot":   # every 50th key scaled up 4x: their scores dominate
        k_idx[:, ::50] *= 4
    elif pattern == "short":
        pos[:, 0] = torch.tensor([T - 1, 2099, 2500], dtype=torch.int32, device=DEV)[:B]
    q = [wl.mla_queries(B, 1, 5, layer, DEV) for layer in range(4)]
    kv = [wl.latent_cache(B, T, 5, layer, DEV) for layer in range(4)]
    outs = [torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    idx = torch.empty(B, 1, 2048, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, 1, T, 4)
    dsa.indexshare_group_forward(cfg, q_idx, w, k_idx, pos, q, kv, outs, idx, ws)
    scores = torch.empty(B, 1, T, device=DEV)
    dsa.indexer_scores(cfg, q_idx, w, k_idx, pos, scores)
    torch.cuda.synchronize()
    ora = oracle.topk_select(scores.cpu().double().numpy(), pos.cpu().numpy(), 2048)
    assert np.array_equal(idx.cpu().numpy(), ora)
    # the histogram the indexer counted (it follows the scores in the
    # workspace, 256-byte aligned) is a count over each row's visible scores
    off = -(-B * T * 4 // 256) * 256
    hist = ws[off:off + B * 8192 * 4].view(torch.int32).view(B, 8192).cpu().numpy()
    g = _workspace_scores(ws, B, 1, T).cpu().numpy()
    for b in range(B):
        assert np.array_equal(hist[b], _digit0_hist(g[b, 0], int(pos[b, 0]) + 1)), b


@pytest.mark.parametrize("B,Q,T,keys", [
    (1, 4, 70_000, "equal"),     # four queries per group, every score of a row equal
    (2, 2, 50_000, "dup"),       # two queries per group
    (3, 7, 40_000, "dup"),       # ragged last group of four
    (1, 300, 40_000, "dup"),     # one block per row, the plan from a sample
    (1, 296, 70_000, "equal"),   # one block per row, one value: exact steps
])
def test_group_multi_query_topk_bit_exact(B, Q, T, keys):
    """Several queries per sequence: the group's index set equals the oracle's
    top-k of the very same fp32 scores, bit for bit."""
    cfg = dsa.default_config()
    q_idx, w, k_idx, pos = _indexer_inputs(B, Q, T, T - Q, seed=T + Q)
    if keys == "equal":     # every key the same: every visible score of a row in one bin
        k_idx[:] = k_idx[:, :1].clone()
    else:                   # identical scores at different positions
        k_idx[:, T // 2:T // 2 + 3000] = k_idx[:, 1000:4000]
        k_idx[:, T - 500:] = k_idx[:, 200:700]
    q = [wl.mla_queries(B, Q, 5, layer, DEV) for layer in range(4)]
    kv = [wl.latent_cache(B, T, 5, layer, DEV) for layer in range(4)]
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    idx = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 4)
    dsa.indexshare_group_forward(cfg, q_idx, w, k_idx, pos, q, kv, outs, idx, ws)
    torch.cuda.synchronize()
    g_scores = _workspace_scores(ws, B, Q, T).cpu().numpy()
    P = pos.cpu().numpy()
    ora = oracle.topk_select(g_scores.astype(np.float64), P, 2048)
    assert np.array_equal(idx.cpu().numpy(), ora)
    if keys == "equal":
        assert np.array_equal(ora[..., :2048], np.broadcast_to(np.arange(2048), ora.shape))


def test_group_is_deterministic():
    w_ = wl.TINY
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    res = []
    for _ in range(2):
        outs = [torch.empty(1, 4, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
        idx = torch.empty(1, 4, 2048, dtype=torch.int32, device=DEV)
        dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs, idx,
                                     dsa.alloc_workspace(cfg, 1, 4, w_.T, 4))
        res.append((idx.clone(), [o.clone() for o in outs]))
    torch.cuda.synchronize()
    assert torch.equal(res[0][0], res[1][0])
    for a, b in zip(res[0][1], res[1][1]):
        assert torch.equal(a, b)


def test_mtp_draft_small():
    cfg = dsa.default_config()
    B, T, S = 3, 6000, 7
    kv = wl.latent_cache(B, T, 9, 0, DEV)
    q_steps = wl.draft_queries(S, B, 9, DEV)
    rng = np.random.default_rng(9)
    idx0 = np.stack([np.sort(rng.choice(T, 2048, replace=False)) for _ in range(B)])[:, None, :].astype(np.int32)
    idx0_t = torch.from_numpy(idx0).to(DEV)
    out = torch.empty(S, B, 64, 512, dtype=torch.bfloat16, device=DEV)
    dsa.mtp_draft_attn(cfg, idx0_t, q_steps, kv, out, dsa.alloc_workspace(cfg, B, 1, T, S))
    torch.cuda.synchronize()
    O = oracle.mtp_draft_attn(idx0, f64(q_steps), f64(kv), SCALE)
    check_attention(f64(out), O)
    # one step at a time gives the same result
    one = torch.empty(1, B, 64, 512, dtype=torch.bfloat16, device=DEV)
    dsa.mtp_draft_attn(cfg, idx0_t, q_steps[2:3].contiguous(), kv, one, dsa.alloc_workspace(cfg, B, 1, T, 1))
    torch.cuda.synchronize()
    assert (one[0].float() - out[2].float()).abs().max().item() <= 4e-3


# --------------------------------------------------------------------------- full-size workloads (sampled rows)

def test_group_eight_layers_ragged():
    """The largest group the ABI takes (8 layers), with a ragged context and
    query positions that leave fewer than k visible keys for some rows."""
    import dataclasses
    w_ = dataclasses.replace(wl.TINY, name="eight_layers", B=2, Q=3, T=3001, first_pos=1000, n_layers=8, seed=777)
    _group_check(w_)


def test_full_verify_q8_sampled():
    """Multi-token verification: 8 query tokens per sequence (the last accepted
    token and 7 drafts) through one indexer pass, 4 layers, 128K context."""
    rows = [(0, 0), (0, 7), (3, 1), (6, 4), (9, 3), (12, 5), (15, 2), (15, 7)]
    _group_check(wl.VERIFY, rows=rows, score_rows=[(0, 0), (9, 3), (15, 7)])
    torch.cuda.empty_cache()


def test_full_decode_128k_sampled():
    rows = [(0, 0), (9, 0), (17, 0), (31, 0)]
    _group_check(wl.DECODE_128K, rows=rows, score_rows=[(0, 0), (31, 0)])
    torch.cuda.empty_cache()


def test_full_decode_1m_sampled_and_deterministic():
    """The headline workload: 4 of the 8 sequences against the oracle (two with
    every one of their 1M scores compared element by element), and a second
    group call bit-identical to the first (the fused histogram uses global
    atomics, whose order must not leak into the result)."""
    ties = _group_check(wl.DECODE_1M, rows=[(0, 0), (3, 0), (5, 0), (7, 0)], score_rows=[(0, 0), (7, 0)],
                        repeat=True)
    print("boundary ties at 1M:", ties)
    torch.cuda.empty_cache()


# prefill rows: the first and last query groups of four, the rows around the
# middle of the chunk, and 20 more spread over it (32 of 4096)
PREFILL_ROWS = sorted(set([0, 1, 2, 3, 2046, 2047, 2048, 2049, 4092, 4093, 4094, 4095]
                          + [int(x) for x in np.linspace(5, 4090, 20)]))
PREFILL_SCORE_ROWS = [0, 1, 3, 4, 1023, 1024, 2047, 2048, 2049, 3071, 3072, 4091, 4092, 4093, 4094, 4095]


def test_full_prefill_sampled():
    """Chunked prefill, 32 of the 4096 query rows against the oracle; 16 of
    them (the first and last query groups, around the middle and quarter
    points) with every score compared element by element: the four-query
    persistent indexer over 131072 keys with its unit ranges crossing groups."""
    assert len(PREFILL_ROWS) >= 32
    _group_check(wl.PREFILL, rows=[(0, t) for t in sorted(set(PREFILL_ROWS) | set(PREFILL_SCORE_ROWS))],
                 score_rows=[(0, t) for t in PREFILL_SCORE_ROWS])
    torch.cuda.empty_cache()


def test_full_mtp_sampled():
    w_ = wl.MTP
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    B, T = w_.B, w_.T
    scores = torch.empty(B, 1, T, device=DEV)
    idx0 = torch.empty(B, 1, 2048, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, 1, T, w_.mtp_steps)
    dsa.indexer_scores(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, scores)
    dsa.topk_select(cfg, scores, inp.q_pos, idx0, ws)
    out = torch.empty(w_.mtp_steps, B, 64, 512, dtype=torch.bfloat16, device=DEV)
    dsa.mtp_draft_attn(cfg, idx0, inp.q_steps, inp.kv[0], out, ws)
    torch.cuda.synchronize()
    g_idx = idx0.cpu().numpy()
    for b in (0, 9, 18, 27, 36, 45, 54, 63):
        S = oracle.indexer_scores_row(f64(inp.q_idx[b, 0]), f64(inp.w[b, 0]), f64(inp.k_idx[b]), T - 1)
        if b in (0, 63):
            check_scores_row(scores[b, 0].cpu().double().numpy(), S, T - 1)
        o_idx = oracle.topk_select_row(S, T - 1, 2048)
        check_topk_row(g_idx[b, 0], o_idx, S, T - 1, 2048)
        gv = g_idx[b, 0]
        rows = f64(inp.kv[0][b, torch.from_numpy(gv).to(DEV)])
        for s in range(w_.mtp_steps):
            O, _ = oracle.sparse_mla_attn_row(f64(inp.q_steps[s, b]), rows, np.arange(gv.size), SCALE)
            check_attention(f64(out[s, b]), O)
    torch.cuda.empty_cache()


def test_per_layer_indexer_variant():
    """Row a5 on the GPU: without IndexShare every layer runs its own indexer
    and top-k (four distinct indexers), the composite the benchmark times
    against the group; checked against oracle.per_layer_indexer_forward."""
    w_ = wl.TINY
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV, per_layer_indexers=True)
    B, Q, T = w_.B, w_.Q, w_.T
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1)
    scores = torch.empty(B, Q, T, device=DEV)
    idxs, outs = [], []
    for layer in range(w_.n_layers):
        idx = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
        out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
        dsa.indexer_scores(cfg, inp.idx_q[layer], inp.idx_w[layer], inp.idx_k[layer], inp.q_pos, scores)
        dsa.topk_select(cfg, scores, inp.q_pos, idx, ws)
        dsa.sparse_mla_attn(cfg, inp.q[layer], inp.kv[layer], idx, out, None, ws)
        idxs.append(idx)
        outs.append(out)
    torch.cuda.synchronize()
    pos = inp.q_pos.cpu().numpy()
    o_idxs, o_outs = oracle.per_layer_indexer_forward(
        [f64(x) for x in inp.idx_q], [f64(x) for x in inp.idx_w], [f64(x) for x in inp.idx_k], pos,
        [f64(q) for q in inp.q], [f64(kv) for kv in inp.kv], 2048, SCALE)
    for layer in range(w_.n_layers):
        S = oracle.indexer_scores(f64(inp.idx_q[layer]), f64(inp.idx_w[layer]), f64(inp.idx_k[layer]), pos)
        g = idxs[layer].cpu().numpy()
        for t in range(Q):
            check_topk_row(g[0, t], o_idxs[layer][0, t], S[0, t], int(pos[0, t]), 2048)
        if np.array_equal(g, o_idxs[layer]):
            ref = o_outs[layer]
        else:
            ref, _ = oracle.sparse_mla_attn(f64(inp.q[layer]), f64(inp.kv[layer]), g, SCALE)
        check_attention(f64(outs[layer]), ref)
    # four independent indexers: the layers do not all select the same set
    assert any(not torch.equal(idxs[0], idxs[layer]) for layer in range(1, w_.n_layers))
