"""Pins for the CPU oracle: each checks it against something other than itself.

The pins are hand-worked fixtures (tests/golden, each with its citation),
closed forms, brute force on tiny inputs, the dense-attention special case
(k >= visible length) computed a different way, and invariants.  The last
test plants plausible mistakes in the oracle (on the CPU) and checks that at
least one pin catches each.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle.dsa_oracle as dsa_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _num(x):
    return -math.inf if x == "-inf" else float(x)


def _dense_attention(q, kv_visible, sm_scale, d_v):
    """Textbook dense attention softmax(scale q K^T) V with V the first d_v dims."""
    z = sm_scale * np.einsum("hd,nd->hn", q, kv_visible)
    return softmax(z, axis=1) @ kv_visible[:, :d_v], logsumexp(z, axis=1)


# ----------------------------------------------------------------------------
# pins (each takes the oracle module, so the mutation test can reuse them)
# ----------------------------------------------------------------------------

def pin_bf16_conversion(o):
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F80], dtype=np.uint16)
    got = o.bf16_bits_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 1.0078125 and got[3] == 0.0
    assert np.signbit(got[4]) and got[5] == math.inf
    # round to nearest, ties to even
    assert o.round_to_bf16(np.array([1.00390625]))[0] == 1.0
    assert o.round_to_bf16(np.array([1.01171875]))[0] == 1.015625
    assert o.round_to_bf16(np.array([1.0078125 + 1e-6]))[0] == 1.0078125


def pin_indexer_golden(o):
    g = _load("indexer_tiny.json")
    q = np.array(g["q_idx"])
    w = np.array(g["w"])
    k = np.array(g["k_idx"])
    for case in g["cases"]:
        got = o.indexer_scores_row(q, w, k, case["pos"])
        exp = np.array([_num(x) for x in case["scores"]])
        assert np.array_equal(got, exp), (case, got)
    # the batched entry point gives the same rows
    got = o.indexer_scores(q[None, None], w[None, None], k[None], np.array([[1]]))
    assert np.array_equal(got[0, 0], np.array([1.5, 4.5, -math.inf]))


def pin_indexer_closed_form(o):
    rng = np.random.default_rng(1)
    qv = rng.standard_normal(16)
    keys = np.stack([qv, -qv, 2 * qv])
    got = o.indexer_scores_row(qv[None, :], np.array([0.25]), keys, 2)
    n2 = float(qv @ qv)
    assert np.allclose(got, [0.25 * n2, 0.0, 0.5 * n2], rtol=1e-14, atol=0)


def pin_indexer_bruteforce(o):
    rng = np.random.default_rng(2)
    B, Q, H, D, T = 2, 3, 3, 5, 9
    q = rng.standard_normal((B, Q, H, D))
    w = rng.uniform(-1, 1, (B, Q, H))          # signed weights too: the formula is general
    k = rng.standard_normal((B, T, D))
    pos = np.array([[0, 4, 8], [8, 3, 12]])
    got = o.indexer_scores(q, w, k, pos)
    for b in range(B):
        for t in range(Q):
            for s in range(T):
                if s > pos[b, t]:
                    assert got[b, t, s] == -math.inf
                    continue
                ref = 0.0
                for j in range(H):
                    dot = sum(q[b, t, j, d] * k[b, s, d] for d in range(D))
                    ref += w[b, t, j] * (dot if dot > 0 else 0.0)
                assert abs(got[b, t, s] - ref) <= 1e-12 * (1 + abs(ref))


def pin_topk_golden(o):
    g = _load("topk_tiny.json")
    s = np.array(g["scores"], dtype=np.float64)
    for case in g["cases"]:
        got = o.topk_select_row(s, case["pos"], case["k"])
        assert list(got) == case["idx"], (case, got)
    ae = g["all_equal"]
    got = o.topk_select_row(np.full(ae["T"], 7.0), ae["pos"], ae["k"])
    assert list(got) == ae["idx"]


def _brute_topk(scores, pos, k):
    L = pos + 1
    n = min(k, L)
    winners = []
    for combo in itertools.combinations(range(L), n):
        chosen = set(combo)
        ok = all((scores[c] > scores[u]) or (scores[c] == scores[u] and c < u)
                 for c in chosen for u in range(L) if u not in chosen)
        if ok:
            winners.append(list(combo) + [-1] * (k - n))
    assert len(winners) == 1
    return winners[0]


def pin_topk_bruteforce(o):
    rng = np.random.default_rng(3)
    for trial in range(40):
        T = int(rng.integers(1, 11))
        k = int(rng.integers(1, 6))
        scores = rng.integers(0, 4, T).astype(np.float64)   # many exact ties
        if trial % 3 == 0:
            scores = rng.standard_normal(T)
        pos = int(rng.integers(0, T))
        got = o.topk_select_row(scores, pos, k)
        assert list(got) == _brute_topk(scores, pos, k), (scores, pos, k, got)
    # batched form agrees row by row and ignores scores past the position
    sc = rng.standard_normal((2, 2, 8))
    pos = np.array([[7, 2], [5, 0]])
    got = o.topk_select(sc, pos, 3)
    for b in range(2):
        for t in range(2):
            assert list(got[b, t]) == _brute_topk(sc[b, t], pos[b, t], 3)


def pin_topk_k_covers_row(o):
    s = np.random.default_rng(4).standard_normal(10)
    got = o.topk_select_row(s, 5, 10)
    assert list(got) == [0, 1, 2, 3, 4, 5] + [-1] * 4


def pin_attn_golden(o):
    g = _load("attn_tiny.json")
    q = np.array(g["q"])
    kv = np.array(g["kv"])
    for case in g["cases"]:
        O, lse = o.sparse_mla_attn_row(q, kv, np.array(case["idx"]), g["sm_scale"], g["d_v"])
        assert np.allclose(O, np.array(case["O"]), rtol=0, atol=1e-13), (case, O)
        exp_lse = np.array([_num(x) for x in case["lse"]])
        if np.isinf(exp_lse).all():
            assert np.isinf(lse).all() and (lse < 0).all()
        else:
            assert np.allclose(lse, exp_lse, rtol=0, atol=1e-13), (case, lse)


def pin_attn_dense_special_case(o):
    """k >= visible length: sparse attention is dense causal attention."""
    rng = np.random.default_rng(5)
    H, Dqk, Dv, T = 4, 12, 8, 20
    scale = 1 / math.sqrt(Dqk)
    kv = rng.standard_normal((T, Dqk))
    for pos in (0, 7, 13, 19):
        q = rng.standard_normal((H, Dqk)) * 2
        idx = np.full(T + 5, -1)
        idx[: pos + 1] = rng.permutation(pos + 1)
        rng.shuffle(idx)
        O, lse = o.sparse_mla_attn_row(q, kv, idx, scale, Dv)
        O_ref, lse_ref = _dense_attention(q, kv[: pos + 1], scale, Dv)
        assert np.allclose(O, O_ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)
    # batched entry point, two sequences with their own caches
    B, Q = 2, 2
    kvb = rng.standard_normal((B, T, Dqk))
    qb = rng.standard_normal((B, Q, H, Dqk))
    idx = np.tile(np.arange(T), (B, Q, 1))
    O, lse = o.sparse_mla_attn(qb, kvb, idx, scale, Dv)
    for b in range(B):
        for t in range(Q):
            O_ref, _ = _dense_attention(qb[b, t], kvb[b], scale, Dv)
            assert np.allclose(O[b, t], O_ref, rtol=1e-12, atol=1e-12)


def pin_attn_one_hot_and_identical(o):
    rng = np.random.default_rng(6)
    H, Dqk, Dv, T = 3, 10, 6, 16
    kv = rng.standard_normal((T, Dqk))
    target = 11
    # each head's query points hard at row `target`: its logit exceeds the rest by > 50
    idx = np.array([3, target, 0, 7, -1, 15])
    others = kv[[3, 0, 7, 15]] @ kv[target]
    c = 60.0 / (kv[target] @ kv[target] - others.max())
    q = np.tile(c * kv[target], (H, 1)) + 1e-3 * rng.standard_normal((H, Dqk))
    z = q @ kv[idx[idx >= 0]].T
    assert (z.max(axis=1) - np.sort(z, axis=1)[:, -2] > 50).all()
    O, _ = o.sparse_mla_attn_row(q, kv, idx, 1.0, Dv)
    assert np.allclose(O, np.tile(kv[target, :Dv], (H, 1)), atol=1e-12)
    # identical rows: output is that row's value, whatever the query
    same = np.tile(rng.standard_normal(Dqk), (T, 1))
    O, lse = o.sparse_mla_attn_row(rng.standard_normal((H, Dqk)), same, np.arange(5), 0.3, Dv)
    assert np.allclose(O, np.tile(same[0, :Dv], (H, 1)), atol=1e-14)


def pin_attn_permutation(o):
    rng = np.random.default_rng(7)
    kv = rng.standard_normal((30, 9))
    q = rng.standard_normal((2, 9))
    idx = rng.permutation(30)[:12]
    a, la = o.sparse_mla_attn_row(q, kv, idx, 0.4, 5)
    b, lb = o.sparse_mla_attn_row(q, kv, idx[::-1].copy(), 0.4, 5)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14) and np.allclose(la, lb, rtol=1e-13)


def _tiny_group_inputs(rng, B=2, Q=2, H_I=3, D_I=6, H=2, Dqk=10, T=24, n_layers=4):
    q_idx = rng.standard_normal((B, Q, H_I, D_I))
    w = rng.uniform(0, 1, (B, Q, H_I))
    k_idx = rng.standard_normal((B, T, D_I))
    q_pos = np.array([[T - 2, T - 1], [9, 17]])[:B, :Q]
    qs = [rng.standard_normal((B, Q, H, Dqk)) for _ in range(n_layers)]
    kvs = [rng.standard_normal((B, T, Dqk)) for _ in range(n_layers)]
    return q_idx, w, k_idx, q_pos, qs, kvs


def pin_group_reuses_one_index_set(o):
    """IndexShare: a group equals 4 independent sparse layers on the same indices."""
    rng = np.random.default_rng(8)
    q_idx, w, k_idx, q_pos, qs, kvs = _tiny_group_inputs(rng)
    k, scale, Dv = 5, 0.3, 6
    idx, outs, lses = o.indexshare_group_forward(q_idx, w, k_idx, q_pos, qs, kvs, k, scale, Dv)
    # the shared set is the indexer's top-k of layer 0's indexer, checked by brute force
    S = o.indexer_scores(q_idx, w, k_idx, q_pos)
    for b in range(2):
        for t in range(2):
            assert list(idx[b, t]) == _brute_topk(S[b, t], q_pos[b, t], k)
    for layer in range(4):
        O, lse = o.sparse_mla_attn(qs[layer], kvs[layer], idx, scale, Dv)
        assert np.array_equal(O, outs[layer]) and np.array_equal(lse, lses[layer])
        # and each layer is dense attention over exactly the selected rows
        for b in range(2):
            for t in range(2):
                rows = kvs[layer][b, idx[b, t][idx[b, t] >= 0]]
                O_ref, _ = _dense_attention(qs[layer][b, t], rows, scale, Dv)
                assert np.allclose(outs[layer][b, t], O_ref, rtol=1e-12, atol=1e-12)
    # with k >= the visible length the group is dense causal attention in every layer
    idx, outs, _ = o.indexshare_group_forward(q_idx, w, k_idx, q_pos, qs, kvs, 64, scale, Dv)
    for layer in range(4):
        for b in range(2):
            for t in range(2):
                O_ref, _ = _dense_attention(qs[layer][b, t], kvs[layer][b, : q_pos[b, t] + 1], scale, Dv)
                assert np.allclose(outs[layer][b, t], O_ref, rtol=1e-12, atol=1e-12)


def pin_per_layer_variant(o):
    rng = np.random.default_rng(9)
    q_idx, w, k_idx, q_pos, qs, kvs = _tiny_group_inputs(rng)
    # the per-layer variant fed four copies of one indexer reproduces the group
    idxs, outs = o.per_layer_indexer_forward([q_idx] * 4, [w] * 4, [k_idx] * 4, q_pos, qs, kvs, 5, 0.3, 6)
    gidx, gouts, _ = o.indexshare_group_forward(q_idx, w, k_idx, q_pos, qs, kvs, 5, 0.3, 6)
    for layer in range(4):
        assert np.array_equal(idxs[layer], gidx) and np.array_equal(outs[layer], gouts[layer])
    # with distinct indexers each layer's set is its own brute-force top-k
    others = [rng.standard_normal(k_idx.shape) for _ in range(4)]
    idxs, _ = o.per_layer_indexer_forward([q_idx] * 4, [w] * 4, others, q_pos, qs, kvs, 5, 0.3, 6)
    for layer in range(4):
        S = o.indexer_scores(q_idx, w, others[layer], q_pos)
        assert list(idxs[layer][1, 1]) == _brute_topk(S[1, 1], q_pos[1, 1], 5)


def pin_mtp_reuse_and_kv_share(o):
    rng = np.random.default_rng(10)
    S_steps, B, H, Dqk, Dv, T = 3, 2, 2, 10, 6, 15
    kv = rng.standard_normal((B, T, Dqk))
    q_steps = rng.standard_normal((S_steps, B, H, Dqk))
    # index set covering the whole cache: every step is dense attention over the target cache
    idx0 = np.tile(np.arange(T + 3) - 3, (B, 1, 1))      # includes -1 padding slots
    O = o.mtp_draft_attn(idx0, q_steps, kv, 0.25, Dv)
    for s in range(S_steps):
        for b in range(B):
            O_ref, _ = _dense_attention(q_steps[s, b], kv[b], 0.25, Dv)
            assert np.allclose(O[s, b], O_ref, rtol=1e-12, atol=1e-12)
    # a partial index set: each step attends to exactly those rows of its own sequence
    idx0 = np.stack([rng.permutation(T)[:4] for _ in range(B)])[:, None, :]
    O = o.mtp_draft_attn(idx0, q_steps, kv, 0.25, Dv)
    for s in range(S_steps):
        for b in range(B):
            O_ref, _ = _dense_attention(q_steps[s, b], kv[b, idx0[b, 0]], 0.25, Dv)
            assert np.allclose(O[s, b], O_ref, rtol=1e-12, atol=1e-12)


def pin_indexer_flops(o):
    """IndexShare: sharing one indexer over 4 layers divides its work by exactly 4."""
    T = 1 << 20
    shared = o.indexer_flops(T, 4, True)
    per_layer = o.indexer_flops(T, 4, False)
    assert shared == 2 * 64 * 128 * T == 17_179_869_184
    assert per_layer == 4 * shared


def pin_gather_pages(o):
    """A pool laid out by hand: pages in reverse order plus an unused page."""
    rng = np.random.default_rng(11)
    B, T, D, ps = 2, 7, 3, 3                      # 3 pages per sequence, the last one partial
    cache = rng.standard_normal((B, T, D))
    pool = np.full((7, ps, D), np.nan)            # page 6 is never used
    table = np.array([[5, 4, 3], [2, 1, 0]])
    for b in range(B):
        for s in range(T):
            pool[table[b, s // ps], s % ps] = cache[b, s]
    assert np.array_equal(o.gather_pages(pool, table, T), cache)
    # hand-checked rows: sequence 1, position 4 is page 1, row 1
    pool2 = np.arange(7 * ps * D, dtype=float).reshape(7, ps, D)
    got = o.gather_pages(pool2, table, T)
    assert np.array_equal(got[1, 4], pool2[1, 1]) and np.array_equal(got[0, 6], pool2[3, 0])


def pin_e4m3_decoding(o):
    """Values fixed by the E4M3 format: bias 7, 3 mantissa bits, subnormals, NaN at S.1111.111."""
    codes = np.array([0x00, 0x38, 0x3C, 0x40, 0x7E, 0x08, 0x01, 0x07, 0xB8, 0xFE, 0x80, 0x30, 0x77])
    want = [0.0, 1.0, 1.5, 2.0, 448.0, 2.0 ** -6, 2.0 ** -9, 7 * 2.0 ** -9, -1.0, -448.0, 0.0, 0.5, 240.0]
    got = o.e4m3_to_f64(codes)
    assert np.array_equal(got, np.array(want)), got
    assert np.signbit(got[10])                   # 0x80 is -0
    assert np.isnan(o.e4m3_to_f64(np.array([0x7F, 0xFF]))).all()
    # every finite code is a distinct value, and ordered codes of one sign are increasing
    pos = o.e4m3_to_f64(np.arange(0x00, 0x7F))
    assert np.all(np.diff(pos) > 0)


def pin_fp8_latent_rows(o):
    """A 656-byte FP8 latent row written byte by byte: codes, four group scales, bf16 RoPE dims."""
    import struct
    row = bytearray(656)
    codes = {0: 0x38, 127: 0x40, 128: 0x3C, 300: 0xB8, 511: 0x7E, 200: 0x01}   # 1, 2, 1.5, -1, 448, 2^-9
    for d, c in codes.items():
        row[d] = c
    row[512:528] = struct.pack("<4f", 0.5, 2.0, 0.25, 4.0)
    for j, bits in {0: 0x3F80, 10: 0x4049, 63: 0xC000}.items():             # 1.0, 3.140625, -2.0
        row[528 + 2 * j: 530 + 2 * j] = struct.pack("<H", bits)
    want = np.zeros(576)
    want[0], want[127], want[128], want[300], want[511], want[200] = 0.5, 1.0, 3.0, -0.25, 1792.0, 2.0 ** -9 * 2.0
    want[512], want[522], want[575] = 1.0, 3.140625, -2.0
    arr = np.frombuffer(bytes(row), dtype=np.uint8)
    got = o.fp8_latent_to_f64(arr)
    assert got.shape == (576,) and np.array_equal(got, want), np.nonzero(got != want)
    # leading dims are kept, rows decode independently
    two = np.stack([arr, np.zeros(656, np.uint8)]).reshape(2, 1, 656)
    g2 = o.fp8_latent_to_f64(two)
    assert g2.shape == (2, 1, 576) and np.array_equal(g2[0, 0], want) and not g2[1].any()


PINS = [
    pin_bf16_conversion, pin_indexer_golden, pin_indexer_closed_form, pin_indexer_bruteforce,
    pin_topk_golden, pin_topk_bruteforce, pin_topk_k_covers_row, pin_attn_golden,
    pin_attn_dense_special_case, pin_attn_one_hot_and_identical, pin_attn_permutation,
    pin_group_reuses_one_index_set, pin_per_layer_variant, pin_mtp_reuse_and_kv_share,
    pin_indexer_flops, pin_gather_pages, pin_e4m3_decoding, pin_fp8_latent_rows,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(dsa_oracle)


def test_context_figure_from_the_pages():
    """The pages' 2.9x whole-model FLOP cut at 1M is context only (parity unpinned).

    If only the indexer changed, (F_o + F_i) / (F_o + F_i / 4) = 2.9 means the
    indexer was F_i / F_o = 6.9 times the rest, about 87% of per-token FLOPs.
    """
    ratio = 2.9
    fi_over_fo = (ratio - 1) / (1 - ratio / 4)
    assert abs(fi_over_fo - 6.909) < 1e-3
    assert abs(fi_over_fo / (1 + fi_over_fo) - 0.8736) < 1e-3


# ----------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# ----------------------------------------------------------------------------

def _mut_relu_after_sum(q_idx, w, k_idx, pos):
    T = k_idx.shape[0]
    out = np.full(T, -np.inf)
    L = min(pos + 1, T)
    out[:L] = np.maximum(w @ (q_idx @ k_idx[:L].T), 0.0)
    return out


def _mut_mask_excludes_self(q_idx, w, k_idx, pos):
    T = k_idx.shape[0]
    out = np.full(T, -np.inf)
    L = min(pos, T)
    out[:L] = w @ np.maximum(q_idx @ k_idx[:L].T, 0.0)
    return out


def _mut_ties_to_higher(scores, pos, k):
    L = min(pos + 1, scores.shape[0])
    out = np.full(k, -1, dtype=np.int64)
    rev = scores[:L][::-1]
    order = (L - 1) - np.argsort(-rev, kind="stable")
    chosen = np.sort(order[: min(k, L)])
    out[: chosen.shape[0]] = chosen
    return out


def _mut_score_order(scores, pos, k):
    L = min(pos + 1, scores.shape[0])
    out = np.full(k, -1, dtype=np.int64)
    order = np.argsort(-scores[:L], kind="stable")[: min(k, L)]
    out[: order.shape[0]] = order
    return out


def _attn_variant(value_tail=False, ignore_scale=False, keep_pad=False, lse_no_max=False):
    def f(q, kv, idx, sm_scale, d_v=512):
        H = q.shape[0]
        valid = idx if keep_pad else idx[idx >= 0]
        if valid.shape[0] == 0:
            return np.zeros((H, d_v)), np.full(H, -np.inf)
        K = np.asarray(kv[valid], dtype=np.float64)
        z = (1.0 if ignore_scale else sm_scale) * (q @ K.T)
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        l = e.sum(axis=1, keepdims=True)
        V = K[:, -d_v:] if value_tail else K[:, :d_v]
        lse = np.log(l)[:, 0] if lse_no_max else (m + np.log(l))[:, 0]
        return (e / l) @ V, lse
    return f


def _mut_group_layer0_cache(q_idx, w, k_idx, q_pos, qs, kvs, k, sm_scale, d_v=512):
    idx = dsa_oracle.topk_select(dsa_oracle.indexer_scores(q_idx, w, k_idx, q_pos), q_pos, k)
    outs, lses = [], []
    for q_l in qs:
        O, lse = dsa_oracle.sparse_mla_attn(q_l, kvs[0], idx, sm_scale, d_v)
        outs.append(O)
        lses.append(lse)
    return idx, outs, lses


def _mut_mtp_first_sequence(idx0, q_steps, kv, sm_scale, d_v=512):
    S, B, H, _ = q_steps.shape
    idx = idx0.reshape(B, -1)
    O = np.empty((S, B, H, d_v))
    for s in range(S):
        for b in range(B):
            O[s, b], _ = dsa_oracle.sparse_mla_attn_row(q_steps[s, b], kv[0], idx[b], sm_scale, d_v)
    return O


def _mut_flops_per_layer_always(T, n_layers, share, n_heads=64, head_dim=128):
    return 2 * n_heads * head_dim * T * n_layers


def _mut_pages_row_major(pool, block_table, T):
    page_size = pool.shape[1]
    B = block_table.shape[0]
    s = np.arange(T)
    out = np.empty((B, T) + pool.shape[2:], dtype=pool.dtype)
    for b in range(B):
        out[b] = pool[block_table[b, s % block_table.shape[1]], s // block_table.shape[1]]
    return out


def _mut_fp8_groups_of_64(rows):
    r = np.asarray(rows, dtype=np.uint8)
    lead = r.shape[:-1]
    scales = np.ascontiguousarray(r[..., 512:528]).view("<f4").astype(np.float64)
    per_dim = scales[..., (np.arange(512) // 64) % 4]
    nope = dsa_oracle.e4m3_to_f64(r[..., :512]) * per_dim
    rope = dsa_oracle.bf16_bits_to_f64(np.ascontiguousarray(r[..., 528:656]).view("<u2"))
    return np.concatenate([nope.reshape(*lead, 512), rope], axis=-1)


MUTANTS = {
    "relu_after_head_sum": ("indexer_scores_row", _mut_relu_after_sum),
    "causal_mask_excludes_self": ("indexer_scores_row", _mut_mask_excludes_self),
    "ties_to_higher_position": ("topk_select_row", _mut_ties_to_higher),
    "indices_in_score_order": ("topk_select_row", _mut_score_order),
    "pad_with_zero": ("topk_select_row", None),
    "value_from_rope_tail": ("sparse_mla_attn_row", _attn_variant(value_tail=True)),
    "softmax_scale_dropped": ("sparse_mla_attn_row", _attn_variant(ignore_scale=True)),
    "padding_slots_attended": ("sparse_mla_attn_row", _attn_variant(keep_pad=True)),
    "lse_without_max": ("sparse_mla_attn_row", _attn_variant(lse_no_max=True)),
    "group_reads_layer0_cache": ("indexshare_group_forward", _mut_group_layer0_cache),
    "mtp_reads_first_sequence": ("mtp_draft_attn", _mut_mtp_first_sequence),
    "indexer_never_shared": ("indexer_flops", _mut_flops_per_layer_always),
    "pages_interleaved": ("gather_pages", _mut_pages_row_major),
    "e4m3_bias_8": ("e4m3_to_f64", lambda codes, _f=dsa_oracle.e4m3_to_f64: _f(codes) / 2.0),
    "fp8_latent_groups_of_64": ("fp8_latent_to_f64", _mut_fp8_groups_of_64),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    if name == "pad_with_zero":
        orig = dsa_oracle.topk_select_row
        def fn(scores, pos, k, _orig=orig):  # noqa: E306
            out = _orig(scores, pos, k)
            out[out < 0] = 0
            return out
    monkeypatch.setattr(dsa_oracle, attr, fn)
    caught = []
    for pin in PINS:
        try:
            pin(dsa_oracle)
        except Exception:  # an assertion, or a shape error from a broken step
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
