"""FP8 (E4M3) indexer caches against the oracle on the rows they stand for
(decoded codes times their fp32 scales)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_26_b300 import binding as dsa
from long_context_sparse_26_b300 import workloads as wl
from parity import check_attention, check_scores_row, check_topk_row, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from long_context_sparse_26_b300.build import build_library
    build_library()
    dsa.lib()
    yield
    assert dsa.get_device_error() == 0


def _fp8_inputs(B, Q, T, first, seed):
    q8, q_scale = wl.to_e4m3_rows(wl.indexer_queries(B, Q, seed, DEV))
    k8, k_scale = wl.to_e4m3_rows(wl.indexer_keys(B, T, seed, DEV))
    w = wl.head_weights(B, Q, seed, DEV)
    pos = torch.arange(first, first + Q, dtype=torch.int32, device=DEV).unsqueeze(0).repeat(B, 1).contiguous()
    return q8, q_scale, w, k8, k_scale, pos


def _decoded(codes, scale):
    return oracle.e4m3_to_f64(codes.cpu().numpy()) * scale.cpu().double().numpy()[..., None]


# one query: 256-key units of two tiles; the cases put the position in either
# tile of a unit, leave units past it unloaded and end T inside either tile
@pytest.mark.parametrize("B,Q,T,first", [(2, 1, 3001, 3000), (3, 1, 5000, 1234), (2, 1, 700, 200), (1, 1, 257, 256),
                                         (1, 1, 256, 100), (1, 4, 2500, 2496), (1, 9, 4100, 4000)])
def test_fp8_indexer_scores(B, Q, T, first):
    cfg = dsa.default_config()
    q8, q_scale, w, k8, k_scale, pos = _fp8_inputs(B, Q, T, first, seed=T + Q)
    scores = torch.full((B, Q, T), float("nan"), device=DEV)
    dsa.indexer_scores_fp8(cfg, q8, q_scale, w, k8, k_scale, pos, scores)
    torch.cuda.synchronize()
    ora = oracle.indexer_scores(_decoded(q8, q_scale), f64(w), _decoded(k8, k_scale), pos.cpu().numpy())
    g = scores.cpu().double().numpy()
    for b in range(B):
        for t in range(Q):
            check_scores_row(g[b, t], ora[b, t], int(pos[b, t]))


def _fp8_group_check(w_, rows=None, fp8_kv=False):
    cfg = dsa.default_config(topk=w_.topk)
    inp = wl.make_inputs(w_, DEV)
    B, Q, T = w_.B, w_.Q, w_.T
    q8, q_scale = wl.to_e4m3_rows(inp.q_idx)
    k8, k_scale = wl.to_e4m3_rows(inp.k_idx)
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(w_.n_layers)]
    idx = torch.empty(B, Q, w_.topk, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, w_.n_layers)
    if fp8_kv:
        kv8s = [wl.to_fp8_latent(kv) for kv in inp.kv]
        inp.kv = None
        torch.cuda.empty_cache()
        dsa.indexshare_group_forward_fp8kv(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, kv8s, outs, idx,
                                           ws)
    else:
        dsa.indexshare_group_forward_fp8(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, inp.kv, outs, idx,
                                         ws)
    torch.cuda.synchronize()
    g_idx = idx.cpu().numpy()
    rows = rows if rows is not None else [(b, t) for b in range(B) for t in range(Q)]
    ties = 0
    for (b, t) in rows:
        pos = int(inp.q_pos[b, t])
        S = oracle.indexer_scores_row(_decoded(q8[b, t], q_scale[b, t]), f64(inp.w[b, t]),
                                      _decoded(k8[b], k_scale[b]), pos)
        o_idx = oracle.topk_select_row(S, pos, w_.topk)
        ties += check_topk_row(g_idx[b, t], o_idx, S, pos, w_.topk)
        gv = g_idx[b, t][g_idx[b, t] >= 0]
        for layer in range(w_.n_layers):
            sel = torch.from_numpy(gv).to(DEV)
            if fp8_kv:
                rows_kv = oracle.fp8_latent_to_f64(kv8s[layer][b, sel].cpu().numpy())
            else:
                rows_kv = f64(inp.kv[layer][b, sel])
            O, _ = oracle.sparse_mla_attn_row(f64(inp.q[layer][b, t]), rows_kv, np.arange(gv.size), wl.SM_SCALE)
            check_attention(f64(outs[layer][b, t]), O)
    return ties


def test_fp8_group_decode():
    import dataclasses
    _fp8_group_check(dataclasses.replace(wl.DECODE_128K, name="fp8_small", B=3, T=50_000, first_pos=49_999))


def test_fp8_group_tiny():
    _fp8_group_check(wl.TINY)


def test_fp8kv_group_decode():
    import dataclasses
    _fp8_group_check(dataclasses.replace(wl.DECODE_128K, name="fp8kv_small", B=3, T=50_000, first_pos=49_999),
                     fp8_kv=True)


def test_fp8kv_group_verify_small():
    import dataclasses
    _fp8_group_check(dataclasses.replace(wl.VERIFY, name="fp8kv_verify", B=2, T=20_000, first_pos=19_992),
                     fp8_kv=True)


# FP8 latent rows: one layer against the oracle on the values the rows stand for
@pytest.mark.parametrize("B,Q,T,k,pad", [
    (1, 1, 5000, 2048, 0),       # one row: many splits
    (2, 2, 9000, 2048, 37),      # padding slots
    (3, 1, 3000, 100, 0),        # ragged last block
    (1, 1, 40, 2048, 0),         # fewer rows than slots
    (40, 8, 2500, 256, 0),       # many rows: single split, no combine
    (32, 1, 3000, 2048, 3),      # four splits a row: merged by a cluster where they fit the GPU at once
])
def test_fp8_latent_attention(B, Q, T, k, pad):
    cfg = dsa.default_config(topk=k)
    seed = B * 1000 + T + 7
    q = wl.mla_queries(B, Q, seed, 0, DEV)
    kv8 = wl.to_fp8_latent(wl.latent_cache(B, T, seed, 0, DEV))
    rng = np.random.default_rng(seed)
    idx = np.full((B, Q, k), -1, dtype=np.int32)
    for b in range(B):
        for t in range(Q):
            n = k - pad if k - pad <= T else T
            idx[b, t, :n] = np.sort(rng.choice(T, n, replace=False))
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=DEV)
    dsa.sparse_mla_attn_fp8(cfg, q, kv8, torch.from_numpy(idx).to(DEV), out, lse,
                            dsa.alloc_workspace(cfg, B, Q, T, 1))
    torch.cuda.synchronize()
    O, LSE = oracle.sparse_mla_attn(f64(q), oracle.fp8_latent_to_f64(kv8.cpu().numpy()), idx, wl.SM_SCALE)
    check_attention(f64(out), O)
    assert np.abs(lse.cpu().double().numpy() - LSE).max() < 1e-3


def test_fp8_latent_zero_group_and_empty_row():
    """A row with an all-zero group (scale 1, codes 0; every other group's amax
    is the largest code, 448 x scale), and a query row with no valid slot."""
    cfg = dsa.default_config(topk=64)
    B, Q, T = 1, 2, 300
    kv = wl.latent_cache(B, T, 5, 0, DEV)
    kv[0, 10, :128] = 0
    kv8 = wl.to_fp8_latent(kv)
    assert int(kv8[0, 10, :128].max()) == 0 and (kv8[0, 11, :128] & 0x7F).max() == 0x7E
    q = wl.mla_queries(B, Q, 5, 0, DEV)
    idx = torch.full((B, Q, 64), -1, dtype=torch.int32, device=DEV)
    idx[0, 0, :6] = torch.tensor([0, 10, 11, 150, 298, 299], dtype=torch.int32)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, device=DEV)
    dsa.sparse_mla_attn_fp8(cfg, q, kv8, idx, out, lse, dsa.alloc_workspace(cfg, B, Q, T, 1))
    torch.cuda.synchronize()
    O, _ = oracle.sparse_mla_attn(f64(q), oracle.fp8_latent_to_f64(kv8.cpu().numpy()), idx.cpu().numpy(),
                                  wl.SM_SCALE)
    check_attention(f64(out[:, :1]), O[:, :1])
    assert torch.all(out[0, 1] == 0)
    assert torch.all(torch.isneginf(lse[0, 1]))


def test_full_decode_1m_fp8_sampled():
    ties = _fp8_group_check(wl.DECODE_1M, rows=[(0, 0), (5, 0)])
    print("boundary ties at 1M (fp8):", ties)
    torch.cuda.empty_cache()


def test_full_decode_1m_fp8kv_sampled():
    ties = _fp8_group_check(wl.DECODE_1M, rows=[(2, 0), (7, 0)], fp8_kv=True)
    print("boundary ties at 1M (fp8 caches):", ties)
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- FP8 caches in pages

@pytest.mark.parametrize("B,Q,T,first,page", [
    (3, 1, 3001, 3000, 64),     # 256-key units over 64-row pages, ragged last page
    (2, 1, 5000, 1234, 128),    # a position inside a unit
    (1, 4, 2500, 2496, 256),    # four queries per group
])
def test_fp8_paged_indexer(B, Q, T, first, page):
    """Paged FP8 key codes and scales equal the contiguous FP8 call bit for bit,
    and the oracle over the cache the pools stand for."""
    cfg = dsa.default_config()
    q8, q_scale, w, k8, k_scale, pos = _fp8_inputs(B, Q, T, first, seed=T + page)
    (k8_pool, ks_pool), table = wl.paginate([k8, k_scale], page, seed=T)
    ref = torch.empty(B, Q, T, device=DEV)
    got = torch.full((B, Q, T), float("nan"), device=DEV)
    dsa.indexer_scores_fp8(cfg, q8, q_scale, w, k8, k_scale, pos, ref)
    dsa.indexer_scores_fp8_paged(cfg, q8, q_scale, w, k8_pool, ks_pool, table, pos, got)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    tab = table.cpu().numpy()
    k_o = oracle.gather_pages(oracle.e4m3_to_f64(k8_pool.cpu().numpy()), tab, T) * \
        oracle.gather_pages(ks_pool.cpu().double().numpy()[..., None], tab, T)
    ora = oracle.indexer_scores(_decoded(q8, q_scale), f64(w), k_o, pos.cpu().numpy())
    g = got.cpu().double().numpy()
    for b in range(B):
        for t in range(Q):
            check_scores_row(g[b, t], ora[b, t], int(pos[b, t]))


def test_fp8_paged_attention():
    cfg = dsa.default_config()
    B, Q, T, page = 2, 2, 9000, 64
    q = wl.mla_queries(B, Q, 17, 0, DEV)
    kv8 = wl.to_fp8_latent(wl.latent_cache(B, T, 17, 0, DEV))
    rng = np.random.default_rng(17)
    idx = np.full((B, Q, 2048), -1, dtype=np.int32)
    for b in range(B):
        for t in range(Q):
            idx[b, t, :2040] = np.sort(rng.choice(T, 2040, replace=False))
    idx = torch.from_numpy(idx).to(DEV)
    (kv8_pool,), table = wl.paginate([kv8], page, seed=17)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1)
    ref = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    got = torch.empty_like(ref)
    ref_lse = torch.empty(B, Q, 64, device=DEV)
    got_lse = torch.empty_like(ref_lse)
    dsa.sparse_mla_attn_fp8(cfg, q, kv8, idx, ref, ref_lse, ws)
    dsa.sparse_mla_attn_fp8_paged(cfg, q, kv8_pool, table, idx, got, T, got_lse, ws)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(got_lse, ref_lse)
    kv_o = oracle.fp8_latent_to_f64(oracle.gather_pages(kv8_pool.cpu().numpy(), table.cpu().numpy(), T))
    O, _ = oracle.sparse_mla_attn(f64(q), kv_o, idx.cpu().numpy(), wl.SM_SCALE)
    check_attention(f64(got), O)


@pytest.mark.parametrize("fp8_kv", [False, True])
def test_fp8_paged_group(fp8_kv):
    """The group with paged FP8 indexer caches (and paged bf16 or FP8 latent
    pools) equals the contiguous FP8 group bit for bit, and the oracle's group
    over the decoded caches the pools stand for."""
    import dataclasses
    B, Q, T, page = 2, 2, 20_000, 128
    w_ = dataclasses.replace(wl.TINY, name="fp8_paged", B=B, Q=Q, T=T, first_pos=T - Q, seed=91)
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    q8, q_scale = wl.to_e4m3_rows(inp.q_idx)
    k8, k_scale = wl.to_e4m3_rows(inp.k_idx)
    kvs = [wl.to_fp8_latent(kv) for kv in inp.kv] if fp8_kv else inp.kv
    pools, table = wl.paginate([k8, k_scale] + kvs, page, seed=91)
    k8_pool, ks_pool, kv_pools = pools[0], pools[1], pools[2:]
    ws = dsa.alloc_workspace(cfg, B, Q, T, 4)
    outs_ref = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    outs_got = [torch.empty_like(o) for o in outs_ref]
    idx_ref = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
    idx_got = torch.empty_like(idx_ref)
    if fp8_kv:
        dsa.indexshare_group_forward_fp8kv(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, kvs, outs_ref,
                                           idx_ref, ws)
        dsa.indexshare_group_forward_fp8kv_paged(cfg, q8, q_scale, inp.w, k8_pool, ks_pool, inp.q_pos, inp.q,
                                                 kv_pools, table, T, outs_got, idx_got, ws)
    else:
        dsa.indexshare_group_forward_fp8(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, kvs, outs_ref,
                                         idx_ref, ws)
        dsa.indexshare_group_forward_fp8_paged(cfg, q8, q_scale, inp.w, k8_pool, ks_pool, inp.q_pos, inp.q,
                                               kv_pools, table, T, outs_got, idx_got, ws)
    torch.cuda.synchronize()
    assert torch.equal(idx_got, idx_ref)
    for a, b in zip(outs_got, outs_ref):
        assert torch.equal(a, b)
    tab = table.cpu().numpy()
    pos = inp.q_pos.cpu().numpy()
    k_o = oracle.gather_pages(oracle.e4m3_to_f64(k8_pool.cpu().numpy()), tab, T) * \
        oracle.gather_pages(ks_pool.cpu().double().numpy()[..., None], tab, T)
    S = oracle.indexer_scores(_decoded(q8, q_scale), f64(inp.w), k_o, pos)
    o_idx = oracle.topk_select(S, pos, 2048)
    g_idx = idx_got.cpu().numpy()
    for b in range(B):
        for t in range(Q):
            check_topk_row(g_idx[b, t], o_idx[b, t], S[b, t], int(pos[b, t]), 2048)
    for layer in range(4):
        if fp8_kv:
            kv_o = oracle.fp8_latent_to_f64(oracle.gather_pages(kv_pools[layer].cpu().numpy(), tab, T))
        else:
            kv_o = oracle.gather_pages(f64(kv_pools[layer]), tab, T)
        ref, _ = oracle.sparse_mla_attn(f64(inp.q[layer]), kv_o, g_idx, wl.SM_SCALE)
        check_attention(f64(outs_got[layer]), ref)
