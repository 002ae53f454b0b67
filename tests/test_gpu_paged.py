"""Paged caches (fixed-size pages in a pool, one block table per sequence).

A paged call reads exactly the rows its contiguous twin reads, in the same
order, so the results must match bit for bit.  Every paged entry point is
also compared with the oracle over the cache its pool stands for
(oracle.gather_pages), element by element at the parity tolerances.
"""
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


def _indexer_inputs(B, Q, T, first, seed):
    q_idx = wl.indexer_queries(B, Q, seed, DEV)
    w = wl.head_weights(B, Q, seed, DEV)
    k_idx = wl.indexer_keys(B, T, seed, DEV)
    pos = torch.arange(first, first + Q, dtype=torch.int32, device=DEV).unsqueeze(0).repeat(B, 1).contiguous()
    return q_idx, w, k_idx, pos


@pytest.mark.parametrize("B,Q,T,first,page", [
    (3, 1, 3001, 3000, 64),     # decode, ragged last page and tile
    (2, 4, 5000, 4990, 128),    # four queries per group
    (1, 9, 4100, 4000, 256),    # several groups, causal, pages of 256
])
def test_paged_indexer_equals_contiguous(B, Q, T, first, page):
    cfg = dsa.default_config()
    q_idx, w, k_idx, pos = _indexer_inputs(B, Q, T, first, seed=T + page)
    (k_pool,), table = wl.paginate([k_idx], page, seed=T)
    ref = torch.empty(B, Q, T, device=DEV)
    got = torch.full((B, Q, T), float("nan"), device=DEV)
    dsa.indexer_scores(cfg, q_idx, w, k_idx, pos, ref)
    dsa.indexer_scores_paged(cfg, q_idx, w, k_pool, table, pos, got)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    # and against the oracle over the cache the pool stands for
    k_o = oracle.gather_pages(f64(k_pool), table.cpu().numpy(), T)
    ora = oracle.indexer_scores(f64(q_idx), f64(w), k_o, pos.cpu().numpy())
    g = got.cpu().double().numpy()
    check_scores_row(g[0, Q - 1], ora[0, Q - 1], int(pos[0, Q - 1]))


@pytest.mark.parametrize("B,Q,T,k,page", [(2, 2, 9000, 2048, 64), (3, 1, 700, 2048, 128)])
def test_paged_attention_equals_contiguous(B, Q, T, k, page):
    cfg = dsa.default_config(topk=k)
    q = wl.mla_queries(B, Q, 7, 0, DEV)
    kv = wl.latent_cache(B, T, 7, 0, DEV)
    rng = np.random.default_rng(T)
    idx = np.full((B, Q, k), -1, dtype=np.int32)
    for b in range(B):
        for t in range(Q):
            n = min(k - 3, T)
            idx[b, t, :n] = np.sort(rng.choice(T, n, replace=False))
    idx = torch.from_numpy(idx).to(DEV)
    (kv_pool,), table = wl.paginate([kv], page, seed=T + 1)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1)
    ref = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    got = torch.empty_like(ref)
    ref_lse = torch.empty(B, Q, 64, device=DEV)
    got_lse = torch.empty_like(ref_lse)
    dsa.sparse_mla_attn(cfg, q, kv, idx, ref, ref_lse, ws)
    dsa.sparse_mla_attn_paged(cfg, q, kv_pool, table, idx, got, T, got_lse, ws)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(got_lse, ref_lse)
    # and against the oracle over the cache the pool stands for
    kv_o = oracle.gather_pages(f64(kv_pool), table.cpu().numpy(), T)
    O, LSE = oracle.sparse_mla_attn(f64(q), kv_o, idx.cpu().numpy(), wl.SM_SCALE)
    check_attention(f64(got), O)
    assert np.abs(got_lse.cpu().double().numpy() - LSE).max() < 1e-3


@pytest.mark.parametrize("B,Q,T,page", [(3, 1, 50_000, 64), (1, 4, 9000, 128)])
def test_paged_group_equals_contiguous(B, Q, T, page):
    import dataclasses
    w_ = dataclasses.replace(wl.TINY, name="paged", B=B, Q=Q, T=T, first_pos=T - Q, seed=T + page)
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    pools, table = wl.paginate([inp.k_idx] + inp.kv, page, seed=T)
    k_pool, kv_pools = pools[0], pools[1:]
    ws = dsa.alloc_workspace(cfg, B, Q, T, 4)
    outs_ref = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    outs_got = [torch.empty_like(o) for o in outs_ref]
    idx_ref = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
    idx_got = torch.empty_like(idx_ref)
    dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs_ref, idx_ref, ws)
    dsa.indexshare_group_forward_paged(cfg, inp.q_idx, inp.w, k_pool, inp.q_pos, inp.q, kv_pools, table, T, outs_got,
                                       idx_got, ws)
    torch.cuda.synchronize()
    assert torch.equal(idx_got, idx_ref)
    for a, b in zip(outs_got, outs_ref):
        assert torch.equal(a, b)
    # and against the oracle's group over the caches the pools stand for
    tab = table.cpu().numpy()
    pos = inp.q_pos.cpu().numpy()
    k_o = oracle.gather_pages(f64(k_pool), tab, T)
    kv_o = [oracle.gather_pages(f64(p_), tab, T) for p_ in kv_pools]
    S = oracle.indexer_scores(f64(inp.q_idx), f64(inp.w), k_o, pos)
    o_idx, o_outs, _ = oracle.indexshare_group_forward(f64(inp.q_idx), f64(inp.w), k_o, pos,
                                                       [f64(q) for q in inp.q], kv_o, 2048, wl.SM_SCALE)
    g_idx = idx_got.cpu().numpy()
    for b in range(B):
        for t in range(Q):
            check_topk_row(g_idx[b, t], o_idx[b, t], S[b, t], int(pos[b, t]), 2048)
    for layer in range(4):
        if np.array_equal(g_idx, o_idx):
            ref = o_outs[layer]
        else:   # boundary ties: the oracle's attention over the GPU's index set
            ref, _ = oracle.sparse_mla_attn(f64(inp.q[layer]), kv_o[layer], g_idx, wl.SM_SCALE)
        check_attention(f64(outs_got[layer]), ref)


def test_full_decode_128k_paged_equals_contiguous():
    """The 128K decode workload laid out in 64-row pages: the group's index set
    and all four layers' outputs equal the contiguous call's."""
    w_ = wl.DECODE_128K
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    B, Q, T = w_.B, w_.Q, w_.T
    pools, table = wl.paginate([inp.k_idx] + inp.kv, 64, seed=5)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 4)
    outs_ref = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    outs_got = [torch.empty_like(o) for o in outs_ref]
    idx_ref = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
    idx_got = torch.empty_like(idx_ref)
    dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs_ref, idx_ref, ws)
    dsa.indexshare_group_forward_paged(cfg, inp.q_idx, inp.w, pools[0], inp.q_pos, inp.q, pools[1:], table, T,
                                       outs_got, idx_got, ws)
    torch.cuda.synchronize()
    assert torch.equal(idx_got, idx_ref)
    for a, b in zip(outs_got, outs_ref):
        assert torch.equal(a, b)
    # sampled sequences against the oracle through the pools: the key cache of
    # sequence b and the pool row of each of its positions come from
    # oracle.gather_pages over b's block-table row
    tab = table.cpu().numpy()
    page = pools[0].shape[1]
    row_ids = np.arange(pools[0].shape[0] * page, dtype=np.int64).reshape(-1, page, 1)
    g_idx = idx_got.cpu().numpy()
    for b in (0, 13, 31):
        rows_b = torch.from_numpy(oracle.gather_pages(row_ids, tab[b:b + 1], T)[0, :, 0]).to(DEV)
        k_b = f64(pools[0].view(-1, 128)[rows_b])
        pos = int(inp.q_pos[b, 0])
        S = oracle.indexer_scores_row(f64(inp.q_idx[b, 0]), f64(inp.w[b, 0]), k_b, pos)
        o_idx = oracle.topk_select_row(S, pos, 2048)
        check_topk_row(g_idx[b, 0], o_idx, S, pos, 2048)
        gv = torch.from_numpy(g_idx[b, 0][g_idx[b, 0] >= 0]).to(DEV)
        for layer in range(4):
            kv_rows = f64(pools[1 + layer].view(-1, 576)[rows_b[gv.long()]])
            O, _ = oracle.sparse_mla_attn_row(f64(inp.q[layer][b, 0]), kv_rows, np.arange(gv.numel()), wl.SM_SCALE)
            check_attention(f64(outs_got[layer][b, 0]), O)
    del pools, inp
    torch.cuda.empty_cache()


def test_page_outside_the_pool_is_reported_not_faulted():
    cfg = dsa.default_config(topk=64)
    B, Q, T = 1, 1, 300
    q = wl.mla_queries(B, Q, 3, 0, DEV)
    kv = wl.latent_cache(B, T, 3, 0, DEV)
    (kv_pool,), table = wl.paginate([kv], 64, seed=3)
    table[0, 2] = kv_pool.shape[0] + 10          # a page the pool does not have
    idx = torch.arange(64, dtype=torch.int32, device=DEV).view(1, 1, 64) * 4
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    dsa.sparse_mla_attn_paged(cfg, q, kv_pool, table, idx, out, T, None, dsa.alloc_workspace(cfg, B, Q, T, 1))
    assert dsa.get_device_error() == 6
    q_idx, w, k_idx, pos = _indexer_inputs(B, 1, T, T - 1, seed=4)
    (k_pool,), table2 = wl.paginate([k_idx], 64, seed=4)
    table2[0, 1] = -3
    scores = torch.empty(B, 1, T, device=DEV)
    dsa.indexer_scores_paged(dsa.default_config(), q_idx, w, k_pool, table2, pos, scores)
    assert dsa.get_device_error() == 6
    assert dsa.get_device_error() == 0
