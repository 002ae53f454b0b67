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


def _fp8_group_check(w_, rows=None):
    cfg = dsa.default_config(topk=w_.topk)
    inp = wl.make_inputs(w_, DEV)
    B, Q, T = w_.B, w_.Q, w_.T
    q8, q_scale = wl.to_e4m3_rows(inp.q_idx)
    k8, k_scale = wl.to_e4m3_rows(inp.k_idx)
    outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(w_.n_layers)]
    idx = torch.empty(B, Q, w_.topk, dtype=torch.int32, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, w_.n_layers)
    dsa.indexshare_group_forward_fp8(cfg, q8, q_scale, inp.w, k8, k_scale, inp.q_pos, inp.q, inp.kv, outs, idx, ws)
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
            rows_kv = f64(inp.kv[layer][b, torch.from_numpy(gv).to(DEV)])
            O, _ = oracle.sparse_mla_attn_row(f64(inp.q[layer][b, t]), rows_kv, np.arange(gv.size), wl.SM_SCALE)
            check_attention(f64(outs[layer][b, t]), O)
    return ties


def test_fp8_group_decode():
    import dataclasses
    _fp8_group_check(dataclasses.replace(wl.DECODE_128K, name="fp8_small", B=3, T=50_000, first_pos=49_999))


def test_fp8_group_tiny():
    _fp8_group_check(wl.TINY)


def test_full_decode_1m_fp8_sampled():
    ties = _fp8_group_check(wl.DECODE_1M, rows=[(0, 0), (5, 0)])
    print("boundary ties at 1M (fp8):", ties)
    torch.cuda.empty_cache()
