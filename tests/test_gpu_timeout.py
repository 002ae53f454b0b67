"""Bounded device waits that run out.

Every wait inside the library's kernels (an mbarrier phase: a tile landing, an
MMA completing, another warp's arrival) gives up after a time limit, records
DSA_ERR_TIMEOUT in the device error word and stops its block in step: copies
and MMAs still in flight are drained on the full limit and tensor memory is
freed after them, so nothing is left running when the block exits.  These
tests shorten the limit through dsa_set_wait_limit_ns so that the ordinary
waits of a valid call run out (no fault, no hang: the calls' inputs are
valid), check that the error word reports the timeout, and then check that a
call with the default limit on the same context is correct again.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_26_b300 import binding as dsa
from long_context_sparse_26_b300 import workloads as wl
from parity import check_attention, check_scores_row, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
TIMEOUT = 7      # DSA_ERR_TIMEOUT
SHORT_NS = 1     # every wait that is not complete at its first few polls gives up


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from long_context_sparse_26_b300.build import build_library
    build_library()
    dsa.lib()
    assert dsa.get_device_error() == 0
    yield
    dsa.set_wait_limit_ns(0)
    assert dsa.get_device_error() == 0


def _until_timeout(call, tries=3):
    """Runs `call` under the short limit until the error word reports a
    timeout (a wait whose phase completes within its first polls does not run
    out, so one call may finish cleanly); returns the statuses seen."""
    seen = []
    try:
        dsa.set_wait_limit_ns(SHORT_NS)
        for _ in range(tries):
            call()
            seen.append(dsa.get_device_error())
            if seen[-1] == TIMEOUT:
                break
    finally:
        dsa.set_wait_limit_ns(0)
    return seen


def test_attention_wait_runs_out_then_recovers():
    cfg = dsa.default_config()
    B, Q, T = 8, 1, 60_000
    q = wl.mla_queries(B, Q, 81, 0, DEV)
    kv = wl.latent_cache(B, T, 81, 0, DEV)
    rng = np.random.default_rng(81)
    idx = torch.from_numpy(np.stack([np.sort(rng.choice(T, 2048, replace=False)) for _ in range(B)])
                           [:, None, :].astype(np.int32)).to(DEV)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    ws = dsa.alloc_workspace(cfg, B, Q, T, 1)
    seen = _until_timeout(lambda: dsa.sparse_mla_attn(cfg, q, kv, idx, out, None, ws))
    assert seen[-1] == TIMEOUT, seen
    assert all(s in (0, TIMEOUT) for s in seen), seen
    # the default limit again: the same call is correct on the same context
    out.fill_(float("nan"))
    dsa.sparse_mla_attn(cfg, q, kv, idx, out, None, ws)
    assert dsa.get_device_error() == 0
    O, _ = oracle.sparse_mla_attn(f64(q), f64(kv), idx.cpu().numpy(), wl.SM_SCALE)
    check_attention(f64(out), O)


def test_indexer_wait_runs_out_then_recovers():
    cfg = dsa.default_config()
    B, Q, T = 2, 1, 300_000
    q_idx = wl.indexer_queries(B, Q, 82, DEV)
    w = wl.head_weights(B, Q, 82, DEV)
    k_idx = wl.indexer_keys(B, T, 82, DEV)
    pos = torch.full((B, Q), T - 1, dtype=torch.int32, device=DEV)
    scores = torch.empty(B, Q, T, device=DEV)
    seen = _until_timeout(lambda: dsa.indexer_scores(cfg, q_idx, w, k_idx, pos, scores))
    assert seen[-1] == TIMEOUT, seen
    scores.fill_(float("nan"))
    dsa.indexer_scores(cfg, q_idx, w, k_idx, pos, scores)
    assert dsa.get_device_error() == 0
    g = scores.cpu().double().numpy()
    for b in range(B):
        S = oracle.indexer_scores_row(f64(q_idx[b, 0]), f64(w[b, 0]), f64(k_idx[b]), T - 1)
        check_scores_row(g[b, 0], S, T - 1)


def test_group_wait_runs_out_then_recovers():
    """The whole group (indexer with its fused histogram, top-k, four layers):
    a timeout anywhere is reported, and the next group call equals one made
    before any timeout, bit for bit."""
    w_ = wl.TINY
    cfg = dsa.default_config()
    inp = wl.make_inputs(w_, DEV)
    B, Q, T = w_.B, w_.Q, w_.T
    ws = dsa.alloc_workspace(cfg, B, Q, T, 4)

    def run():
        outs = [torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
        idx = torch.empty(B, Q, 2048, dtype=torch.int32, device=DEV)
        dsa.indexshare_group_forward(cfg, inp.q_idx, inp.w, inp.k_idx, inp.q_pos, inp.q, inp.kv, outs, idx, ws)
        return idx, outs

    idx0, outs0 = run()
    assert dsa.get_device_error() == 0
    seen = _until_timeout(run)
    assert seen[-1] == TIMEOUT, seen
    idx1, outs1 = run()
    assert dsa.get_device_error() == 0
    assert torch.equal(idx0, idx1)
    for a, b in zip(outs0, outs1):
        assert torch.equal(a, b)
