"""The workspace-free attention entry point (dsa_sparse_mla_attn_noalloc).

It exists for callers that cannot allocate device memory when they call the
library, so it takes its split-k scratch from a fixed array inside the
library instead of a caller workspace.  These tests call it through the C ABI
twice in a row and check each result against dsa_sparse_mla_attn on the same
inputs, within the attention tolerance the other parity tests use.  The file
is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from long_context_sparse_26_b300 import binding as dsa
from long_context_sparse_26_b300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
MAX_ABS, MEAN_ABS = 2e-2, 2e-3   # the attention tolerance of tests/parity.py


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from long_context_sparse_26_b300.build import build_library
    build_library()
    dsa.lib()


def _case(B, Q, T, k, seed):
    q = wl.mla_queries(B, Q, seed, 0, DEV)
    kv = wl.latent_cache(B, T, seed, 0, DEV)
    rng = np.random.default_rng(seed)
    idx = np.full((B, Q, k), -1, dtype=np.int32)
    for b in range(B):
        for t in range(Q):
            n = min(k - 5, T)
            idx[b, t, :n] = np.sort(rng.choice(T, n, replace=False))
    return q, kv, torch.from_numpy(idx).to(DEV)


def _compare(B, Q, T, k, seed):
    cfg = dsa.default_config(topk=k)
    q, kv, idx = _case(B, Q, T, k, seed)
    ref = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    ref_lse = torch.empty(B, Q, 64, device=DEV)
    dsa.sparse_mla_attn(cfg, q, kv, idx, ref, ref_lse, dsa.alloc_workspace(cfg, B, Q, T, 1))
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    dsa.sparse_mla_attn_noalloc(cfg, q, kv, idx, out, lse)
    torch.cuda.synchronize()
    assert dsa.get_device_error() == 0
    err = (out.float() - ref.float()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (lse - ref_lse).abs().max().item() < 1e-3


def test_noalloc_matches_workspace_entry_point_twice():
    # first call: 8 decode rows, the key range split over many blocks
    _compare(B=8, Q=1, T=20000, k=2048, seed=71)
    # second call reuses the same static scratch with a different shape
    _compare(B=2, Q=3, T=7000, k=1000, seed=72)


def test_noalloc_at_its_row_limit():
    # 64 rows: the scratch holds one partial per row, so the key range of each
    # row runs unsplit in one block (the edge of the partial-result limit)
    _compare(B=64, Q=1, T=9000, k=2048, seed=74)
    # 64 rows spread over several query tokens per sequence
    _compare(B=16, Q=4, T=5000, k=2048, seed=75)


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    cfg = dsa.default_config()
    q, kv, idx = _case(65, 1, 300, 2048, seed=73)
    out = torch.empty(65, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dsa.DsaError) as e:
        dsa.sparse_mla_attn_noalloc(cfg, q, kv, idx, out)
    assert e.value.status == 4  # DSA_ERR_WORKSPACE
