"""CPU-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from long_context_sparse_26_b300 import binding
from long_context_sparse_26_b300.build import LIB, build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_library()
    assert os.path.exists(LIB)
    return binding.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("dsa_indexer_scores", "dsa_topk_select", "dsa_sparse_mla_attn", "dsa_indexshare_group_forward",
                 "dsa_mtp_draft_attn", "dsa_workspace_bytes", "dsa_status_string", "dsa_get_device_error"):
        assert name in syms
    assert set(syms) <= set(binding.EXPORTS) | {"dsa_config_default"}


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_default_config(L):
    cfg = binding.default_config()
    assert (cfg.n_idx_heads, cfg.idx_dim, cfg.topk, cfg.topk_freq, cfg.kv_lora_rank, cfg.rope_dim, cfg.n_heads,
            cfg.index_share_for_mtp) == (64, 128, 2048, 4, 512, 64, 64, 1)
    assert abs(cfg.sm_scale - 576 ** -0.5) < 1e-7


def test_status_strings(L):
    assert binding.status_string(0) == "DSA_OK"
    assert binding.status_string(7) == "DSA_ERR_TIMEOUT"


def _call_scores(L, cfg, ptrs, B=1, Q=1, T=16):
    return L.dsa_indexer_scores(ctypes.byref(cfg), *[ctypes.c_void_p(p) for p in ptrs[:4]], B, Q, T,
                                ctypes.c_void_p(ptrs[4]), None)


def test_host_validation_rejects_before_launch(L):
    cfg = binding.default_config()
    good = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000]   # never dereferenced: validation fails first
    bad_cfg = binding.default_config()
    bad_cfg.n_heads = 32
    assert _call_scores(L, bad_cfg, good) == 2            # unsupported shape constant
    bad_cfg = binding.default_config()
    bad_cfg.topk = 4096
    assert _call_scores(L, bad_cfg, good) == 2
    bad_cfg = binding.default_config()
    bad_cfg.sm_scale = -1.0
    assert _call_scores(L, bad_cfg, good) == 1
    assert _call_scores(L, cfg, [0] + good[1:]) == 1     # null pointer
    assert _call_scores(L, cfg, good, B=-1) == 1          # negative batch
    assert _call_scores(L, cfg, good, T=-5) == 1
    assert _call_scores(L, cfg, good, B=70000) == 1       # rows beyond the launch limit
    assert _call_scores(L, cfg, [0x1008] + good[1:]) == 3  # misaligned
    assert L.dsa_indexshare_group_forward(ctypes.byref(cfg), *[ctypes.c_void_p(p) for p in good[:4]], None, None, 9,
                                          1, 1, 16, None, None, None, 0, None) == 1   # 9 layers > 8
    cfg_nomtp = binding.default_config()
    cfg_nomtp.index_share_for_mtp = 0
    assert L.dsa_mtp_draft_attn(ctypes.byref(cfg_nomtp), *[ctypes.c_void_p(p) for p in good[:3]], 7, 1, 16,
                                ctypes.c_void_p(good[4]), None, 0, None) == 2


def test_empty_calls_are_a_no_op(L):
    """No query rows: DSA_OK at once, with null pointers that are never read."""
    cfg = binding.default_config()
    n = None
    assert L.dsa_indexer_scores(ctypes.byref(cfg), n, n, n, n, 0, 4, 16, n, n) == 0
    assert L.dsa_indexer_scores(ctypes.byref(cfg), n, n, n, n, 3, 0, 16, n, n) == 0
    assert L.dsa_topk_select(ctypes.byref(cfg), n, n, 0, 1, 16, n, n, 0, n) == 0
    assert L.dsa_sparse_mla_attn(ctypes.byref(cfg), n, n, n, 0, 1, 16, n, n, n, 0, n) == 0
    assert L.dsa_sparse_mla_attn_noalloc(ctypes.byref(cfg), n, n, n, 2, 0, 16, n, n, n) == 0
    assert L.dsa_indexshare_group_forward(ctypes.byref(cfg), n, n, n, n, n, n, 4, 0, 1, 16, n, n, n, 0, n) == 0
    assert L.dsa_mtp_draft_attn(ctypes.byref(cfg), n, n, n, 0, 4, 16, n, n, 0, n) == 0
    assert L.dsa_mtp_draft_attn(ctypes.byref(cfg), n, n, n, 7, 0, 16, n, n, 0, n) == 0
    assert binding.workspace_bytes(cfg, 0, 1, 16, 4) > 0
    assert binding.workspace_bytes(cfg, -1, 1, 16, 4) == 0


def test_paged_validation_rejects_before_launch(L):
    cfg = binding.default_config()
    vp = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(6)]
    pg = binding.DsaPages(0x7000, 10, 48, 4)           # page size not a multiple of 64
    assert L.dsa_indexer_scores_paged(ctypes.byref(cfg), vp[0], vp[1], vp[2], ctypes.byref(pg), vp[3], 1, 1, 100,
                                      vp[4], None) == 2
    pg = binding.DsaPages(0x7000, 10, 64, 1)           # max_pages * page_size < T
    assert L.dsa_indexer_scores_paged(ctypes.byref(cfg), vp[0], vp[1], vp[2], ctypes.byref(pg), vp[3], 1, 1, 100,
                                      vp[4], None) == 1
    pg = binding.DsaPages(0x7004, 10, 64, 4)           # misaligned block table
    assert L.dsa_sparse_mla_attn_paged(ctypes.byref(cfg), vp[0], vp[1], ctypes.byref(pg), vp[2], 1, 1, 100, vp[3],
                                       None, None, 0, None) == 3
    assert L.dsa_indexer_scores_paged(ctypes.byref(cfg), vp[0], vp[1], vp[2], None, vp[3], 1, 1, 100, vp[4],
                                      None) == 1     # no block table


def test_fp8_validation_rejects_before_launch(L):
    """The FP8 entry points check their extra arguments on the host first."""
    cfg = binding.default_config()
    n = None
    vp = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(8)]
    odd = ctypes.c_void_p(0x1004)
    # indexer: q_idx8, q_scale, w, k_idx8, k_scale, q_pos, B, Q, T, scores, stream
    assert L.dsa_indexer_scores_fp8(ctypes.byref(cfg), vp[0], n, vp[1], vp[2], vp[3], vp[4], 1, 1, 64, vp[5], n) == 1
    assert L.dsa_indexer_scores_fp8(ctypes.byref(cfg), vp[0], vp[1], vp[2], vp[3], odd, vp[4], 1, 1, 64, vp[5], n) == 3
    assert L.dsa_indexer_scores_fp8(ctypes.byref(cfg), n, n, n, n, n, n, 0, 1, 64, n, n) == 0
    # FP8 latent attention: q, kv8, idx, B, Q, T, out, lse, ws, ws_bytes, stream
    assert L.dsa_sparse_mla_attn_fp8(ctypes.byref(cfg), vp[0], n, vp[1], 1, 1, 64, vp[2], n, n, 0, n) == 1
    assert L.dsa_sparse_mla_attn_fp8(ctypes.byref(cfg), vp[0], odd, vp[1], 1, 1, 64, vp[2], n, n, 0, n) == 3
    assert L.dsa_sparse_mla_attn_fp8(ctypes.byref(cfg), n, n, n, 1, 0, 64, n, n, n, 0, n) == 0
    # groups: the scales are checked, then the layer count
    layers = (ctypes.c_void_p * 1)(0x9000)
    for fn in (L.dsa_indexshare_group_forward_fp8, L.dsa_indexshare_group_forward_fp8kv):
        assert fn(ctypes.byref(cfg), vp[0], n, vp[1], vp[2], vp[3], vp[4], layers, layers, 1, 1, 1, 64, layers,
                  n, n, 0, n) == 1                       # no query scales
        assert fn(ctypes.byref(cfg), vp[0], vp[1], vp[2], vp[3], odd, vp[4], layers, layers, 1, 1, 1, 64, layers,
                  n, n, 0, n) == 3                       # misaligned key scales
        assert fn(ctypes.byref(cfg), vp[0], vp[1], vp[2], vp[3], vp[5], vp[4], layers, layers, 9, 1, 1, 64, layers,
                  n, n, 0, n) == 1                       # 9 layers > 8
        assert fn(ctypes.byref(cfg), n, n, n, n, n, n, n, n, 4, 0, 1, 64, n, n, n, 0, n) == 0
