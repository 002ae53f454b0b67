"""Thin ctypes binding of libdsa (include/dsa.h), with the same names.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors are torch CUDA tensors (device memory and streams come from
PyTorch); each call enqueues on the current torch stream unless a stream is
given.  If libdsa.so is missing, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsa.so")

STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_ALIGNMENT",
          4: "DSA_ERR_WORKSPACE", 5: "DSA_ERR_CUDA", 6: "DSA_ERR_DEVICE_CHECK", 7: "DSA_ERR_TIMEOUT"}

# every symbol include/dsa.h declares
EXPORTS = ("dsa_config_default", "dsa_workspace_bytes", "dsa_indexer_scores", "dsa_topk_select",
           "dsa_sparse_mla_attn", "dsa_indexshare_group_forward", "dsa_mtp_draft_attn",
           "dsa_status_string", "dsa_get_device_error", "dsa_sparse_mla_attn_noalloc",
           "dsa_indexer_scores_paged", "dsa_sparse_mla_attn_paged", "dsa_indexshare_group_forward_paged",
           "dsa_indexer_scores_fp8", "dsa_indexshare_group_forward_fp8", "dsa_sparse_mla_attn_fp8",
           "dsa_indexshare_group_forward_fp8kv", "dsa_set_wait_limit_ns", "dsa_sparse_mla_attn_shared",
           "dsa_indexer_scores_fp8_paged", "dsa_sparse_mla_attn_fp8_paged", "dsa_indexshare_group_forward_fp8_paged",
           "dsa_indexshare_group_forward_fp8kv_paged")

FP8_LATENT_ROW_BYTES = 656  # 512 E4M3 codes, 4 fp32 group scales, 64 bf16 RoPE dims


class DsaConfig(ctypes.Structure):
    _fields_ = [("n_idx_heads", ctypes.c_int), ("idx_dim", ctypes.c_int), ("topk", ctypes.c_int),
                ("topk_freq", ctypes.c_int), ("kv_lora_rank", ctypes.c_int), ("rope_dim", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("sm_scale", ctypes.c_float), ("index_share_for_mtp", ctypes.c_int)]


class DsaPages(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("num_pages", ctypes.c_int), ("page_size", ctypes.c_int),
                ("max_pages", ctypes.c_int)]


class DsaError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what} failed: {STATUS.get(status, status)}")
        self.status = status


_lib = None
_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_CFG = ctypes.POINTER(DsaConfig)


def lib() -> ctypes.CDLL:
    """Loads libdsa.so (built in-tree by long_context_sparse_26_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m long_context_sparse_26_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.dsa_config_default.argtypes = [_CFG]
        L.dsa_config_default.restype = None
        L.dsa_workspace_bytes.argtypes = [_CFG, _I, _I, _I, _I]
        L.dsa_workspace_bytes.restype = _SZ
        L.dsa_indexer_scores.argtypes = [_CFG, _VP, _VP, _VP, _VP, _I, _I, _I, _VP, _VP]
        L.dsa_topk_select.argtypes = [_CFG, _VP, _VP, _I, _I, _I, _VP, _VP, _SZ, _VP]
        L.dsa_sparse_mla_attn.argtypes = [_CFG, _VP, _VP, _VP, _I, _I, _I, _VP, _VP, _VP, _SZ, _VP]
        L.dsa_indexshare_group_forward.argtypes = [_CFG, _VP, _VP, _VP, _VP, ctypes.POINTER(_VP),
                                                   ctypes.POINTER(_VP), _I, _I, _I, _I, ctypes.POINTER(_VP),
                                                   _VP, _VP, _SZ, _VP]
        L.dsa_mtp_draft_attn.argtypes = [_CFG, _VP, _VP, _VP, _I, _I, _I, _VP, _VP, _SZ, _VP]
        L.dsa_sparse_mla_attn_shared.argtypes = [_CFG, ctypes.POINTER(_VP), ctypes.POINTER(_VP), _I, _VP, _I, _I,
                                                 _I, ctypes.POINTER(_VP), _VP, _SZ, _VP]
        L.dsa_sparse_mla_attn_noalloc.argtypes = [_CFG, _VP, _VP, _VP, _I, _I, _I, _VP, _VP, _VP]
        _PG = ctypes.POINTER(DsaPages)
        L.dsa_indexer_scores_paged.argtypes = [_CFG, _VP, _VP, _VP, _PG, _VP, _I, _I, _I, _VP, _VP]
        L.dsa_sparse_mla_attn_paged.argtypes = [_CFG, _VP, _VP, _PG, _VP, _I, _I, _I, _VP, _VP, _VP, _SZ, _VP]
        L.dsa_indexshare_group_forward_paged.argtypes = [_CFG, _VP, _VP, _VP, _VP, ctypes.POINTER(_VP),
                                                         ctypes.POINTER(_VP), _I, _PG, _I, _I, _I,
                                                         ctypes.POINTER(_VP), _VP, _VP, _SZ, _VP]
        L.dsa_indexer_scores_fp8.argtypes = [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _VP, _VP]
        L.dsa_indexshare_group_forward_fp8.argtypes = [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(_VP),
                                                       ctypes.POINTER(_VP), _I, _I, _I, _I, ctypes.POINTER(_VP),
                                                       _VP, _VP, _SZ, _VP]
        L.dsa_sparse_mla_attn_fp8.argtypes = [_CFG, _VP, _VP, _VP, _I, _I, _I, _VP, _VP, _VP, _SZ, _VP]
        L.dsa_indexer_scores_fp8_paged.argtypes = [_CFG, _VP, _VP, _VP, _VP, _VP, _PG, _VP, _I, _I, _I, _VP, _VP]
        L.dsa_sparse_mla_attn_fp8_paged.argtypes = [_CFG, _VP, _VP, _PG, _VP, _I, _I, _I, _VP, _VP, _VP, _SZ, _VP]
        for name in ("dsa_indexshare_group_forward_fp8_paged", "dsa_indexshare_group_forward_fp8kv_paged"):
            getattr(L, name).argtypes = [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(_VP), ctypes.POINTER(_VP),
                                         _I, _PG, _I, _I, _I, ctypes.POINTER(_VP), _VP, _VP, _SZ, _VP]
        L.dsa_indexshare_group_forward_fp8kv.argtypes = [_CFG, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(_VP),
                                                         ctypes.POINTER(_VP), _I, _I, _I, _I, ctypes.POINTER(_VP),
                                                         _VP, _VP, _SZ, _VP]
        for name in ("dsa_indexer_scores", "dsa_topk_select", "dsa_sparse_mla_attn",
                     "dsa_indexshare_group_forward", "dsa_mtp_draft_attn", "dsa_get_device_error",
                     "dsa_sparse_mla_attn_noalloc", "dsa_indexer_scores_paged", "dsa_sparse_mla_attn_paged",
                     "dsa_indexshare_group_forward_paged", "dsa_indexer_scores_fp8",
                     "dsa_indexshare_group_forward_fp8", "dsa_sparse_mla_attn_fp8",
                     "dsa_indexshare_group_forward_fp8kv", "dsa_set_wait_limit_ns",
                     "dsa_sparse_mla_attn_shared", "dsa_indexer_scores_fp8_paged", "dsa_sparse_mla_attn_fp8_paged",
                     "dsa_indexshare_group_forward_fp8_paged", "dsa_indexshare_group_forward_fp8kv_paged"):
            getattr(L, name).restype = ctypes.c_int
        L.dsa_get_device_error.argtypes = [_VP]
        L.dsa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        L.dsa_set_wait_limit_ns.restype = ctypes.c_int
        L.dsa_status_string.argtypes = [ctypes.c_int]
        L.dsa_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def default_config(topk: int = 2048) -> DsaConfig:
    cfg = DsaConfig()
    lib().dsa_config_default(ctypes.byref(cfg))
    cfg.topk = topk
    return cfg


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor with {ndim} dims, got {t.dtype} {tuple(t.shape)}")


def _check(status: int, what: str):
    if status != 0:
        raise DsaError(what, status)


def workspace_bytes(cfg: DsaConfig, B: int, Q: int, T: int, n_layers: int) -> int:
    return int(lib().dsa_workspace_bytes(ctypes.byref(cfg), B, Q, T, n_layers))


def alloc_workspace(cfg: DsaConfig, B: int, Q: int, T: int, n_layers: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg, B, Q, T, n_layers)
    if n == 0:
        raise DsaError("dsa_workspace_bytes", 1)
    return torch.empty(n, dtype=torch.uint8, device=device)


def indexer_scores(cfg, q_idx, w, k_idx, q_pos, scores, stream=None):
    """q_idx [B,Q,64,128] bf16, w [B,Q,64] f32, k_idx [B,T,128] bf16, q_pos [B,Q] i32 -> scores [B,Q,T] f32."""
    _need(q_idx, "q_idx", torch.bfloat16, 4); _need(w, "w", torch.float32, 3)
    _need(k_idx, "k_idx", torch.bfloat16, 3); _need(q_pos, "q_pos", torch.int32, 2)
    _need(scores, "scores", torch.float32, 3)
    B, Q, T = q_idx.shape[0], q_idx.shape[1], k_idx.shape[1]
    _check(lib().dsa_indexer_scores(ctypes.byref(cfg), _p(q_idx), _p(w), _p(k_idx), _p(q_pos), B, Q, T,
                                    _p(scores), _s(stream)), "dsa_indexer_scores")


def topk_select(cfg, scores, q_pos, idx, ws=None, stream=None):
    """scores [B,Q,T] f32, q_pos [B,Q] i32 -> idx [B,Q,topk] i32."""
    _need(scores, "scores", torch.float32, 3); _need(q_pos, "q_pos", torch.int32, 2)
    _need(idx, "idx", torch.int32, 3)
    B, Q, T = scores.shape
    _check(lib().dsa_topk_select(ctypes.byref(cfg), _p(scores), _p(q_pos), B, Q, T, _p(idx), _p(ws),
                                 0 if ws is None else ws.numel(), _s(stream)), "dsa_topk_select")


def sparse_mla_attn(cfg, q, kv, idx, out, lse=None, ws=None, stream=None):
    """q [B,Q,64,576] bf16, kv [B,T,576] bf16, idx [B,Q,topk] i32 -> out [B,Q,64,512] bf16 (+ lse [B,Q,64] f32)."""
    _need(q, "q", torch.bfloat16, 4); _need(kv, "kv", torch.bfloat16, 3); _need(idx, "idx", torch.int32, 3)
    _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    B, Q, T = q.shape[0], q.shape[1], kv.shape[1]
    _check(lib().dsa_sparse_mla_attn(ctypes.byref(cfg), _p(q), _p(kv), _p(idx), B, Q, T, _p(out), _p(lse),
                                     _p(ws), 0 if ws is None else ws.numel(), _s(stream)), "dsa_sparse_mla_attn")


def sparse_mla_attn_noalloc(cfg, q, kv, idx, out, lse=None, stream=None):
    """Same as sparse_mla_attn, for callers that cannot allocate device memory:
    no workspace argument; the library's own fixed 16 MiB scratch is used
    instead.  At most 64 query rows (B * Q) per call; calls that run at the same
    time on one GPU share that scratch and must not overlap."""
    _need(q, "q", torch.bfloat16, 4); _need(kv, "kv", torch.bfloat16, 3); _need(idx, "idx", torch.int32, 3)
    _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    B, Q, T = q.shape[0], q.shape[1], kv.shape[1]
    _check(lib().dsa_sparse_mla_attn_noalloc(ctypes.byref(cfg), _p(q), _p(kv), _p(idx), B, Q, T, _p(out), _p(lse),
                                             _s(stream)), "dsa_sparse_mla_attn_noalloc")


def indexshare_group_forward(cfg, q_idx, w, k_idx, q_pos, qs: Sequence[torch.Tensor], kvs: Sequence[torch.Tensor],
                             outs: Sequence[torch.Tensor], idx_out=None, ws=None, stream=None):
    """One IndexShare group: one indexer + top-k, then len(qs) attention layers over the same indices."""
    _need(q_idx, "q_idx", torch.bfloat16, 4); _need(w, "w", torch.float32, 3)
    _need(k_idx, "k_idx", torch.bfloat16, 3); _need(q_pos, "q_pos", torch.int32, 2)
    n = len(qs)
    if len(kvs) != n or len(outs) != n:
        raise ValueError("qs, kvs and outs must have one tensor per layer")
    for i in range(n):
        _need(qs[i], f"q[{i}]", torch.bfloat16, 4); _need(kvs[i], f"kv[{i}]", torch.bfloat16, 3)
        _need(outs[i], f"out[{i}]", torch.bfloat16, 4)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, 3)
    B, Q, T = q_idx.shape[0], q_idx.shape[1], k_idx.shape[1]
    arr = _VP * n
    qa = arr(*[t.data_ptr() for t in qs])
    ka = arr(*[t.data_ptr() for t in kvs])
    oa = arr(*[t.data_ptr() for t in outs])
    _check(lib().dsa_indexshare_group_forward(ctypes.byref(cfg), _p(q_idx), _p(w), _p(k_idx), _p(q_pos), qa, ka, n,
                                              B, Q, T, oa, _p(idx_out), _p(ws), 0 if ws is None else ws.numel(),
                                              _s(stream)), "dsa_indexshare_group_forward")


def sparse_mla_attn_shared(cfg, qs: Sequence[torch.Tensor], kvs: Sequence[torch.Tensor], idx,
                           outs: Sequence[torch.Tensor], ws=None, stream=None):
    """len(qs) attention layers over one shared index set, in one launch:
    qs[l] [B,Q,64,576] bf16, kvs[l] [B,T,576] bf16, idx [B,Q,topk] i32 -> outs[l] [B,Q,64,512] bf16."""
    _need(idx, "idx", torch.int32, 3)
    n = len(qs)
    if len(kvs) != n or len(outs) != n:
        raise ValueError("qs, kvs and outs must have one tensor per layer")
    for i in range(n):
        _need(qs[i], f"q[{i}]", torch.bfloat16, 4); _need(kvs[i], f"kv[{i}]", torch.bfloat16, 3)
        _need(outs[i], f"out[{i}]", torch.bfloat16, 4)
    B, Q, T = qs[0].shape[0], qs[0].shape[1], kvs[0].shape[1]
    arr = _VP * n
    qa = arr(*[t.data_ptr() for t in qs])
    ka = arr(*[t.data_ptr() for t in kvs])
    oa = arr(*[t.data_ptr() for t in outs])
    _check(lib().dsa_sparse_mla_attn_shared(ctypes.byref(cfg), qa, ka, n, _p(idx), B, Q, T, oa, _p(ws),
                                            0 if ws is None else ws.numel(), _s(stream)),
           "dsa_sparse_mla_attn_shared")


def mtp_draft_attn(cfg, idx0, q_steps, kv, out, ws=None, stream=None):
    """idx0 [B,1,topk] i32, q_steps [S,B,64,576] bf16, kv [B,T,576] bf16 -> out [S,B,64,512] bf16."""
    _need(idx0, "idx0", torch.int32, 3); _need(q_steps, "q_steps", torch.bfloat16, 4)
    _need(kv, "kv", torch.bfloat16, 3); _need(out, "out", torch.bfloat16, 4)
    S, B, T = q_steps.shape[0], q_steps.shape[1], kv.shape[1]
    _check(lib().dsa_mtp_draft_attn(ctypes.byref(cfg), _p(idx0), _p(q_steps), _p(kv), S, B, T, _p(out), _p(ws),
                                    0 if ws is None else ws.numel(), _s(stream)), "dsa_mtp_draft_attn")


def pages_of(block_table: torch.Tensor, pool: torch.Tensor) -> DsaPages:
    """Block-table description of a paged pool [num_pages, page_size, row]."""
    _need(block_table, "block_table", torch.int32, 2)
    return DsaPages(block_table.data_ptr(), pool.shape[0], pool.shape[1], block_table.shape[1])


def indexer_scores_paged(cfg, q_idx, w, k_pool, block_table, q_pos, scores, stream=None):
    """indexer_scores over a paged key cache k_pool [num_pages, page_size, 128] bf16; T = scores.shape[2]."""
    _need(q_idx, "q_idx", torch.bfloat16, 4); _need(w, "w", torch.float32, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 3); _need(q_pos, "q_pos", torch.int32, 2)
    _need(scores, "scores", torch.float32, 3)
    pg = pages_of(block_table, k_pool)
    B, Q, T = q_idx.shape[0], q_idx.shape[1], scores.shape[2]
    _check(lib().dsa_indexer_scores_paged(ctypes.byref(cfg), _p(q_idx), _p(w), _p(k_pool), ctypes.byref(pg),
                                          _p(q_pos), B, Q, T, _p(scores), _s(stream)), "dsa_indexer_scores_paged")


def sparse_mla_attn_paged(cfg, q, kv_pool, block_table, idx, out, T, lse=None, ws=None, stream=None):
    """sparse_mla_attn over a paged latent cache kv_pool [num_pages, page_size, 576] bf16 of context T."""
    _need(q, "q", torch.bfloat16, 4); _need(kv_pool, "kv_pool", torch.bfloat16, 3)
    _need(idx, "idx", torch.int32, 3); _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    pg = pages_of(block_table, kv_pool)
    B, Q = q.shape[0], q.shape[1]
    _check(lib().dsa_sparse_mla_attn_paged(ctypes.byref(cfg), _p(q), _p(kv_pool), ctypes.byref(pg), _p(idx), B, Q, T,
                                           _p(out), _p(lse), _p(ws), 0 if ws is None else ws.numel(), _s(stream)),
           "dsa_sparse_mla_attn_paged")


def indexshare_group_forward_paged(cfg, q_idx, w, k_pool, q_pos, qs, kv_pools, block_table, T, outs, idx_out=None,
                                   ws=None, stream=None):
    """indexshare_group_forward over a paged key cache and paged latent caches sharing one block table."""
    _need(q_idx, "q_idx", torch.bfloat16, 4); _need(w, "w", torch.float32, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 3); _need(q_pos, "q_pos", torch.int32, 2)
    n = len(qs)
    if len(kv_pools) != n or len(outs) != n:
        raise ValueError("qs, kv_pools and outs must have one tensor per layer")
    for i in range(n):
        _need(qs[i], f"q[{i}]", torch.bfloat16, 4); _need(kv_pools[i], f"kv_pool[{i}]", torch.bfloat16, 3)
        _need(outs[i], f"out[{i}]", torch.bfloat16, 4)
        if kv_pools[i].shape[:2] != k_pool.shape[:2]:
            raise ValueError("every pool must have the key pool's pages")
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, 3)
    pg = pages_of(block_table, k_pool)
    B, Q = q_idx.shape[0], q_idx.shape[1]
    arr = _VP * n
    qa = arr(*[t.data_ptr() for t in qs])
    ka = arr(*[t.data_ptr() for t in kv_pools])
    oa = arr(*[t.data_ptr() for t in outs])
    _check(lib().dsa_indexshare_group_forward_paged(ctypes.byref(cfg), _p(q_idx), _p(w), _p(k_pool), _p(q_pos), qa,
                                                    ka, n, ctypes.byref(pg), B, Q, T, oa, _p(idx_out), _p(ws),
                                                    0 if ws is None else ws.numel(), _s(stream)),
           "dsa_indexshare_group_forward_paged")


def indexer_scores_fp8(cfg, q8, q_scale, w, k8, k_scale, q_pos, scores, stream=None):
    """FP8 indexer caches: q8 [B,Q,64,128] u8 + q_scale [B,Q,64] f32, k8 [B,T,128] u8 + k_scale [B,T] f32."""
    _need(q8, "q8", torch.uint8, 4); _need(q_scale, "q_scale", torch.float32, 3); _need(w, "w", torch.float32, 3)
    _need(k8, "k8", torch.uint8, 3); _need(k_scale, "k_scale", torch.float32, 2); _need(q_pos, "q_pos", torch.int32, 2)
    _need(scores, "scores", torch.float32, 3)
    B, Q, T = q8.shape[0], q8.shape[1], k8.shape[1]
    _check(lib().dsa_indexer_scores_fp8(ctypes.byref(cfg), _p(q8), _p(q_scale), _p(w), _p(k8), _p(k_scale), _p(q_pos),
                                        B, Q, T, _p(scores), _s(stream)), "dsa_indexer_scores_fp8")


def indexshare_group_forward_fp8(cfg, q8, q_scale, w, k8, k_scale, q_pos, qs, kvs, outs, idx_out=None, ws=None,
                                 stream=None):
    """One IndexShare group with FP8 indexer caches; the latent caches stay bf16."""
    _need(q8, "q8", torch.uint8, 4); _need(q_scale, "q_scale", torch.float32, 3); _need(w, "w", torch.float32, 3)
    _need(k8, "k8", torch.uint8, 3); _need(k_scale, "k_scale", torch.float32, 2); _need(q_pos, "q_pos", torch.int32, 2)
    n = len(qs)
    if len(kvs) != n or len(outs) != n:
        raise ValueError("qs, kvs and outs must have one tensor per layer")
    for i in range(n):
        _need(qs[i], f"q[{i}]", torch.bfloat16, 4); _need(kvs[i], f"kv[{i}]", torch.bfloat16, 3)
        _need(outs[i], f"out[{i}]", torch.bfloat16, 4)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, 3)
    B, Q, T = q8.shape[0], q8.shape[1], k8.shape[1]
    arr = _VP * n
    qa = arr(*[t.data_ptr() for t in qs])
    ka = arr(*[t.data_ptr() for t in kvs])
    oa = arr(*[t.data_ptr() for t in outs])
    _check(lib().dsa_indexshare_group_forward_fp8(ctypes.byref(cfg), _p(q8), _p(q_scale), _p(w), _p(k8), _p(k_scale),
                                                  _p(q_pos), qa, ka, n, B, Q, T, oa, _p(idx_out), _p(ws),
                                                  0 if ws is None else ws.numel(), _s(stream)),
           "dsa_indexshare_group_forward_fp8")


def get_device_error(stream=None) -> int:
    """Synchronizes the stream, reads and clears the device error word; returns the status code."""
    return int(lib().dsa_get_device_error(_s(stream)))


def set_wait_limit_ns(limit_ns: int) -> None:
    """Time limit of the kernels' bounded device waits (0: the default 2 s)."""
    _check(lib().dsa_set_wait_limit_ns(int(limit_ns)), "dsa_set_wait_limit_ns")


def status_string(status: int) -> str:
    return lib().dsa_status_string(status).decode()


def sm_scale() -> float:
    return 1.0 / math.sqrt(576)


def _need_fp8_latent(t, name):
    _need(t, name, torch.uint8, 3)
    if t.shape[2] != FP8_LATENT_ROW_BYTES:
        raise ValueError(f"{name}: FP8 latent rows are {FP8_LATENT_ROW_BYTES} bytes, got {t.shape[2]}")


def sparse_mla_attn_fp8(cfg, q, kv8, idx, out, lse=None, ws=None, stream=None):
    """q [B,Q,64,576] bf16, kv8 [B,T,656] u8 (FP8 latent rows), idx [B,Q,topk] i32 -> out [B,Q,64,512] bf16."""
    _need(q, "q", torch.bfloat16, 4); _need_fp8_latent(kv8, "kv8"); _need(idx, "idx", torch.int32, 3)
    _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    B, Q, T = q.shape[0], q.shape[1], kv8.shape[1]
    _check(lib().dsa_sparse_mla_attn_fp8(ctypes.byref(cfg), _p(q), _p(kv8), _p(idx), B, Q, T, _p(out), _p(lse),
                                         _p(ws), 0 if ws is None else ws.numel(), _s(stream)), "dsa_sparse_mla_attn_fp8")


def indexshare_group_forward_fp8kv(cfg, q8, q_scale, w, k8, k_scale, q_pos, qs, kv8s, outs, idx_out=None, ws=None,
                                   stream=None):
    """One IndexShare group with FP8 indexer caches and FP8 latent caches kv8s[l] [B,T,656] u8."""
    _need(q8, "q8", torch.uint8, 4); _need(q_scale, "q_scale", torch.float32, 3); _need(w, "w", torch.float32, 3)
    _need(k8, "k8", torch.uint8, 3); _need(k_scale, "k_scale", torch.float32, 2); _need(q_pos, "q_pos", torch.int32, 2)
    n = len(qs)
    if len(kv8s) != n or len(outs) != n:
        raise ValueError("qs, kv8s and outs must have one tensor per layer")
    for i in range(n):
        _need(qs[i], f"q[{i}]", torch.bfloat16, 4); _need_fp8_latent(kv8s[i], f"kv8[{i}]")
        _need(outs[i], f"out[{i}]", torch.bfloat16, 4)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, 3)
    B, Q, T = q8.shape[0], q8.shape[1], k8.shape[1]
    arr = _VP * n
    qa = arr(*[t.data_ptr() for t in qs])
    ka = arr(*[t.data_ptr() for t in kv8s])
    oa = arr(*[t.data_ptr() for t in outs])
    _check(lib().dsa_indexshare_group_forward_fp8kv(ctypes.byref(cfg), _p(q8), _p(q_scale), _p(w), _p(k8),
                                                    _p(k_scale), _p(q_pos), qa, ka, n, B, Q, T, oa, _p(idx_out),
                                                    _p(ws), 0 if ws is None else ws.numel(), _s(stream)),
           "dsa_indexshare_group_forward_fp8kv")


def _pages_of_pool(block_table: torch.Tensor, num_pages: int, page_size: int) -> DsaPages:
    _need(block_table, "block_table", torch.int32, 2)
    return DsaPages(block_table.data_ptr(), num_pages, page_size, block_table.shape[1])


def indexer_scores_fp8_paged(cfg, q8, q_scale, w, k8_pool, k_scale_pool, block_table, q_pos, scores, stream=None):
    """indexer_scores_fp8 over a paged FP8 key cache: k8_pool [num_pages, page_size, 128] u8 and
    k_scale_pool [num_pages, page_size] f32 sharing block_table; T = scores.shape[2]."""
    _need(q8, "q8", torch.uint8, 4); _need(q_scale, "q_scale", torch.float32, 3); _need(w, "w", torch.float32, 3)
    _need(k8_pool, "k8_pool", torch.uint8, 3); _need(k_scale_pool, "k_scale_pool", torch.float32, 2)
    _need(q_pos, "q_pos", torch.int32, 2); _need(scores, "scores", torch.float32, 3)
    if k_scale_pool.shape != k8_pool.shape[:2]:
        raise ValueError("the scale pool must have the code pool's pages")
    pg = _pages_of_pool(block_table, k8_pool.shape[0], k8_pool.shape[1])
    B, Q, T = q8.shape[0], q8.shape[1], scores.shape[2]
    _check(lib().dsa_indexer_scores_fp8_paged(ctypes.byref(cfg), _p(q8), _p(q_scale), _p(w), _p(k8_pool),
                                              _p(k_scale_pool), ctypes.byref(pg), _p(q_pos), B, Q, T, _p(scores),
                                              _s(stream)), "dsa_indexer_scores_fp8_paged")


def sparse_mla_attn_fp8_paged(cfg, q, kv8_pool, block_table, idx, out, T, lse=None, ws=None, stream=None):
    """sparse_mla_attn_fp8 over a paged FP8 latent cache kv8_pool [num_pages, page_size, 656] u8 of context T."""
    _need(q, "q", torch.bfloat16, 4); _need_fp8_latent(kv8_pool, "kv8_pool"); _need(idx, "idx", torch.int32, 3)
    _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    pg = _pages_of_pool(block_table, kv8_pool.shape[0], kv8_pool.shape[1])
    B, Q = q.shape[0], q.shape[1]
    _check(lib().dsa_sparse_mla_attn_fp8_paged(ctypes.byref(cfg), _p(q), _p(kv8_pool), ctypes.byref(pg), _p(idx), B,
                                               Q, T, _p(out), _p(lse), _p(ws), 0 if ws is None else ws.numel(),
                                               _s(stream)), "dsa_sparse_mla_attn_fp8_paged")


def _group_fp8_paged(fn, what, cfg, q8, q_scale, w, k8_pool, k_scale_pool, q_pos, qs, kv_pools, block_table, T, outs,
                     idx_out, ws, stream, fp8_kv):
    _need(q8, "q8", torch.uint8, 4); _need(q_scale, "q_scale", torch.float32, 3); _need(w, "w", torch.float32, 3)
    _need(k8_pool, "k8_pool", torch.uint8, 3); _need(k_scale_pool, "k_scale_pool", torch.float32, 2)
    _need(q_pos, "q_pos", torch.int32, 2)
    if k_scale_pool.shape != k8_pool.shape[:2]:
        raise ValueError("the scale pool must have the code pool's pages")
    n = len(qs)
    if len(kv_pools) != n or len(outs) != n:
        raise ValueError("qs, kv_pools and outs must have one tensor per layer")
    for i in range(n):
        _need(qs[i], f"q[{i}]", torch.bfloat16, 4)
        if fp8_kv:
            _need_fp8_latent(kv_pools[i], f"kv8_pool[{i}]")
        else:
            _need(kv_pools[i], f"kv_pool[{i}]", torch.bfloat16, 3)
        _need(outs[i], f"out[{i}]", torch.bfloat16, 4)
        if kv_pools[i].shape[:2] != k8_pool.shape[:2]:
            raise ValueError("every pool must have the key pool's pages")
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32, 3)
    pg = _pages_of_pool(block_table, k8_pool.shape[0], k8_pool.shape[1])
    B, Q = q8.shape[0], q8.shape[1]
    arr = _VP * n
    qa = arr(*[t.data_ptr() for t in qs])
    ka = arr(*[t.data_ptr() for t in kv_pools])
    oa = arr(*[t.data_ptr() for t in outs])
    _check(fn(ctypes.byref(cfg), _p(q8), _p(q_scale), _p(w), _p(k8_pool), _p(k_scale_pool), _p(q_pos), qa, ka, n,
              ctypes.byref(pg), B, Q, T, oa, _p(idx_out), _p(ws), 0 if ws is None else ws.numel(), _s(stream)), what)


def indexshare_group_forward_fp8_paged(cfg, q8, q_scale, w, k8_pool, k_scale_pool, q_pos, qs, kv_pools, block_table,
                                       T, outs, idx_out=None, ws=None, stream=None):
    """One IndexShare group with paged FP8 indexer caches and paged bf16 latent pools (one block table)."""
    _group_fp8_paged(lib().dsa_indexshare_group_forward_fp8_paged, "dsa_indexshare_group_forward_fp8_paged", cfg, q8,
                     q_scale, w, k8_pool, k_scale_pool, q_pos, qs, kv_pools, block_table, T, outs, idx_out, ws,
                     stream, False)


def indexshare_group_forward_fp8kv_paged(cfg, q8, q_scale, w, k8_pool, k_scale_pool, q_pos, qs, kv8_pools,
                                         block_table, T, outs, idx_out=None, ws=None, stream=None):
    """One IndexShare group with paged FP8 indexer caches and paged FP8 latent pools (one block table)."""
    _group_fp8_paged(lib().dsa_indexshare_group_forward_fp8kv_paged, "dsa_indexshare_group_forward_fp8kv_paged", cfg,
                     q8, q_scale, w, k8_pool, k_scale_pool, q_pos, qs, kv8_pools, block_table, T, outs, idx_out, ws,
                     stream, True)
