"""Seeded synthetic workloads for DSA sparse attention with IndexShare.

This module only draws random tensors of the right shapes and distributions.
It holds none of the method's arithmetic (no scores, no selection, no
attention), so both the CUDA path and the CPU oracle can take their inputs
from it without sharing any computation.

Shapes and distributions follow the five decode / prefill / MTP workloads of
the GLM-5.2 DSA + IndexShare description (GLM-5.2 config: ``index_topk=2048``,
``index_topk_freq=4``, ``kv_lora_rank=512``, 64 attention heads, maximum
position 1048576):

* indexer queries ``q_idx`` [B, Q, 64, 128] and keys ``k_idx`` [B, T, 128]:
  N(0, 1)/sqrt(128), rounded to bf16.  3% of the cached positions of every
  sequence (exactly ``round(0.03*T)``, drawn without replacement) get ``2*u``
  added to their key, ``u`` being one random unit vector shared by the whole
  workload.  The per-coordinate std is sigma = 1/sqrt(128), so ``2*u`` is a
  displacement of 2*sigma*sqrt(128): twice the typical key norm.  Adding
  2*sigma*u literally would move q.k by a small fraction of its spread and
  would not make the top-k selection structured.
* head weights ``w`` [B, Q, 64]: U(0, 1)/64, fp32.
* MLA queries ``q`` [B, Q, 64, 576] and latent cache ``kv`` [B, T, 576] per
  layer: N(0, 1), bf16 (512 latent dims then 64 already-rotated RoPE dims).
* query positions ``q_pos`` [B, Q] int32.

Every tensor has its own seed, derived from (workload seed, tensor, layer,
step).  Values depend on the device's generator: a tensor drawn on the GPU is
not the one drawn on the CPU with the same seed, so parity checks always copy
one drawn tensor to both sides.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

N_IDX_HEADS = 64
IDX_DIM = 128
N_HEADS = 64
KV_LORA_RANK = 512
ROPE_DIM = 64
D_QK = KV_LORA_RANK + ROPE_DIM  # 576
D_V = KV_LORA_RANK              # 512
TOPK = 2048
TOPK_FREQ = 4                   # layers per IndexShare group
MTP_STEPS = 7
SM_SCALE = 1.0 / math.sqrt(D_QK)
BOOST_FRACTION = 0.03
BOOST_SCALE = 2.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.

    ``kind`` is "decode" (one IndexShare group over Q query tokens per
    sequence), "prefill" (a chunk of Q new tokens at the end of the context)
    or "mtp" (one indexer pass at the last position, then ``mtp_steps`` draft
    attentions that reuse its indices).
    """
    name: str
    kind: str
    B: int
    Q: int
    T: int
    first_pos: int          # q_pos[b, q] = first_pos + q
    n_layers: int = TOPK_FREQ
    mtp_steps: int = 0
    topk: int = TOPK
    seed: int = 0

    def q_positions(self) -> torch.Tensor:
        pos = torch.arange(self.first_pos, self.first_pos + self.Q, dtype=torch.int32)
        return pos.unsqueeze(0).expand(self.B, self.Q).contiguous()

    @property
    def rows(self) -> int:
        return self.B * self.Q

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["boost_fraction"] = BOOST_FRACTION
        return d


# The five workloads: tiny decode, 128K decode, 1M decode, chunked prefill, MTP.
TINY = Workload("tiny_decode_T8192", "decode", B=1, Q=4, T=8192, first_pos=8188, seed=100)
DECODE_128K = Workload("decode_B32_T131072", "decode", B=32, Q=1, T=131072, first_pos=131071, seed=200)
DECODE_1M = Workload("decode_B8_T1048576", "decode", B=8, Q=1, T=1048576, first_pos=1048575, seed=300)
PREFILL = Workload("prefill_Q4096_T131072", "prefill", B=1, Q=4096, T=131072, first_pos=126976, seed=400)
MTP = Workload("mtp_B64_T262144_S7", "mtp", B=64, Q=1, T=262144, first_pos=262143,
               n_layers=1, mtp_steps=MTP_STEPS, seed=500)

# Multi-token verification: each sequence's last accepted token plus 7 MTP
# draft tokens, scored through one indexer pass (8 query tokens per sequence)
# and 4 sparse layers over a 128K context.
VERIFY = Workload("verify_B16_Q8_T131072", "decode", B=16, Q=8, T=131072, first_pos=131064, seed=600)

WORKLOADS = {w.name: w for w in (TINY, DECODE_128K, DECODE_1M, PREFILL, MTP, VERIFY)}

_TENSOR_IDS = {"q_idx": 1, "k_idx": 2, "w": 3, "q": 4, "kv": 5, "boost_pos": 6, "boost_dir": 7, "q_step": 8}


def tensor_seed(base: int, tensor: str, layer: int = 0, step: int = 0) -> int:
    """Seed of one tensor: a fixed mix of the workload seed and the tensor's role."""
    return (base * 1_000_003 + _TENSOR_IDS[tensor] * 10_007 + layer * 101 + step * 7) & 0x7FFF_FFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def indexer_keys(B: int, T: int, seed: int, device="cpu", boost: bool = True) -> torch.Tensor:
    """k_idx [B, T, 128] bf16: N(0,1)/sqrt(128) with 3% of positions shifted by 2u."""
    k = torch.randn(B, T, IDX_DIM, generator=_gen(device, tensor_seed(seed, "k_idx")),
                    device=device, dtype=torch.float32)
    k.mul_(1.0 / math.sqrt(IDX_DIM))
    if boost and T > 0:
        u = torch.randn(IDX_DIM, generator=_gen(device, tensor_seed(seed, "boost_dir")),
                        device=device, dtype=torch.float32)
        u = u / u.norm()
        n_boost = int(round(BOOST_FRACTION * T))
        gp = _gen(device, tensor_seed(seed, "boost_pos"))
        for b in range(B):
            pos = torch.randperm(T, generator=gp, device=device)[:n_boost]
            k[b, pos] += BOOST_SCALE * u
    return k.to(torch.bfloat16)


def indexer_queries(B: int, Q: int, seed: int, device="cpu") -> torch.Tensor:
    """q_idx [B, Q, 64, 128] bf16: N(0,1)/sqrt(128)."""
    q = torch.randn(B, Q, N_IDX_HEADS, IDX_DIM, generator=_gen(device, tensor_seed(seed, "q_idx")),
                    device=device, dtype=torch.float32)
    return (q * (1.0 / math.sqrt(IDX_DIM))).to(torch.bfloat16)


def head_weights(B: int, Q: int, seed: int, device="cpu") -> torch.Tensor:
    """w [B, Q, 64] fp32: U(0,1)/64."""
    w = torch.rand(B, Q, N_IDX_HEADS, generator=_gen(device, tensor_seed(seed, "w")),
                   device=device, dtype=torch.float32)
    return w / N_IDX_HEADS


def mla_queries(B: int, Q: int, seed: int, layer: int = 0, device="cpu") -> torch.Tensor:
    """q [B, Q, 64, 576] bf16: N(0,1)."""
    return torch.randn(B, Q, N_HEADS, D_QK, generator=_gen(device, tensor_seed(seed, "q", layer)),
                       device=device, dtype=torch.bfloat16)


def latent_cache(B: int, T: int, seed: int, layer: int = 0, device="cpu") -> torch.Tensor:
    """kv [B, T, 576] bf16: N(0,1) (512 latent dims, then 64 rotated RoPE dims)."""
    return torch.randn(B, T, D_QK, generator=_gen(device, tensor_seed(seed, "kv", layer)),
                       device=device, dtype=torch.bfloat16)


def draft_queries(S: int, B: int, seed: int, device="cpu") -> torch.Tensor:
    """q_steps [S, B, 64, 576] bf16: an independent N(0,1) query per draft step."""
    out = torch.empty(S, B, N_HEADS, D_QK, device=device, dtype=torch.bfloat16)
    for s in range(S):
        out[s] = torch.randn(B, N_HEADS, D_QK, generator=_gen(device, tensor_seed(seed, "q_step", 0, s + 1)),
                             device=device, dtype=torch.bfloat16)
    return out


@dataclasses.dataclass
class Inputs:
    q_idx: torch.Tensor
    w: torch.Tensor
    k_idx: torch.Tensor
    q_pos: torch.Tensor
    q: list            # per layer [B, Q, 64, 576]   (decode / prefill)
    kv: list           # per layer [B, T, 576]
    q_steps: Optional[torch.Tensor] = None   # [S, B, 64, 576] (mtp)
    idx_q: Optional[list] = None             # per-layer indexer queries (per-layer variant)
    idx_w: Optional[list] = None
    idx_k: Optional[list] = None


def make_inputs(wl: Workload, device="cpu", per_layer_indexers: bool = False,
                B: Optional[int] = None, T: Optional[int] = None) -> Inputs:
    """Draw every tensor of a workload (optionally with a smaller B or T)."""
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    first = wl.first_pos if T == wl.T else T - (wl.T - wl.first_pos)
    pos = torch.arange(first, first + wl.Q, dtype=torch.int32)
    q_pos = pos.unsqueeze(0).expand(B, wl.Q).contiguous().to(device)
    q_idx = indexer_queries(B, wl.Q, wl.seed, device)
    w = head_weights(B, wl.Q, wl.seed, device)
    k_idx = indexer_keys(B, T, wl.seed, device)
    qs, kvs = [], []
    for layer in range(wl.n_layers):
        if wl.kind != "mtp":
            qs.append(mla_queries(B, wl.Q, wl.seed, layer, device))
        kvs.append(latent_cache(B, T, wl.seed, layer, device))
    q_steps = draft_queries(wl.mtp_steps, B, wl.seed, device) if wl.kind == "mtp" else None
    inp = Inputs(q_idx, w, k_idx, q_pos, qs, kvs, q_steps)
    if per_layer_indexers:
        inp.idx_q, inp.idx_w, inp.idx_k = per_layer_indexers_of(wl, q_idx, w, k_idx, device)
    return inp


def per_layer_indexers_of(wl: Workload, q_idx: torch.Tensor, w: torch.Tensor, k_idx: torch.Tensor,
                          device="cpu"):
    """Indexer inputs of every layer when each layer has its own indexer (no
    IndexShare): layer 0 keeps the given ones, layers 1.. draw their own."""
    B, Q, T = q_idx.shape[0], q_idx.shape[1], k_idx.shape[1]
    qs, ws, ks = [q_idx], [w], [k_idx]
    for layer in range(1, wl.n_layers):
        s = wl.seed + 17 * layer
        qs.append(indexer_queries(B, Q, s, device))
        ws.append(head_weights(B, Q, s, device))
        ks.append(indexer_keys(B, T, s, device))
    return qs, ws, ks


def paginate(caches, page_size: int, seed: int, spare_pages: int = 3):
    """Lays contiguous caches [B, T, D] (one per tensor, same B and T) out as
    pools [num_pages, page_size, D] in a random page order, with a shared
    block table [B, ceil(T / page_size)] int32 and a few spare pages no
    sequence uses.  Only moves data: the pools hold the same rows."""
    B, T = caches[0].shape[0], caches[0].shape[1]
    device = caches[0].device
    max_pages = (T + page_size - 1) // page_size
    num_pages = B * max_pages + spare_pages
    g = _gen("cpu", (seed * 7919 + page_size) & 0x7FFF_FFFF)
    perm = torch.randperm(num_pages, generator=g)[: B * max_pages].to(torch.int32)
    block_table = perm.view(B, max_pages).contiguous().to(device)
    pools = []
    for c in caches:
        pool = torch.zeros(num_pages, page_size, *c.shape[2:], dtype=c.dtype, device=device)
        padded = torch.zeros(B, max_pages * page_size, *c.shape[2:], dtype=c.dtype, device=device)
        padded[:, :T] = c
        pool[block_table.view(-1).long()] = padded.view(B * max_pages, page_size, *c.shape[2:])
        pools.append(pool)
    return pools, block_table


E4M3_MAX = 448.0


def to_e4m3_rows(x: torch.Tensor):
    """Stores x [..., 128] as FP8 E4M3 rows with one fp32 scale per row
    (amax / 448, 1 for an all-zero row): returns (codes uint8 [..., 128],
    scale fp32 [...]).  A storage format for the inputs; each row stands for
    codes * scale."""
    xf = x.float()
    amax = xf.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (xf / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.contiguous()


FP8_LATENT_ROW_BYTES = 656


def to_fp8_latent(kv: torch.Tensor) -> torch.Tensor:
    """Stores latent rows kv [B, T, 576] bf16 as FP8 latent rows [B, T, 656]
    uint8: dims 0..511 as E4M3 codes with one fp32 scale per 128-dim group
    (group amax / 448, 1 for an all-zero group) in bytes 512..527, and the 64
    RoPE dims unchanged as bf16 in bytes 528..655.  A storage format for the
    inputs (one sequence at a time, to bound the temporaries)."""
    B, T, D = kv.shape
    if D != 576 or kv.dtype != torch.bfloat16:
        raise ValueError("latent rows are [B, T, 576] bf16")
    out = torch.empty(B, T, FP8_LATENT_ROW_BYTES, dtype=torch.uint8, device=kv.device)
    for b in range(B):
        x = kv[b, :, :512].float().reshape(T, 4, 128)
        amax = x.abs().amax(dim=-1)
        scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        out[b, :, :512] = (x / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8).reshape(T, 512)
        out[b, :, 512:528] = scale.contiguous().view(torch.uint8).reshape(T, 16)
        out[b, :, 528:] = kv[b, :, 512:].contiguous().view(torch.uint8).reshape(T, 128)
        del x, amax, scale
    return out
