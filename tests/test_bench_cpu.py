"""The benchmark's roofline denominators, written out from their definitions:
keys read once per group (bf16 256 B, FP8 128 + 4 B per key) plus the latent
rows each layer or draft step gathers (bf16 1152 B, FP8 656 B per row), and
the indexer's 2 x 64 x 128 FLOPs per causal (query, key) pair."""
import bench
from long_context_sparse_26_b300 import workloads as wl


def test_decode_1m_bytes():
    b = bench.algorithmic_bytes(wl.DECODE_1M, 8)
    assert b["indexer_keys"] == 8 * 1048576 * 256 == 2_147_483_648
    assert b["gathered_rows"] == 4 * 8 * 2048 * 1152 == 75_497_472
    assert b["total"] == b["indexer_keys"] + b["gathered_rows"]


def test_fp8_bytes():
    b = bench.algorithmic_bytes(wl.DECODE_1M, 8, fp8_keys=True, fp8_kv=True)
    assert b["indexer_keys"] == 8 * 1048576 * 132
    assert b["gathered_rows"] == 4 * 8 * 2048 * 656


def test_mtp_gathers_once_per_draft_step():
    w = wl.MTP
    b = bench.algorithmic_bytes(w, w.B)
    assert b["gathered_rows"] == w.mtp_steps * w.B * 2048 * 1152


def test_prefill_flops_count_causal_pairs():
    w = wl.PREFILL
    # query t at position first_pos + t sees first_pos + t + 1 keys (capped at T)
    pairs = sum(min(w.first_pos + t + 1, w.T) for t in range(w.Q))
    assert bench.indexer_flops(w, 1) == 2 * 64 * 128 * pairs == 8_658_687_623_168
