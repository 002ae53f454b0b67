"""CPU oracle (test infrastructure only; never on the product path)."""
from .dsa_oracle import (  # noqa: F401
    bf16_bits_to_f64,
    round_to_bf16,
    indexer_scores,
    indexer_scores_row,
    topk_select,
    topk_select_row,
    sparse_mla_attn,
    sparse_mla_attn_row,
    indexshare_group_forward,
    per_layer_indexer_forward,
    mtp_draft_attn,
    indexer_flops,
    gather_pages,
    e4m3_to_f64,
    fp8_latent_to_f64,
    FP8_LATENT_ROW_BYTES,
)
