"""Float64 CPU oracle (test infrastructure; never on the product path)."""
from .dcp_oracle import (  # noqa: F401
    NEG_INF, attention, bf16_bits_to_f64, blocks_needed, merge, mla_attention,
    owner, paged_slot, scatter_gqa, scatter_mla, shard_capacity_tokens,
    shard_chunk, shard_starts, shard_token_range, sharded_attention,
    mtp_limits, mtp_attention, sharded_mtp_attention, e4m3_to_f64, fp8_kv,
)
