"""dcp_kv_append on the GPU is bit-exact against the oracle's CPU scatter.

The pools are canary-filled, every context token is written through
dcp_kv_append (many tokens per call), then the step's appended token (one
per sequence); the pools read back must equal the oracle's scatter of the
same tokens with the oracle's own routing and block tables, canaries
included.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sequence_sharded_decode_gb300 import configs, inputs
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

CANARY = 0x5A5A

CASES = [
    ("gqa_tiny", {}),
    ("gqa_tiny", dict(shards=3, ctx_fixed=100, block_size=32)),
    ("gqa_mid", dict(batch=3, ctx_kind="lognormal", median=700, sigma=1.0, ctx_lo=0, ctx_hi=3000, shards=5)),
    ("gqa_mid", dict(batch=2, q_heads=8, kv_heads=8, dk=64, dv=64, ctx_fixed=37, shards=16)),
    ("mla_decode", dict(batch=3, ctx_kind="fixed", ctx_fixed=777, shards=5)),
    ("mla_high_concurrency", dict(batch=4, median=900, ctx_lo=1, ctx_hi=4000, shards=3)),
]


def _expected_pools(wl):
    ctx = wl.ctx_lens()
    starts = O.shard_starts(ctx, wl.shards)
    blocks = O.blocks_needed(ctx, wl.shards, wl.block_size, 1)
    tables = inputs.block_tables(wl.seed + 1, blocks, wl.capacity_factor)
    seq = np.concatenate([np.full(int(L) + 1, b) for b, L in enumerate(ctx)])
    pos = np.concatenate([np.arange(int(L) + 1) for L in ctx])
    if wl.kind == configs.MLA:
        pools = [np.full((cap, wl.block_size, wl.dk), CANARY, dtype=np.uint16) for cap, _ in tables]
        lat = inputs.bf16_bits(inputs.kv_tokens(wl.seed, inputs.STREAM_LATENT, seq, pos, 1, wl.dk))
        O.scatter_mla(pools, starts, [t for _, t in tables], wl.block_size, seq, pos, lat[:, 0, :])
        return pools, None
    pk = [np.full((cap, wl.kv_heads, wl.block_size, wl.dk), CANARY, dtype=np.uint16) for cap, _ in tables]
    pv = [np.full((cap, wl.kv_heads, wl.block_size, wl.dv), CANARY, dtype=np.uint16) for cap, _ in tables]
    k = inputs.bf16_bits(inputs.kv_tokens(wl.seed, inputs.STREAM_K, seq, pos, wl.kv_heads, wl.dk))
    v = inputs.bf16_bits(inputs.kv_tokens(wl.seed, inputs.STREAM_V, seq, pos, wl.kv_heads, wl.dv))
    O.scatter_gqa(pk, pv, starts, [t for _, t in tables], wl.block_size, seq, pos, k, v)
    return pk, pv


@pytest.mark.parametrize("name,over", CASES)
def test_fill_and_append_bit_exact(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl, canary=CANARY, fill_chunk=517)  # odd chunk: calls cut across sequences
    st.append()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    pk, pv = _expected_pools(wl)
    for i, sh in enumerate(st.shards):
        got_k = inputs.bf16_bits(sh.k_pool)
        assert got_k.shape == pk[i].shape
        assert np.array_equal(got_k, pk[i]), f"K pool of shard {i} differs"
        if pv is not None:
            assert np.array_equal(inputs.bf16_bits(sh.v_pool), pv[i]), f"V pool of shard {i} differs"


def test_append_flags_bad_tables():
    wl = configs.get("gqa_tiny")
    st = DecodeState(wl, canary=CANARY, fill=False)
    before = [inputs.bf16_bits(s.k_pool).copy() for s in st.shards]
    # point sequence 0's last logical block of the last shard outside the pool
    tab = st.shards[-1].block_table
    tab[0, int(st.blocks_host[0, -1]) - 1] = st.shards[-1].k_pool.shape[0]
    st.append()
    torch.cuda.synchronize()
    assert int(st.err.item()) & 1  # DCP_DEVERR_BLOCK_RANGE
    for i, s in enumerate(st.shards):
        assert np.array_equal(inputs.bf16_bits(s.k_pool), before[i])  # nothing written anywhere
    # a position before shard 0 (negative) is flagged too
    st.err.zero_()
    st.positions.fill_(-3)
    st.append()
    torch.cuda.synchronize()
    assert int(st.err.item()) & 4  # DCP_DEVERR_POSITION
