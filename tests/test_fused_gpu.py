"""Steps 2 and 3 in one call (dcp_attention_all: GQA: per-shard partial
attention, then one pass merging every output row's pieces across shards and
split ranges; MLA: the attention kernel merges the shards itself) against the
float64 oracle, and against the two-call path (partial + dcp_merge) on the
same device state."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_mtp_sequence, oracle_sequence
from sequence_sharded_decode_gb300 import configs
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

RAGGED = dict(batch=5, ctx_kind="lognormal", median=300, sigma=1.2, ctx_lo=0, ctx_hi=3000)
CASES = [
    ("gqa_tiny", 1, dict()),
    ("gqa_tiny", 1, dict(shards=16, **RAGGED)),                                  # empty shards
    ("gqa_mid", 1, dict(batch=3, ctx_fixed=3000, shards=2)),
    ("gqa_mid", 1, dict(batch=2, q_heads=64, kv_heads=2, ctx_fixed=999, shards=3)),  # two head groups
    ("gqa_mid", 2, dict(batch=2, ctx_fixed=1500, shards=3)),                     # teams of two tokens
    ("gqa_mid", 4, dict(batch=2, ctx_fixed=1500, shards=3)),                     # tcgen05, half-full lanes
    ("gqa_mid", 40, dict(batch=2, ctx_fixed=900, shards=4)),                     # a prefill chunk, two blocks
    ("gqa_tiny", 1, dict(batch=3, ctx_fixed=700, shards=3, kv_dtype="fp8")),
    ("mla_decode", 1, dict(batch=3, ctx_kind="lognormal", median=900, sigma=1.0, ctx_lo=0, ctx_hi=5000, shards=4)),
    ("mla_decode", 3, dict(batch=2, ctx_fixed=1200, shards=3)),
]


@pytest.mark.parametrize("name,q_len,over", CASES)
def test_attention_all_matches_oracle_and_two_calls(name, q_len, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl, q_len=q_len)
    st.append()
    st.partial()
    st.merge()
    torch.cuda.synchronize()
    o2, l2 = st.o.clone(), st.lse.clone()
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    st.attention()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(l2.cpu().numpy()))
    fin = np.isfinite(lse)
    if wl.kind == configs.MLA:
        # the MLA kernel merges the shards inside its online softmax (its own
        # rounding): the two paths agree to the parity bar
        assert_close(o, o2.cpu().numpy(), "one call vs two calls")
        assert_lse_close(lse, l2.cpu().numpy(), "one call vs two calls")
    else:
        # the two paths differ only in the order of the fp32 merge
        assert np.allclose(o, o2.cpu().numpy(), atol=2e-6, rtol=1e-5)
        assert np.allclose(lse[fin], l2.cpu().numpy()[fin], atol=1e-5)
    for b in range(wl.batch):
        ctx_b = int(st.ctx[b])
        starts_b = O.shard_starts([ctx_b], wl.shards)[0]
        if q_len == 1:
            ro, rl, _, _ = oracle_sequence(wl, b, ctx_b + 1, starts_b)
        else:
            ro, rl, _, _ = oracle_mtp_sequence(wl, b, ctx_b, q_len, starts_b)
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")


def test_attention_all_full_size_gqa_mid_sampled():
    wl = configs.get("gqa_mid")
    st = DecodeState(wl)
    st.append()
    st.attention()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    for b in (0, 31):
        ro, rl, _, _ = oracle_sequence(wl, b, int(st.ctx[b]) + 1, O.shard_starts([st.ctx[b]], wl.shards)[0])
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
