"""Multi-token decode steps on the GPU (q_len new tokens per sequence, each
query causal at its own position) against the float64 oracle: per-shard
partials and the merged output, for GQA and MLA."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_mtp_sequence
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

RAGGED = dict(batch=5, ctx_kind="lognormal", median=300, sigma=1.2, ctx_lo=0, ctx_hi=3000)
RAGGED_MLA = dict(batch=4, ctx_kind="lognormal", median=900, sigma=1.0, ctx_lo=0, ctx_hi=5000)

CASES = [
    ("gqa_tiny", 2, {}),
    ("gqa_tiny", 4, dict(shards=3, **RAGGED)),                 # contexts down to 0
    ("gqa_tiny", 8, dict(batch=2, ctx_fixed=20, shards=16)),   # causal limits cut through tiny shards
    ("gqa_tiny", 64, dict(batch=2, ctx_fixed=100, shards=4)),  # the largest q_len
    ("gqa_mid", 8, dict(batch=3, ctx_fixed=3000, shards=2)),
    ("gqa_mid", 3, dict(batch=2, q_heads=64, kv_heads=2, ctx_fixed=999, shards=3)),  # two head groups
    ("gqa_mid", 2, dict(shards=5, **RAGGED)),
    ("gqa_mid", 4, dict(batch=2, ctx_fixed=2000, shards=4, needles=3)),
    ("mla_decode", 2, dict(shards=4, **RAGGED_MLA)),
    ("mla_decode", 4, dict(batch=2, ctx_fixed=3000, shards=8)),
    ("mla_decode", 3, dict(batch=2, ctx_fixed=2500, shards=3, needles=3)),
    ("mla_decode", 5, dict(batch=2, ctx_fixed=0, shards=3)),   # only the new tokens
]


def _check(st, wl, q_len, seqs=None):
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o = st.o.cpu().numpy()
    lse = st.lse.cpu().numpy()
    parts = st.o_parts.cpu().numpy()
    lses = st.lses.cpu().numpy()
    for b in (range(wl.batch) if seqs is None else seqs):
        ctx_b = int(st.ctx[b])
        starts_b = O.shard_starts([ctx_b], wl.shards)[0]
        ro, rl, rparts, rlses = oracle_mtp_sequence(wl, b, ctx_b, q_len, starts_b)
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
        for i in range(wl.shards):
            assert_close(parts[i, b], rparts[i], f"O_part[shard={i}, b={b}]")
            assert_lse_close(lses[i, b], rlses[i], f"LSE_part[shard={i}, b={b}]")


@pytest.mark.parametrize("name,q_len,over", CASES)
def test_multi_token_step_matches_oracle(name, q_len, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl, q_len=q_len)
    st.step()
    _check(st, wl, q_len)


@pytest.mark.parametrize("name", ["gqa_mid", "mla_decode"])
def test_one_query_token_is_the_decode_call(name):
    wl = configs.get(name).with_(batch=3, ctx_fixed=1500, shards=3)
    st = DecodeState(wl)
    st.step()
    o_parts = torch.empty_like(st.o_parts).unsqueeze(2)
    lses = torch.empty_like(st.lses).unsqueeze(2)
    dcp.dcp_decode_partial_all_mtp(st.desc, st.q.unsqueeze(1), st.shards, st.seq_lens, st.starts, o_parts, lses,
                                   st.workspace, err=st.err)
    torch.cuda.synchronize()
    assert torch.equal(o_parts[:, :, 0], st.o_parts) and torch.equal(lses[:, :, 0], st.lses)


def test_full_size_gqa_mid_sampled():
    wl = configs.get("gqa_mid")
    st = DecodeState(wl, q_len=4)
    st.step()
    _check(st, wl, 4, seqs=[0, 31])
