"""MLA-absorbed decode step on the GPU (append -> tcgen05 partial on every
shard -> merge) against the float64 oracle: per-shard partials and the
merged output, at small sizes in full and at the workload sizes on sampled
sequences."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_sequence
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

RAGGED = dict(ctx_kind="lognormal", median=900, sigma=1.0, ctx_lo=1, ctx_hi=6000)

CASES = [
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=300, shards=4)),
    ("mla_decode", dict(batch=1, ctx_kind="fixed", ctx_fixed=63, shards=1)),      # exactly one tile
    ("mla_decode", dict(batch=1, ctx_kind="fixed", ctx_fixed=0, shards=2)),       # one token
    ("mla_decode", dict(batch=5, shards=8, **RAGGED)),                            # ragged, partial tiles
    ("mla_decode", dict(batch=3, shards=16, **RAGGED)),
    ("mla_decode", dict(batch=3, shards=32, ctx_kind="fixed", ctx_fixed=700)),    # many short/empty shards
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=5000, shards=3, scale=1.0)),  # peaky: lazy rescale
    ("mla_high_concurrency", dict(batch=6, shards=8, **RAGGED)),                  # fragmented pools
    ("mla_decode", dict(batch=3, ctx_kind="fixed", ctx_fixed=3000, shards=4, needles=3)),  # planted keys
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=900, shards=3, scale=0.0)),   # uniform weights
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=900, shards=2, scale=-0.0417)),  # negative scale
]


def _check(st, wl, seqs=None, parts=True):
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o = st.o.cpu().numpy()
    lse = st.lse.cpu().numpy()
    op = st.o_parts.cpu().numpy()
    lp = st.lses.cpu().numpy()
    seqs = range(wl.batch) if seqs is None else seqs
    for b in seqs:
        L = int(st.ctx[b]) + 1
        ro, rl, rparts, rlses = oracle_sequence(wl, b, L, O.shard_starts([st.ctx[b]], wl.shards)[0])
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
        if parts:
            for i in range(wl.shards):
                assert_close(op[i, b], rparts[i], f"O_part[shard={i}, b={b}]")
                assert_lse_close(lp[i, b], rlses[i], f"LSE_part[shard={i}, b={b}]")


@pytest.mark.parametrize("name,over", CASES)
def test_step_matches_oracle(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl)
    st.step()
    _check(st, wl)


def test_shard_count_invariance():
    base = configs.get("mla_decode").with_(batch=2, ctx_kind="fixed", ctx_fixed=3000)
    outs = []
    for n in (1, 2, 5, 8, 16):
        st = DecodeState(base.with_(shards=n))
        st.step()
        torch.cuda.synchronize()
        outs.append(st.o.cpu().numpy())
    for o in outs[1:]:
        assert_close(o, outs[0], "O(N) vs O(1)")


def test_block_table_permutation_is_bitwise_invariant():
    wl = configs.get("mla_high_concurrency").with_(batch=3, shards=4, **RAGGED)
    a = DecodeState(wl)
    b = DecodeState(wl, table_seed=4242)
    a.step()
    b.step()
    torch.cuda.synchronize()
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)


def test_device_flag_bad_block():
    wl = configs.get("mla_decode").with_(batch=2, ctx_kind="fixed", ctx_fixed=500, shards=2)
    st = DecodeState(wl)
    st.shards[0].block_table[1, 1] = st.shards[0].k_pool.shape[0] + 5
    st.step()
    torch.cuda.synchronize()
    assert int(st.err.item()) & dcp.DCP_DEVERR_BLOCK_RANGE
    assert np.isfinite(st.o.cpu().numpy()).all()


def _check_fused(st, wl, seqs):
    """The path bench.py times (append, then dcp_attention_all: partial
    attention and the one-pass merge in one call) on the same state: the
    merged output of the sampled sequences against the oracle. The append
    already ran, so only the fused call runs here."""
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    st.attention()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o = st.o.cpu().numpy()
    lse = st.lse.cpu().numpy()
    for b in seqs:
        L = int(st.ctx[b]) + 1
        ro, rl, _, _ = oracle_sequence(wl, b, L, O.shard_starts([st.ctx[b]], wl.shards)[0])
        assert_close(o[b], ro, f"fused O[b={b}]")
        assert_lse_close(lse[b], rl, f"fused LSE[b={b}]")


@pytest.mark.parametrize("shards", [8, 16])
def test_mla_long_sampled(shards):
    """Full-size long-context workload (8 x 200,001 tokens): the two-call path
    per shard and merged, then the fused call bench.py times."""
    wl = configs.get("mla_long").with_(shards=shards)
    st = DecodeState(wl)
    st.step()
    _check(st, wl, seqs=[0, 7])
    _check_fused(st, wl, seqs=[0, 3, 7])


def test_mla_decode_full_size_sampled():
    wl = configs.get("mla_decode")
    st = DecodeState(wl)
    st.step()
    ctx = wl.ctx_lens()
    seqs = [int(np.argmin(ctx)), int(np.argmax(ctx)), 17]
    _check(st, wl, seqs=seqs)
    _check_fused(st, wl, seqs=seqs)


def test_mla_high_concurrency_full_size_sampled():
    """The 512-sequence workload with fragmented pools, at full size: the
    shortest and the longest sequence and one in between, every shard, on the
    two-call path and on the fused call bench.py times (append +
    dcp_attention_all)."""
    wl = configs.get("mla_high_concurrency")
    st = DecodeState(wl)
    st.step()
    ctx = wl.ctx_lens()
    seqs = [int(np.argmin(ctx)), int(np.argmax(ctx)), 255]
    _check(st, wl, seqs=seqs)
    _check_fused(st, wl, seqs=seqs)
