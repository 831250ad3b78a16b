"""The one-call MLA path (dcp_attention_all): the attention kernel merges the
shards itself. A CTA pair carries one online softmax through the consecutive
shards of a query row group; row groups cut by a CTA-run boundary leave
pieces in the workspace, which the CTA completing the group merges (up to
four pieces) or a short finishing kernel merges (more pieces; it also writes
the groups without tokens). Checked against the float64 oracle on shapes
that produce every kind of row group: one piece (many short sequences), two
to four pieces, many pieces (long sequences over few CTA runs), empty shards,
empty row groups, multi-token steps, the 8-bit cache."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_mtp_sequence, oracle_sequence
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

RAGGED = dict(ctx_kind="lognormal", median=900, sigma=1.0, ctx_lo=1, ctx_hi=6000)

CASES = [
    ("mla_decode", 1, dict(batch=2, ctx_kind="fixed", ctx_fixed=300, shards=4)),
    ("mla_decode", 1, dict(batch=1, ctx_kind="fixed", ctx_fixed=0, shards=2)),        # one token
    ("mla_decode", 1, dict(batch=2, ctx_kind="fixed", ctx_fixed=63, shards=1)),       # one shard, one tile
    ("mla_decode", 1, dict(batch=3, ctx_kind="fixed", ctx_fixed=9000, shards=1)),     # one shard over several runs
    ("mla_decode", 1, dict(batch=5, shards=8, **RAGGED)),                             # ragged, partial tiles
    ("mla_decode", 1, dict(batch=3, shards=32, ctx_kind="fixed", ctx_fixed=700)),     # many empty shards
    ("mla_decode", 1, dict(batch=300, shards=2, ctx_kind="lognormal", median=90, sigma=0.8,
                           ctx_lo=1, ctx_hi=400)),                                    # most groups in one run
    ("mla_decode", 1, dict(batch=2, ctx_kind="fixed", ctx_fixed=40000, shards=8)),    # ~40 pieces a group
    ("mla_decode", 1, dict(batch=25, ctx_kind="fixed", ctx_fixed=2000, shards=4)),    # 3-4 pieces: in the kernel
    ("mla_decode", 1, dict(batch=40, ctx_kind="fixed", ctx_fixed=2000, shards=4)),    # 2-3 pieces
    ("mla_decode", 1, dict(batch=2, ctx_kind="fixed", ctx_fixed=5000, shards=3, scale=1.0)),  # peaky
    ("mla_decode", 1, dict(batch=3, ctx_kind="fixed", ctx_fixed=3000, shards=4, needles=3)),  # planted keys
    ("mla_decode", 1, dict(batch=2, ctx_kind="fixed", ctx_fixed=900, shards=2, scale=-0.0417)),  # negative scale
    ("mla_high_concurrency", 1, dict(batch=6, shards=8, **RAGGED)),                   # fragmented pools
    ("mla_decode", 3, dict(batch=2, ctx_fixed=1200, shards=3)),                       # three query tokens
    ("mla_decode", 2, dict(batch=40, shards=4, ctx_kind="lognormal", median=200, sigma=1.0,
                           ctx_lo=0, ctx_hi=2000)),
    ("mla_decode", 1, dict(batch=3, shards=4, kv_dtype="fp8", k_scale=0.5, v_scale=2.0, **RAGGED)),
]


def _oracle(st, wl, b):
    starts_b = O.shard_starts([st.ctx[b]], wl.shards)[0]
    if st.q_len == 1:
        ro, rl, _, _ = oracle_sequence(wl, b, int(st.ctx[b]) + 1, starts_b)
    else:
        ro, rl, _, _ = oracle_mtp_sequence(wl, b, int(st.ctx[b]), st.q_len, starts_b)
    return ro, rl


@pytest.mark.parametrize("name,q_len,over", CASES)
def test_one_call_matches_oracle(name, q_len, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl, q_len=q_len)
    st.append()
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    st.attention()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    seqs = range(wl.batch) if wl.batch <= 40 else sorted({0, 1, 7, 99, 150, 222, wl.batch - 1})
    for b in seqs:
        ro, rl = _oracle(st, wl, b)
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
    # the two-call path on the same state: both are the oracle's result within
    # the parity bar (they round differently: here the shards meet inside the
    # online softmax, there through the fp32 LSE merge)
    o1 = o.copy()
    st.partial()
    st.merge()
    torch.cuda.synchronize()
    assert_close(o1, st.o.cpu().numpy(), "one call vs two calls")


def test_groups_without_tokens_are_zero():
    """A row group with no token in any shard (length 0: nothing appended)
    gets o = 0 and LSE = -inf; the others are unaffected."""
    wl = configs.get("mla_decode").with_(batch=4, ctx_kind="fixed", ctx_fixed=700, shards=4)
    st = DecodeState(wl)
    st.append()
    lens = st.seq_lens.clone()
    lens[1] = 0
    lens[3] = 0
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    dcp.dcp_attention_all(st.desc, st.q, st.shards, lens, st.starts, st.o_parts, st.lses, st.o, st.lse,
                          st.workspace, err=st.err)
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    for b in (1, 3):
        assert (o[b] == 0).all() and np.isneginf(lse[b]).all()
    for b in (0, 2):
        ro, rl = _oracle(st, wl, b)
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")


def test_one_call_without_lse_out():
    wl = configs.get("mla_decode").with_(batch=3, shards=4, **RAGGED)
    st = DecodeState(wl)
    st.append()
    st.o.fill_(float("nan"))
    dcp.dcp_attention_all(st.desc, st.q, st.shards, st.seq_lens, st.starts, st.o_parts, st.lses, st.o, None,
                          st.workspace, err=st.err)
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o = st.o.cpu().numpy()
    for b in range(wl.batch):
        assert_close(o[b], _oracle(st, wl, b)[0], f"O[b={b}]")


def test_one_call_block_table_permutation_is_bitwise_invariant():
    wl = configs.get("mla_high_concurrency").with_(batch=5, shards=4, **RAGGED)
    a = DecodeState(wl)
    b = DecodeState(wl, table_seed=4242)
    a.append()
    b.append()
    a.attention()
    b.attention()
    torch.cuda.synchronize()
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)


def test_one_call_repeats_bitwise():
    """The piece counters are reset by every call's plan: calling twice on
    the same state gives the same bits."""
    wl = configs.get("mla_decode").with_(batch=3, ctx_kind="fixed", ctx_fixed=20000, shards=8)
    st = DecodeState(wl)
    st.append()
    st.attention()
    torch.cuda.synchronize()
    o1, l1 = st.o.clone(), st.lse.clone()
    st.o.fill_(float("nan"))
    st.attention()
    torch.cuda.synchronize()
    assert torch.equal(st.o, o1) and torch.equal(st.lse, l1)


def test_one_call_flags_bad_block():
    wl = configs.get("mla_decode").with_(batch=2, ctx_kind="fixed", ctx_fixed=500, shards=2)
    st = DecodeState(wl)
    st.append()
    st.shards[0].block_table[1, 1] = st.shards[0].k_pool.shape[0] + 5
    st.attention()
    torch.cuda.synchronize()
    assert int(st.err.item()) & dcp.DCP_DEVERR_BLOCK_RANGE
    assert np.isfinite(st.o.cpu().numpy()).all()
