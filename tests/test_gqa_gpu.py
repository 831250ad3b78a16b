"""GQA decode step on the GPU (append -> partial on every shard -> merge)
against the float64 oracle: per-shard partials and the merged output."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_sequence
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

RAGGED = dict(batch=6, ctx_kind="lognormal", median=300, sigma=1.2, ctx_lo=0, ctx_hi=3000)

CASES = [
    ("gqa_tiny", {}),                                        # the page-shaped tiny case: 4 shards of 128
    ("gqa_tiny", dict(shards=1)),
    ("gqa_tiny", dict(shards=2)),
    ("gqa_tiny", dict(shards=8)),
    ("gqa_tiny", dict(shards=16)),
    ("gqa_tiny", dict(shards=3, **RAGGED)),
    ("gqa_tiny", dict(shards=32, **RAGGED)),                 # many empty shards
    ("gqa_mid", dict(batch=3, ctx_fixed=3000, shards=2)),    # D=128, g=16
    ("gqa_mid", dict(shards=5, **RAGGED)),
    ("gqa_mid", dict(batch=2, q_heads=64, kv_heads=2, ctx_fixed=999, shards=3)),   # g=32: two head groups
    ("gqa_mid", dict(batch=2, q_heads=8, kv_heads=8, ctx_fixed=555, shards=4)),    # g=1 (MHA)
    ("gqa_mid", dict(batch=2, q_heads=12, kv_heads=4, ctx_fixed=700, shards=2, block_size=32)),  # g=3, Bs 32
    ("gqa_tiny", dict(batch=2, ctx_fixed=1500, shards=4, block_size=64, scale=1.0)),  # peaky softmax
    ("gqa_mid", dict(batch=1, ctx_fixed=0, shards=4)),       # one token only
    ("gqa_mid", dict(batch=3, ctx_fixed=4000, shards=4, needles=3)),   # planted q-aligned keys
    ("gqa_mid", dict(batch=2, q_heads=256, kv_heads=2, ctx_fixed=700, shards=3)),  # largest Hq: g=128, 8 head groups
    ("gqa_tiny", dict(batch=2, ctx_fixed=900, shards=3, scale=0.0)),   # uniform weights: O = mean of V
    ("gqa_mid", dict(batch=2, ctx_fixed=800, shards=2, scale=-0.0884)),  # negative scale
]


def _check(st, wl, seqs=None):
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o = st.o.cpu().numpy()
    lse = st.lse.cpu().numpy()
    parts = st.o_parts.cpu().numpy()
    lses = st.lses.cpu().numpy()
    seqs = range(wl.batch) if seqs is None else seqs
    for b in seqs:
        L = int(st.ctx[b]) + 1
        ro, rl, rparts, rlses = oracle_sequence(wl, b, L, O.shard_starts([st.ctx[b]], wl.shards)[0])
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
        for i in range(wl.shards):
            assert_close(parts[i, b], rparts[i], f"O_part[shard={i}, b={b}]")
            assert_lse_close(lses[i, b], rlses[i], f"LSE_part[shard={i}, b={b}]")


@pytest.mark.parametrize("name,over", CASES)
def test_step_matches_oracle(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl)
    st.step()
    _check(st, wl)


def test_shard_count_invariance():
    base = configs.get("gqa_tiny").with_(batch=3, ctx_fixed=2000)
    outs = []
    for n in (1, 2, 4, 8, 16):
        st = DecodeState(base.with_(shards=n))
        st.step()
        torch.cuda.synchronize()
        outs.append(st.o.cpu().numpy())
    for o in outs[1:]:
        assert_close(o, outs[0], "O(N) vs O(1)")


def test_block_table_permutation_is_bitwise_invariant():
    wl = configs.get("gqa_mid").with_(batch=4, ctx_fixed=1000, shards=3)
    a = DecodeState(wl)
    b = DecodeState(wl, table_seed=999)
    assert not all(np.array_equal(x[1], y[1]) for x, y in zip(a.tables_host, b.tables_host))
    a.step()
    b.step()
    torch.cuda.synchronize()
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)
    assert torch.equal(a.o_parts, b.o_parts)


def test_single_shard_entry_point():
    wl = configs.get("gqa_mid").with_(batch=3, ctx_fixed=1800, shards=3)
    st = DecodeState(wl)
    st.append()
    B, N = wl.batch, wl.shards
    starts = st.starts.cpu().numpy()
    for i in range(N):
        rng = np.zeros((B, 2), dtype=np.int32)
        rng[:, 0] = starts[:, i]
        rng[:, 1] = starts[:, i + 1] if i + 1 < N else np.iinfo(np.int32).max
        o = torch.empty((B, wl.q_heads, wl.dv), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, wl.q_heads), dtype=torch.float32, device="cuda")
        ws = torch.empty(dcp.dcp_workspace_size(st.desc, B, 1), dtype=torch.uint8, device="cuda")
        dcp.dcp_decode_partial(st.desc, st.q, st.shards[i], st.seq_lens, torch.from_numpy(rng).cuda(), o, lse, ws,
                               err=st.err)
        torch.cuda.synchronize()
        st.o_parts[i].copy_(o)
        st.lses[i].copy_(lse)
    st.merge()
    _check(st, wl)


def test_full_size_gqa_mid_sampled():
    wl = configs.get("gqa_mid")
    st = DecodeState(wl)
    st.step()
    _check(st, wl, seqs=[0, 13, 31])


def test_device_flags_bad_block_and_table_range():
    wl = configs.get("gqa_tiny")
    st = DecodeState(wl)
    st.shards[1].block_table[0, 2] = -1
    st.step()
    torch.cuda.synchronize()
    assert int(st.err.item()) & dcp.DCP_DEVERR_BLOCK_RANGE
    st.err.zero_()
    st.shards[1].block_table[0, 2] = 0
    st.seq_lens.fill_(100000)  # far past the tables: the last shard's lookups run off its table
    st.partial()
    torch.cuda.synchronize()
    assert int(st.err.item()) & dcp.DCP_DEVERR_TABLE_RANGE


def test_workspace_too_small_is_rejected():
    wl = configs.get("gqa_tiny")
    st = DecodeState(wl)
    small = st.workspace[: st.workspace.numel() - 256]
    with pytest.raises(dcp.DcpError) as e:
        dcp.dcp_decode_partial_all(st.desc, st.q, st.shards, st.seq_lens, st.starts, st.o_parts, st.lses, small)
    assert e.value.status == dcp.DCP_ERR_WORKSPACE
