"""Seeded random MLA steps on the GPU against the float64 oracle: shard
counts from 1 to 16, context lengths on and around the 64-token page and the
32-token half page each CTA of the pair scores (1, 63, 64, 65, 127, 128, ...)
and ragged mixes, one to three query tokens, through both call paths
(dcp_attention_all, which merges inside the attention kernel, and
partial + dcp_merge). The cases are drawn once from a fixed seed, so a
failure names a reproducible shape."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_mtp_sequence, oracle_sequence
from sequence_sharded_decode_gb300 import configs
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu


def _cases(n=14, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        shards = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        q_len = int(rng.choice([1, 1, 1, 2, 3]))
        one_call = bool(i % 2 == 0)
        if rng.random() < 0.5:
            ctx = int(rng.choice([0, 31, 32, 62, 63, 64, 126, 127, 191, 1000 + int(rng.integers(0, 3000))]))
            over = dict(batch=int(rng.integers(1, 5)), ctx_kind="fixed", ctx_fixed=ctx, shards=shards)
        else:
            over = dict(batch=int(rng.integers(2, 10)), ctx_kind="lognormal", median=int(rng.integers(40, 2500)),
                        sigma=float(rng.uniform(0.5, 1.5)), ctx_lo=int(rng.integers(0, 2)), ctx_hi=6000,
                        shards=shards)
        out.append((over, q_len, one_call))
    return out


@pytest.mark.parametrize("over,q_len,one_call", _cases())
def test_random_step_matches_oracle(over, q_len, one_call):
    wl = configs.get("mla_decode").with_(**over)
    st = DecodeState(wl, q_len=q_len)
    st.append()
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    if one_call:
        st.attention()
    else:
        st.partial()
        st.merge()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    for b in range(wl.batch):
        ctx_b = int(st.ctx[b])
        starts_b = O.shard_starts([ctx_b], wl.shards)[0]
        if q_len == 1:
            ro, rl, _, _ = oracle_sequence(wl, b, ctx_b + 1, starts_b)
        else:
            ro, rl, _, _ = oracle_mtp_sequence(wl, b, ctx_b, q_len, starts_b)
        assert_close(o[b], ro, f"O[b={b}] ({over}, q_len {q_len}, one call {one_call})")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
