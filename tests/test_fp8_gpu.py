"""GQA decode steps over an 8-bit cache (FP8 E4M3 codes with per-tensor
scales) on the GPU against the float64 oracle, which decodes the same codes
exactly: per-shard partials and the merged output; the appended codes land
bit-exactly (values transposed within a block)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, assert_lse_close, oracle_mtp_sequence, oracle_sequence
from sequence_sharded_decode_gb300 import configs, inputs
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

F8 = dict(kv_dtype="fp8")
RAGGED = dict(batch=6, ctx_kind="lognormal", median=300, sigma=1.2, ctx_lo=0, ctx_hi=3000)

CASES = [
    ("gqa_tiny", dict(**F8)),                                            # D=64, 4 shards of 128
    ("gqa_tiny", dict(shards=1, **F8)),
    ("gqa_tiny", dict(shards=3, **RAGGED, **F8)),                        # ragged, contexts down to 0
    ("gqa_tiny", dict(shards=16, **RAGGED, **F8)),                       # many empty shards
    ("gqa_mid", dict(batch=3, ctx_fixed=3000, shards=2, **F8)),          # D=128, g=16
    ("gqa_mid", dict(shards=5, **RAGGED, **F8)),
    ("gqa_mid", dict(batch=2, q_heads=64, kv_heads=2, ctx_fixed=999, shards=3, **F8)),   # two head groups
    ("gqa_mid", dict(batch=2, q_heads=8, kv_heads=8, ctx_fixed=555, shards=4, **F8)),    # g=1
    ("gqa_mid", dict(batch=2, q_heads=12, kv_heads=4, ctx_fixed=700, shards=2, block_size=32, **F8)),
    ("gqa_mid", dict(batch=2, ctx_fixed=1000, shards=3, block_size=48, **F8)),  # block size not a power of two
    ("gqa_tiny", dict(batch=2, ctx_fixed=1500, shards=4, block_size=64, scale=1.0, **F8)),  # peaky softmax
    ("gqa_mid", dict(batch=1, ctx_fixed=0, shards=4, **F8)),             # one token only
    ("gqa_mid", dict(batch=3, ctx_fixed=4000, shards=4, needles=3, **F8)),
    ("gqa_mid", dict(batch=2, ctx_fixed=1200, shards=3, k_scale=0.5, v_scale=2.0, **F8)),   # the scales
    ("gqa_tiny", dict(batch=2, ctx_fixed=900, shards=3, k_scale=0.25, v_scale=0.125, **F8)),
]


def _check(st, wl, q_len=1, seqs=None):
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o = st.o.cpu().numpy()
    lse = st.lse.cpu().numpy()
    parts = st.o_parts.cpu().numpy()
    lses = st.lses.cpu().numpy()
    for b in (range(wl.batch) if seqs is None else seqs):
        ctx_b = int(st.ctx[b])
        starts_b = O.shard_starts([ctx_b], wl.shards)[0]
        if q_len == 1:
            ro, rl, rparts, rlses = oracle_sequence(wl, b, ctx_b + 1, starts_b)
        else:
            ro, rl, rparts, rlses = oracle_mtp_sequence(wl, b, ctx_b, q_len, starts_b)
        assert_close(o[b], ro, f"O[b={b}]")
        assert_lse_close(lse[b], rl, f"LSE[b={b}]")
        for i in range(wl.shards):
            assert_close(parts[i, b], rparts[i], f"O_part[shard={i}, b={b}]")
            assert_lse_close(lses[i, b], rlses[i], f"LSE_part[shard={i}, b={b}]")


@pytest.mark.parametrize("name,over", CASES)
def test_fp8_step_matches_oracle(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl)
    st.step()
    _check(st, wl)


@pytest.mark.parametrize("q_len", [2, 3, 4, 8])
def test_fp8_multi_token_step_matches_oracle(q_len):
    wl = configs.get("gqa_mid").with_(batch=3, ctx_fixed=1700, shards=3, **F8)
    st = DecodeState(wl, q_len=q_len)
    st.step()
    _check(st, wl, q_len)


def test_fp8_codes_land_bit_exactly():
    wl = configs.get("gqa_tiny").with_(batch=2, ctx_fixed=300, shards=3, block_size=32, **F8)
    st = DecodeState(wl, canary=0x55)
    st.append()
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for b in range(wl.batch):
        L = int(st.ctx[b]) + 1
        k = inputs.e4m3_codes(inputs.sequence_kv(wl.seed, inputs.STREAM_K, b, 0, L, wl.kv_heads, wl.dk)).numpy()
        v = inputs.e4m3_codes(inputs.sequence_kv(wl.seed, inputs.STREAM_V, b, 0, L, wl.kv_heads, wl.dv)).numpy()
        for t in list(rng.choice(L, size=12, replace=False)) + [L - 1]:
            i, phys, slot = O.paged_slot(int(t), st.starts_host[b], [tab for _, tab in st.tables_host], b,
                                         wl.block_size)
            kp = st.shards[i].k_pool[phys, :, slot, :].cpu().numpy()
            vp = st.shards[i].v_pool[phys, :, :, slot].cpu().numpy()    # transposed within the block
            assert np.array_equal(kp, k[t]) and np.array_equal(vp, v[t]), (b, t)


def test_fp8_full_size_gqa_mid_sampled():
    wl = configs.get("gqa_mid").with_(**F8)
    st = DecodeState(wl)
    st.step()
    _check(st, wl, seqs=[0, 13, 31])


# The MLA latent cache over 8-bit codes: one row of 576 codes per token; the
# key is k_scale x the decoded row, the value v_scale x its first 512 entries.
MLA_RAGGED = dict(ctx_kind="lognormal", median=900, sigma=1.0, ctx_lo=0, ctx_hi=5000)
MLA_CASES = [
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=300, shards=4, **F8)),
    ("mla_decode", dict(batch=1, ctx_kind="fixed", ctx_fixed=63, shards=1, **F8)),      # exactly one page
    ("mla_decode", dict(batch=1, ctx_kind="fixed", ctx_fixed=0, shards=2, **F8)),       # one token
    ("mla_decode", dict(batch=5, shards=8, **MLA_RAGGED, **F8)),                        # ragged, empty shards
    ("mla_high_concurrency", dict(batch=6, shards=8, **MLA_RAGGED, **F8)),              # fragmented pools
    ("mla_decode", dict(batch=3, ctx_kind="fixed", ctx_fixed=3000, shards=4, needles=3, **F8)),
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=5000, shards=3, scale=1.0, **F8)),  # peaky
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=1200, shards=3, k_scale=0.5, v_scale=2.0, **F8)),
    ("mla_decode", dict(batch=2, ctx_kind="fixed", ctx_fixed=900, shards=2, scale=-0.0417, k_scale=0.25,
                        v_scale=0.125, **F8)),
]


@pytest.mark.parametrize("name,over", MLA_CASES)
def test_fp8_mla_step_matches_oracle(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl)
    st.step()
    _check(st, wl)
    # the fused call on the same state
    st.o.fill_(float("nan"))
    st.attention()
    torch.cuda.synchronize()
    o = st.o.cpu().numpy()
    lse = st.lse.cpu().numpy()
    for b in range(wl.batch):
        ro, rl, _, _ = oracle_sequence(wl, b, int(st.ctx[b]) + 1, O.shard_starts([st.ctx[b]], wl.shards)[0])
        assert_close(o[b], ro, f"fused O[b={b}]")
        assert_lse_close(lse[b], rl, f"fused LSE[b={b}]")


def test_fp8_mla_codes_land_bit_exactly():
    wl = configs.get("mla_decode").with_(batch=2, ctx_kind="fixed", ctx_fixed=300, shards=3, **F8)
    st = DecodeState(wl, canary=0x55)
    st.append()
    torch.cuda.synchronize()
    for b in range(wl.batch):
        L = int(st.ctx[b]) + 1
        lat = inputs.e4m3_codes(inputs.sequence_kv(wl.seed, inputs.STREAM_LATENT, b, 0, L, 1, wl.dk)).numpy()
        for t in (0, 1, L // 2, L - 2, L - 1):
            i, phys, slot = O.paged_slot(int(t), st.starts_host[b], [tab for _, tab in st.tables_host], b,
                                         wl.block_size)
            assert np.array_equal(st.shards[i].k_pool[phys, slot, :].cpu().numpy(), lat[t, 0]), (b, t)


def test_fp8_mla_long_sampled():
    wl = configs.get("mla_long").with_(**F8)
    st = DecodeState(wl)
    st.step()
    _check(st, wl, seqs=[0, 7])
