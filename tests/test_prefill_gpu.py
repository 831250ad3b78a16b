"""Chunked and cached prefill against the sharded cache on the GPU: a chunk
of C new tokens per sequence is appended after the cached context and each
token attends the context and the chunk causally (the multi-token entry
point with q_len = C), against the float64 oracle."""
import pytest

from test_mtp_gpu import _check
from sequence_sharded_decode_gb300 import configs
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

CASES = [
    ("gqa_tiny", 128, dict()),                                                   # 512 cached + a 128-token chunk, 4 shards
    ("gqa_tiny", 200, dict(batch=3, ctx_kind="lognormal", median=300, sigma=1.0, ctx_lo=0, ctx_hi=1500, shards=3)),
    ("gqa_mid", 256, dict(batch=2, ctx_fixed=0, shards=2)),                       # the first chunk of a prompt
    ("gqa_mid", 300, dict(batch=2, ctx_fixed=1700, shards=3)),
    ("gqa_mid", 160, dict(batch=2, ctx_fixed=900, shards=4, kv_dtype="fp8")),
    ("mla_decode", 64, dict(batch=2, ctx_fixed=1000, shards=4)),
]


@pytest.mark.parametrize("name,chunk,over", CASES)
def test_prefill_chunk_matches_oracle(name, chunk, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl, q_len=chunk)
    st.step()
    _check(st, wl, chunk)


# Steps with q_len * g >= 128 query rows per KV head (GQA, head dim 128)
# take the tcgen05 kernel: lanes of 128 rows = 128/g tokens x g heads; the
# token groups of one KV range run on gangs of up to 8 CTAs (2, 3, 4, 6 and 8
# below).
TC_CASES = [
    ("gqa_mid", 8, dict(batch=2, ctx_fixed=700, shards=2)),                             # g=16: 8 tokens per lane
    ("gqa_mid", 20, dict(batch=2, ctx_fixed=1000, shards=3)),                           # a partial last token group
    ("gqa_mid", 64, dict(batch=3, ctx_kind="lognormal", median=600, sigma=1.0, ctx_lo=0, ctx_hi=3000, shards=4)),
    ("gqa_mid", 4, dict(batch=2, q_heads=64, kv_heads=2, ctx_fixed=900, shards=3)),     # g=32: 4 tokens per lane
    ("gqa_mid", 16, dict(batch=2, q_heads=32, kv_heads=4, ctx_fixed=500, shards=2)),    # g=8
    ("gqa_mid", 128, dict(batch=1, q_heads=8, kv_heads=8, ctx_fixed=300, shards=3)),    # g=1: 128 tokens per lane
    ("gqa_mid", 32, dict(batch=2, ctx_fixed=800, shards=2, block_size=32)),
    ("gqa_mid", 32, dict(batch=2, ctx_fixed=800, shards=2, block_size=64)),
    ("gqa_mid", 32, dict(batch=2, ctx_fixed=900, shards=2, block_size=128)),
    ("gqa_mid", 16, dict(batch=2, ctx_fixed=1500, shards=4, needles=3)),
    ("gqa_mid", 24, dict(batch=2, ctx_fixed=1200, shards=3, scale=1.0)),                # peaky softmax
    ("gqa_mid", 40, dict(batch=2, ctx_fixed=0, shards=2)),                              # the first chunk only
    ("gqa_mid", 32, dict(batch=2, ctx_fixed=1000, shards=3, scale=-0.0884)),            # negative scale, two blocks
    ("gqa_mid", 8, dict(batch=2, ctx_fixed=700, shards=2, scale=0.0)),                  # zero scale: prefix means
    ("gqa_mid", 2, dict(batch=2, q_heads=128, kv_heads=2, ctx_fixed=600, shards=2)),    # g=64: 2 tokens per block
    ("gqa_mid", 3, dict(batch=2, q_heads=128, kv_heads=1, ctx_fixed=500, shards=3)),    # g=128: one token per block
    ("gqa_mid", 32, dict(batch=2, ctx_kind="lognormal", median=400, sigma=1.0, ctx_lo=0, ctx_hi=2000,
                         shards=32)),                                                   # the most shards, many empty
    ("gqa_mid", 128, dict(batch=2, ctx_fixed=6000, shards=2)),     # gangs of 8 CTAs; their ranges cut across runs
    ("gqa_mid", 96, dict(batch=3, ctx_kind="lognormal", median=900, sigma=1.0, ctx_lo=0, ctx_hi=4000,
                         shards=3)),                                                    # gangs of 6, ragged
]


@pytest.mark.parametrize("name,chunk,over", TC_CASES)
def test_tc_rows_match_oracle(name, chunk, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl, q_len=chunk)
    st.step()
    _check(st, wl, chunk)
