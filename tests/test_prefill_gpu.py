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
