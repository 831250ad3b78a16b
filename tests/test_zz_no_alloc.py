"""dcp_decode_partial_all_noalloc: the partial-attention entry point for
callers that cannot allocate device memory where they call it (a plugin in a
serving engine whose allocator owns all device memory and gives extensions no
scratch, or a decode loop that must not call cudaMalloc because it can
synchronise the device). It runs on the library's fixed device scratch array
instead of a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test. It must pass alone in a
fresh process (where its first call also does the one-time scratch lookup)
and after the other tests.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close, assert_lse_close
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [
    ("gqa_tiny", {}),
    ("gqa_mid", dict(batch=4, ctx_kind="lognormal", median=3000, sigma=1.0, ctx_lo=0, ctx_hi=20000, shards=3)),
    # 64 query heads on one KV head: the tcgen05 many-row GQA kernel
    ("gqa_mid", dict(batch=3, q_heads=64, kv_heads=1, ctx_kind="lognormal", median=2000, sigma=1.0, ctx_lo=0,
                     ctx_hi=9000, shards=4)),
    # the MLA pair kernel, with ranges split across CTAs (workspace rows used)
    ("mla_decode", dict(batch=3, ctx_kind="lognormal", median=20000, sigma=1.0, ctx_lo=0, ctx_hi=60000, shards=8)),
])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl)
    st.append()
    st.partial()  # the existing entry point, with a caller-allocated workspace
    torch.cuda.synchronize()
    ref_o = st.o_parts.cpu().numpy()
    ref_l = st.lses.cpu().numpy()
    for call in range(2):
        o = torch.full_like(st.o_parts, float("nan"))
        lse = torch.full_like(st.lses, float("nan"))
        dcp.dcp_decode_partial_all_noalloc(st.desc, st.q, st.shards, st.seq_lens, st.starts, o, lse, err=st.err)
        torch.cuda.synchronize()
        assert int(st.err.item()) == 0
        assert_close(o.cpu().numpy(), ref_o, f"no-alloc O_parts, call {call}")
        assert_lse_close(lse.cpu().numpy(), ref_l, f"no-alloc LSE, call {call}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 4096 sequences x 32 shards x 16 KV heads = 2M lanes: the work list alone
    # needs more than the fixed scratch, so the call must return
    # DCP_ERR_SCRATCH_LIMIT on the host before any launch.
    B, N, hkv = 4096, 32, 16
    desc = dcp.AttnDesc(dcp.DCP_KIND_GQA, 16 * hkv, hkv, 128, 128, 16, 0.088)
    assert dcp.dcp_workspace_size(desc, B, N) > dcp.DCP_NOALLOC_SCRATCH_BYTES
    dev = "cuda"
    pool = torch.zeros((1, hkv, 16, 128), dtype=torch.bfloat16, device=dev)
    table = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    shards = [dcp.Shard(pool, pool, table) for _ in range(N)]
    q = torch.zeros((B, 16 * hkv, 128), dtype=torch.bfloat16, device=dev)
    seq_lens = torch.ones(B, dtype=torch.int32, device=dev)
    starts = torch.zeros((B, N), dtype=torch.int32, device=dev)
    o = torch.zeros((1, 1, 1, 128), dtype=torch.float32, device=dev)
    lse = torch.zeros((1, 1, 1), dtype=torch.float32, device=dev)
    with pytest.raises(dcp.DcpError) as e:
        dcp.dcp_decode_partial_all_noalloc(desc, q, shards, seq_lens, starts, o, lse)
    assert e.value.status == dcp.DCP_ERR_SCRATCH_LIMIT
    assert np.all(o.cpu().numpy() == 0)
