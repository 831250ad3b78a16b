"""The C-ABI library loads, exports every declared symbol, and its host-only
logic (routing plan, argument validation) matches the oracle -- no GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
from sequence_sharded_decode_gb300 import build, configs, dcp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(dcp.lib_path()):
        build.build()
    return dcp.load()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "dcp.h")).read()
    return sorted(set(re.findall(r"DCP_API\s+[\w\s\*]+?\b(dcp_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert set(declared) == set(dcp.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_version_and_status_strings(lib):
    assert dcp.dcp_version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert dcp.dcp_status_string(code) != "unknown status"
    assert dcp.dcp_status_string(17) == "unknown status"


@pytest.mark.parametrize("name", sorted(configs.PRESETS))
def test_shard_plan_matches_oracle(lib, name):
    wl = configs.get(name)
    ctx = wl.ctx_lens()
    starts, blocks = dcp.dcp_shard_plan(ctx, wl.shards, wl.block_size, 1)
    assert np.array_equal(starts, O.shard_starts(ctx, wl.shards))
    assert np.array_equal(blocks, O.blocks_needed(ctx, wl.shards, wl.block_size, 1))


def test_shard_plan_edge_cases(lib):
    rng = np.random.default_rng(3)
    for _ in range(200):
        B = int(rng.integers(1, 6))
        N = int(rng.integers(1, 33))
        bs = int(rng.choice([1, 3, 16, 64]))
        reserve = int(rng.integers(0, 70))
        ctx = rng.integers(0, 5000, size=B)
        starts, blocks = dcp.dcp_shard_plan(ctx, N, bs, reserve)
        assert np.array_equal(starts, O.shard_starts(ctx, N))
        assert np.array_equal(blocks, O.blocks_needed(ctx, N, bs, reserve))


def test_shard_plan_page_example(lib):
    starts, _ = dcp.dcp_shard_plan([200000], 4, 64, 0)
    assert starts.tolist() == [[0, 50000, 100000, 150000]]


@pytest.mark.parametrize("args", [
    dict(n=0), dict(n=33), dict(bs=0), dict(reserve=-1), dict(ctx=[-1]), dict(ctx=[2**31 - 10], reserve=100),
])
def test_shard_plan_rejects(lib, args):
    with pytest.raises(dcp.DcpError) as e:
        dcp.dcp_shard_plan(args.get("ctx", [10]), args.get("n", 2), args.get("bs", 16), args.get("reserve", 1))
    assert e.value.status == dcp.DCP_ERR_INVALID_ARG


def _desc(**kw):
    base = dict(kind=dcp.DCP_KIND_GQA, num_q_heads=8, num_kv_heads=2, head_dim_k=64, head_dim_v=64,
                block_size=16, scale=0.125)
    base.update(kw)
    return dcp.AttnDesc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(kind=7), dcp.DCP_ERR_INVALID_ARG),
    (dict(num_q_heads=0), dcp.DCP_ERR_SHAPE),
    (dict(num_q_heads=6, num_kv_heads=4), dcp.DCP_ERR_SHAPE),
    (dict(head_dim_k=96, head_dim_v=96), dcp.DCP_ERR_UNSUPPORTED),
    (dict(head_dim_v=128), dcp.DCP_ERR_UNSUPPORTED),
    (dict(block_size=8), dcp.DCP_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), dcp.DCP_ERR_INVALID_ARG),
    (dict(kind=dcp.DCP_KIND_MLA, num_q_heads=128, num_kv_heads=2, head_dim_k=576, head_dim_v=512,
          block_size=64), dcp.DCP_ERR_SHAPE),
    (dict(kind=dcp.DCP_KIND_MLA, num_q_heads=64, num_kv_heads=1, head_dim_k=576, head_dim_v=512,
          block_size=64), dcp.DCP_ERR_UNSUPPORTED),
])
def test_descriptor_validation_before_any_launch(lib, kw, status):
    d = _desc(**kw).c()
    shard = dcp._Shard(16, 16, 1, 16, 1)
    rc = lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(shard), 1, 16, 1, None, 16, 16, 16, 1, None, None)
    assert rc == status
    assert lib.dcp_workspace_size(ctypes.byref(d), 1, 1) == 0


def test_shard_and_pointer_validation(lib):
    d = _desc().c()
    good = dcp._Shard(16, 16, 4, 16, 2)
    # N out of range, NULL pool, zero blocks, misaligned pool, NULL positions
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(good), 0, 16, 1, None, 16, 16, 16, 1, None,
                             None) == dcp.DCP_ERR_INVALID_ARG
    bad = dcp._Shard(None, 16, 4, 16, 2)
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(bad), 1, 16, 1, None, 16, 16, 16, 1, None,
                             None) == dcp.DCP_ERR_INVALID_ARG
    bad = dcp._Shard(16, 16, 0, 16, 2)
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(bad), 1, 16, 1, None, 16, 16, 16, 1, None,
                             None) == dcp.DCP_ERR_SHAPE
    bad = dcp._Shard(18, 16, 4, 16, 2)
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(bad), 1, 16, 1, None, 16, 16, 16, 1, None,
                             None) == dcp.DCP_ERR_INVALID_ARG
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(good), 1, 16, 1, None, None, 16, 16, 1, None,
                             None) == dcp.DCP_ERR_INVALID_ARG
    # seq_ids NULL needs T == B
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(good), 1, 16, 2, None, 16, 16, 16, 3, None,
                             None) == dcp.DCP_ERR_SHAPE
    # T == 0 is a no-op that never launches
    assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(good), 1, 16, 2, 16, 16, 16, 16, 0, None,
                             None) == dcp.DCP_OK
    # GQA needs a V pool; MLA must not have one
    md = _desc(kind=dcp.DCP_KIND_MLA, num_q_heads=128, num_kv_heads=1, head_dim_k=576, head_dim_v=512,
               block_size=64).c()
    assert lib.dcp_kv_append(ctypes.byref(md), ctypes.byref(good), 1, 16, 1, None, 16, 16, None, 1, None,
                             None) == dcp.DCP_ERR_INVALID_ARG


def test_partial_and_merge_validation(lib):
    d = _desc().c()
    good = dcp._Shard(16, 16, 4, 16, 2)
    # NULL outputs / workspace problems are caught on the host
    assert lib.dcp_decode_partial(ctypes.byref(d), 16, ctypes.byref(good), 16, 16, 1, None, 16, 256, 1 << 20,
                                  None, None) == dcp.DCP_ERR_INVALID_ARG
    assert lib.dcp_decode_partial_all(ctypes.byref(d), 16, ctypes.byref(good), 33, 16, 16, 1, 16, 16, 256,
                                      1 << 20, None, None) == dcp.DCP_ERR_INVALID_ARG
    assert lib.dcp_decode_partial(ctypes.byref(d), 16, ctypes.byref(good), 16, 16, 0, 16, 16, None, 0, None,
                                  None) == dcp.DCP_OK
    assert lib.dcp_merge(16, 16, 0, 1, 1, 4, 16, None, None) == dcp.DCP_ERR_INVALID_ARG
    assert lib.dcp_merge(16, 16, 2, 1, 1, 6, 16, None, None) == dcp.DCP_ERR_UNSUPPORTED
    assert lib.dcp_merge(None, 16, 2, 1, 1, 4, 16, None, None) == dcp.DCP_ERR_INVALID_ARG
    assert lib.dcp_merge(16, 16, 2, 0, 1, 4, 16, None, None) == dcp.DCP_OK


def test_multi_token_validation(lib):
    d = _desc().c()
    good = dcp._Shard(16, 16, 4, 16, 2)
    mtp = lib.dcp_decode_partial_all_mtp
    # q_len outside [1, DCP_MAX_QUERY_TOKENS], NULL outputs, N out of range: rejected on the host
    for q_len in (0, -1, dcp.DCP_MAX_QUERY_TOKENS + 1):
        assert mtp(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 2, q_len, 16, 16, 256, 1 << 20, None,
                   None) == dcp.DCP_ERR_INVALID_ARG
    assert mtp(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 2, 4, None, 16, 256, 1 << 20, None,
               None) == dcp.DCP_ERR_INVALID_ARG
    assert mtp(ctypes.byref(d), 16, ctypes.byref(good), 33, 16, 16, 2, 4, 16, 16, 256, 1 << 20, None,
               None) == dcp.DCP_ERR_INVALID_ARG
    # B * q_len must fit the int32 row count
    assert mtp(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 2 ** 30, 4, 16, 16, 256, 1 << 20, None,
               None) == dcp.DCP_ERR_SHAPE
    # no sequences: nothing to do, no launch
    assert mtp(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 0, 4, None, None, None, 0, None,
               None) == dcp.DCP_OK


def test_fp8_cache_validation(lib):
    good = dcp._Shard(16, 16, 4, 16, 2)
    ok = _desc(kv_dtype=dcp.DCP_KV_FP8_E4M3, k_scale=0.5, v_scale=2.0).c()
    assert lib.dcp_kv_append(ctypes.byref(ok), ctypes.byref(good), 1, 16, 2, 16, 16, 16, 16, 0, None,
                             None) == dcp.DCP_OK
    for kw, status in [
        (dict(kv_dtype=2), dcp.DCP_ERR_INVALID_ARG),
        (dict(kv_dtype=dcp.DCP_KV_FP8_E4M3, k_scale=0.0), dcp.DCP_ERR_INVALID_ARG),
        (dict(kv_dtype=dcp.DCP_KV_FP8_E4M3, v_scale=-1.0), dcp.DCP_ERR_INVALID_ARG),
        (dict(kv_dtype=dcp.DCP_KV_FP8_E4M3, k_scale=float("inf")), dcp.DCP_ERR_INVALID_ARG),
        (dict(kv_dtype=dcp.DCP_KV_FP8_E4M3, v_scale=float("nan")), dcp.DCP_ERR_INVALID_ARG),
        (dict(kind=dcp.DCP_KIND_MLA, num_q_heads=128, num_kv_heads=1, head_dim_k=576, head_dim_v=512,
              block_size=64, kv_dtype=dcp.DCP_KV_FP8_E4M3, k_scale=0.0), dcp.DCP_ERR_INVALID_ARG),
    ]:
        d = _desc(**kw).c()
        assert lib.dcp_kv_append(ctypes.byref(d), ctypes.byref(good), 1, 16, 1, None, 16, 16, 16, 1, None,
                                 None) == status, kw
        assert lib.dcp_workspace_size(ctypes.byref(d), 1, 1) == 0
    # the MLA latent cache takes 8-bit codes too (one row per token, no value pool)
    mla = _desc(kind=dcp.DCP_KIND_MLA, num_q_heads=128, num_kv_heads=1, head_dim_k=576, head_dim_v=512,
                block_size=64, kv_dtype=dcp.DCP_KV_FP8_E4M3, k_scale=0.5, v_scale=2.0).c()
    mla_shard = dcp._Shard(16, None, 4, 16, 2)
    assert lib.dcp_kv_append(ctypes.byref(mla), ctypes.byref(mla_shard), 1, 16, 2, 16, 16, 16, None, 0, None,
                             None) == dcp.DCP_OK


def test_attention_all_validation(lib):
    d = _desc().c()
    good = dcp._Shard(16, 16, 4, 16, 2)
    f = lib.dcp_attention_all
    # NULL merged output, q_len out of range, N out of range: rejected on the host
    assert f(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 2, 1, 16, 16, None, None, 256, 1 << 20, None,
             None) == dcp.DCP_ERR_INVALID_ARG
    assert f(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 2, 0, 16, 16, 16, None, 256, 1 << 20, None,
             None) == dcp.DCP_ERR_INVALID_ARG
    assert f(ctypes.byref(d), 16, ctypes.byref(good), 33, 16, 16, 2, 1, 16, 16, 16, None, 256, 1 << 20, None,
             None) == dcp.DCP_ERR_INVALID_ARG
    # misaligned merged output
    assert f(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 2, 1, 16, 16, 18, None, 256, 1 << 20, None,
             None) == dcp.DCP_ERR_INVALID_ARG
    # no sequences: nothing to do
    assert f(ctypes.byref(d), 16, ctypes.byref(good), 1, 16, 16, 0, 1, None, None, None, None, None, 0, None,
             None) == dcp.DCP_OK
