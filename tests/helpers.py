"""Shared test helpers: oracle inputs regenerated on the CPU, and the tolerance.

The oracle side regenerates the logical (unsharded) K/V of a sequence on
the CPU from the same seeded generator the GPU path used to fill its pools,
widens the bf16 bits to float64 exactly, and calls the oracle. Nothing here
reads a value produced by the CUDA path.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from sequence_sharded_decode_gb300 import configs, inputs

# Parity bar for bf16 KV with fp32 accumulation: elementwise max-abs 2e-3, and
# max-rel 1e-2 where |ref| >= 0.2 (where the two bounds meet); LSE within 1e-3.
ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 0.2
LSE_ATOL = 1e-3


def f64(x: torch.Tensor) -> np.ndarray:
    return O.bf16_bits_to_f64(inputs.bf16_bits(x))


def oracle_query(wl: configs.Workload, b: int) -> np.ndarray:
    stream = inputs.STREAM_Q_MLA if wl.kind == configs.MLA else inputs.STREAM_Q
    return f64(inputs.query(wl.seed, [b], wl.q_heads, wl.dk, "cpu", stream=stream))[0]


def oracle_kv(wl: configs.Workload, b: int, L: int):
    """Logical K [L, Hkv, Dk] and V [L, Hkv, Dv] (float64) of sequence b,
    with the workload's planted needles (if any) applied on the CPU."""
    plan = wl.needle_plan()
    plan_b = {b: plan[b]} if b in plan else {}
    pos = np.arange(L)
    bids = np.full(L, b)
    if wl.kind == configs.MLA:
        lat = inputs.sequence_kv(wl.seed, inputs.STREAM_LATENT, b, 0, L, 1, wl.dk)
        if plan_b:
            q = inputs.query(wl.seed, np.arange(b + 1), wl.q_heads, wl.dk, stream=inputs.STREAM_Q_MLA)
            lat = inputs.plant_needles(lat.view(L, wl.dk), bids, pos, q, plan_b, wl.q_heads).view(L, 1, wl.dk)
        if wl.kv_dtype == "fp8":  # one row of codes: key = k_scale * decode, value = v_scale * decode[:dv]
            codes = inputs.e4m3_codes(lat).numpy()
            return O.fp8_kv(codes, codes[:, :, :wl.dv], wl.k_scale, wl.v_scale)
        lat = f64(lat)
        return lat, lat[:, :, :wl.dv]
    k = inputs.sequence_kv(wl.seed, inputs.STREAM_K, b, 0, L, wl.kv_heads, wl.dk)
    if plan_b:
        q = inputs.query(wl.seed, np.arange(b + 1), wl.q_heads, wl.dk)
        k = inputs.plant_needles(k, bids, pos, q, plan_b, wl.q_heads)
    v = inputs.sequence_kv(wl.seed, inputs.STREAM_V, b, 0, L, wl.kv_heads, wl.dv)
    if wl.kv_dtype == "fp8":  # the cache holds the E4M3 codes of the same draws
        return O.fp8_kv(inputs.e4m3_codes(k).numpy(), inputs.e4m3_codes(v).numpy(), wl.k_scale, wl.v_scale)
    return f64(k), f64(v)


def oracle_sequence(wl: configs.Workload, b: int, L: int, starts_b):
    """(O, LSE, O_parts, LSE_parts) from the oracle for sequence b attending L tokens."""
    q = oracle_query(wl, b)
    K, V = oracle_kv(wl, b, L)
    return O.sharded_attention(q, K, V, wl.scale, starts_b, L)


def oracle_mtp_sequence(wl: configs.Workload, b: int, ctx_b: int, q_len: int, starts_b):
    """(O [q_len, Hq, Dv], LSE, O_parts [N, q_len, ...], LSE_parts) from the
    oracle for sequence b with q_len new tokens after ctx_b context tokens."""
    stream = inputs.STREAM_Q_MLA if wl.kind == configs.MLA else inputs.STREAM_Q
    q = f64(inputs.query_tokens(wl.seed, [b], q_len, wl.q_heads, wl.dk, "cpu", stream=stream))[0]
    L = int(ctx_b) + q_len
    K, V = oracle_kv(wl, b, L)
    return O.sharded_mtp_attention(q, K, V, wl.scale, starts_b, L)


def assert_close(got, ref, what: str, atol: float = ATOL, rtol: float = RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got - ref)
    i = int(np.argmax(d))
    assert d.max() <= atol, f"{what}: max-abs {d.max():.3e} at {np.unravel_index(i, d.shape)} (bound {atol})"
    big = np.abs(ref) >= REL_FLOOR
    if big.any():
        rel = (d[big] / np.abs(ref[big])).max()
        assert rel <= rtol, f"{what}: max-rel {rel:.3e} (bound {rtol})"


def assert_lse_close(got, ref, what: str, atol: float = LSE_ATOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    inf_r = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_r), f"{what}: -inf pattern differs"
    if (~inf_r).any():
        d = np.abs(got[~inf_r] - ref[~inf_r]).max()
        assert d <= atol, f"{what}: LSE max-abs {d:.3e} (bound {atol})"


def oracle_routing(wl: configs.Workload, reserve: int = 1):
    """Oracle shard starts and blocks needed for a workload's context lengths."""
    ctx = wl.ctx_lens()
    return O.shard_starts(ctx, wl.shards), O.blocks_needed(ctx, wl.shards, wl.block_size, reserve)
