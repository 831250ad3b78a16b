"""Pins for the oracle's multi-token decode queries (CPU only).

A step that verifies q_len new tokens: query token i sits at position
seq_len - q_len + i and attends every token at or before it. The oracle's
functions are checked against torch's scaled-dot-product attention with an
explicit boolean mask and scipy's logsumexp (an independent route through a
full masked score matrix), closed forms, the causal invariant, and the
exactness of the sharded merge.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle as O

RNG = np.random.default_rng(4321)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _masked_route(q, K, V, scale, seq_len):
    """Every query against the whole sequence with a causal boolean mask."""
    ql, hq, dk = q.shape
    L, hkv, _ = K.shape
    g = hq // hkv
    pos = np.arange(seq_len - ql, seq_len)                      # query positions
    allowed = np.arange(L)[None, :] <= pos[:, None]             # [q_len, L]
    Kt = torch.from_numpy(np.repeat(K, g, axis=1)).permute(1, 0, 2)[None]   # [1, Hq, L, Dk]
    Vt = torch.from_numpy(np.repeat(V, g, axis=1)).permute(1, 0, 2)[None]
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]  # [1, Hq, q_len, Dk]
    mask = torch.from_numpy(allowed)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask, scale=scale)
    o = o[0].permute(1, 0, 2).numpy()                           # [q_len, Hq, Dv]
    lse = np.empty((ql, hq))
    for i in range(ql):
        for h in range(hq):
            s = scale * (K[:, h // g, :] @ q[i, h])
            lse[i, h] = logsumexp(np.where(allowed[i], s, -np.inf))
    return o, lse


@pytest.mark.parametrize("L,ql,hq,hkv,d", [(40, 4, 8, 2, 16), (300, 8, 16, 16, 32), (129, 2, 4, 1, 64),
                                           (200, 150, 4, 2, 16), (96, 96, 4, 1, 8)])  # prefill chunks
def test_matches_masked_sdpa(L, ql, hq, hkv, d):
    q, K, V = _rand(ql, hq, d), _rand(L, hkv, d), _rand(L, hkv, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = O.mtp_attention(q, K, V, scale, L)
    ro, rl = _masked_route(q, K, V, scale, L)
    assert np.max(np.abs(o - ro)) < 1e-12
    assert np.max(np.abs(lse - rl)) < 1e-11


def test_one_query_is_plain_decode():
    q, K, V = _rand(1, 8, 16), _rand(50, 2, 16), _rand(50, 2, 16)
    o, lse = O.mtp_attention(q, K, V, 0.25, 50)
    ro, rl = O.attention(q[0], K, V, 0.25)
    assert np.array_equal(o[0], ro) and np.array_equal(lse[0], rl)
    starts = O.shard_starts([49], 3)[0]
    so, sl, _, _ = O.sharded_mtp_attention(q, K, V, 0.25, starts, 50)
    ro2, rl2, _, _ = O.sharded_attention(q[0], K, V, 0.25, starts, 50)
    assert np.array_equal(so[0], ro2) and np.array_equal(sl[0], rl2)


def test_later_tokens_do_not_leak_backwards():
    L, ql = 30, 5
    q, K, V = _rand(ql, 4, 8), _rand(L, 1, 8), _rand(L, 1, 8)
    o, lse = O.mtp_attention(q, K, V, 0.3, L)
    K2, V2 = K.copy(), V.copy()
    K2[L - 1] += 5.0
    V2[L - 1] -= 3.0          # only the last query sees position L-1
    o2, lse2 = O.mtp_attention(q, K2, V2, 0.3, L)
    assert np.array_equal(o[:-1], o2[:-1]) and np.array_equal(lse[:-1], lse2[:-1])
    assert np.max(np.abs(o[-1] - o2[-1])) > 1e-3
    K3 = K.copy()
    K3[L - ql] += 5.0          # the first query's own position: every query sees it
    o3, _ = O.mtp_attention(q, K3, V, 0.3, L)
    assert all(np.max(np.abs(o[i] - o3[i])) > 1e-6 for i in range(ql))


def test_equal_keys_give_prefix_means():
    L, ql = 20, 4
    K = np.ones((L, 1, 6))
    V = _rand(L, 1, 3)
    q = _rand(ql, 2, 6)
    o, lse = O.mtp_attention(q, K, V, 0.5, L)
    for i in range(ql):
        n = L - ql + i + 1
        assert np.allclose(o[i], V[:n, 0].mean(axis=0)[None], atol=1e-13)
        assert np.allclose(lse[i], 0.5 * q[i].sum(axis=1) + math.log(n), atol=1e-12)


@pytest.mark.parametrize("L,N,ql", [(100, 4, 3), (17, 8, 8), (5, 16, 4), (64, 2, 1)])
def test_sharded_merge_is_exact(L, N, ql):
    q, K, V = _rand(ql, 4, 8), _rand(L, 2, 8), _rand(L, 2, 8)
    starts = O.shard_starts([L - ql], N)[0]
    so, sl, parts, plses = O.sharded_mtp_attention(q, K, V, 0.4, starts, L)
    o, lse = O.mtp_attention(q, K, V, 0.4, L)
    assert parts.shape == (N, ql, 4, 8) and plses.shape == (N, ql, 4)
    assert np.max(np.abs(so - o)) < 1e-12
    assert np.max(np.abs(sl - lse)) < 1e-12


def test_queries_before_position_zero_attend_nothing():
    q, K, V = _rand(4, 2, 8), _rand(2, 1, 8), _rand(2, 1, 8)
    assert O.mtp_limits(2, 4) == [0, 0, 1, 2]
    o, lse = O.mtp_attention(q, K, V, 0.3, 2)
    assert np.all(o[:2] == 0) and np.all(np.isneginf(lse[:2]))
    assert np.isfinite(lse[2:]).all()


def test_pin_catches_an_off_by_one_limit():
    L, ql = 40, 4
    q, K, V = _rand(ql, 4, 8), _rand(L, 2, 8), _rand(L, 2, 8)
    # a plausible mistake: the query excludes its own position
    wrong = np.stack([O.attention(q[i], K, V, 0.3, 0, L - ql + i)[0] for i in range(ql)])
    ro, _ = _masked_route(q, K, V, 0.3, L)
    assert np.max(np.abs(wrong - ro)) > 1e-3
