"""Pins for the float64 oracle's attention and merge (CPU only).

Each check ties the oracle to something other than itself: a pure-Python
brute force, closed forms, torch's own scaled-dot-product attention in
float64, scipy's logsumexp, or an invariant the pages fix (merging the
shards reproduces full-context attention exactly).
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle as O

RNG = np.random.default_rng(1234)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# --------------------------------------------------------------------------
# brute force: pure Python, math.fsum, no numpy arithmetic
# --------------------------------------------------------------------------
def _brute(q, K, V, scale, lo, hi):
    hq, dk = q.shape
    hkv = K.shape[1]
    g = hq // hkv
    out, lses = [], []
    for h in range(hq):
        kv = h // g
        s = [scale * math.fsum(float(q[h, d]) * float(K[t, kv, d]) for d in range(dk))
             for t in range(lo, hi)]
        if not s:
            out.append([0.0] * V.shape[2])
            lses.append(-math.inf)
            continue
        m = max(s)
        e = [math.exp(x - m) for x in s]
        l = math.fsum(e)
        out.append([math.fsum(e[j] * float(V[lo + j, kv, d]) for j in range(len(e))) / l
                    for d in range(V.shape[2])])
        lses.append(m + math.log(l))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("L,hq,hkv,dk,dv,lo,hi", [
    (1, 2, 1, 3, 2, 0, 1),
    (5, 4, 2, 4, 3, 0, 5),
    (8, 4, 2, 3, 4, 2, 7),
    (8, 6, 3, 4, 4, 3, 8),
    (7, 4, 4, 2, 2, 0, 7),
    (6, 4, 1, 4, 3, 1, 4),
])
def test_brute_force(L, hq, hkv, dk, dv, lo, hi):
    q, K, V = _rand(hq, dk), _rand(L, hkv, dk), _rand(L, hkv, dv)
    scale = 0.7
    o, lse = O.attention(q, K, V, scale, lo, hi)
    ob, lb = _brute(q, K, V, scale, lo, hi)
    assert np.max(np.abs(o - ob)) < 1e-13
    assert np.max(np.abs(lse - lb)) < 1e-13


def test_single_token_returns_v():
    q, K, V = _rand(8, 16), _rand(1, 2, 16), _rand(1, 2, 12)
    scale = 0.25
    o, lse = O.attention(q, K, V, scale)
    for h in range(8):
        kv = h // 4
        assert np.array_equal(o[h], V[0, kv])
        assert lse[h] == pytest.approx(scale * float(np.dot(q[h], K[0, kv])), abs=1e-13)


def test_uniform_scores_give_mean_and_log_len():
    L = 37
    q = np.zeros((4, 8))
    K, V = _rand(L, 2, 8), _rand(L, 2, 5)
    o, lse = O.attention(q, K, V, 1.0, 3, 30)
    n = 27
    for h in range(4):
        assert np.allclose(o[h], V[3:30, h // 2].mean(axis=0), atol=1e-14)
        assert lse[h] == pytest.approx(math.log(n), abs=1e-14)


def test_two_tokens_closed_form():
    q, K, V = _rand(2, 6), _rand(2, 1, 6), _rand(2, 1, 3)
    scale = 1.3
    o, lse = O.attention(q, K, V, scale)
    for h in range(2):
        s0 = scale * float(q[h] @ K[0, 0])
        s1 = scale * float(q[h] @ K[1, 0])
        sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        want = sig * V[0, 0] + (1.0 - sig) * V[1, 0]
        assert np.allclose(o[h], want, atol=1e-14)
        assert lse[h] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), abs=1e-13)


def test_empty_range():
    q, K, V = _rand(4, 8), _rand(10, 2, 8), _rand(10, 2, 8)
    o, lse = O.attention(q, K, V, 1.0, 5, 5)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def _sdpa(q, K, V, scale):
    """torch SDPA in float64 on CPU, GQA by expanding the KV heads."""
    hq = q.shape[0]
    g = hq // K.shape[1]
    Kt = torch.from_numpy(np.repeat(K, g, axis=1)).permute(1, 0, 2)[None]
    Vt = torch.from_numpy(np.repeat(V, g, axis=1)).permute(1, 0, 2)[None]
    qt = torch.from_numpy(q)[None, :, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return out[0, :, 0, :].numpy()


@pytest.mark.parametrize("L,hq,hkv,d", [(512, 8, 2, 64), (4096, 64, 4, 128), (300, 16, 16, 32)])
def test_matches_torch_sdpa(L, hq, hkv, d):
    q, K, V = _rand(hq, d), _rand(L, hkv, d), _rand(L, hkv, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = O.attention(q, K, V, scale)
    assert np.max(np.abs(o - _sdpa(q, K, V, scale))) < 1e-12
    g = hq // hkv
    for h in range(hq):
        s = scale * (K[:, h // g, :] @ q[h])
        assert lse[h] == pytest.approx(logsumexp(s), abs=1e-11)


def test_mla_matches_sdpa_with_value_prefix():
    L, hq, dk, dv = 700, 16, 576, 512
    q, lat = _rand(hq, dk), _rand(L, dk)
    scale = 1.0 / math.sqrt(dk)
    o, lse = O.mla_attention(q, lat, scale, dv)
    qt = torch.from_numpy(q)[None, :, None, :]
    kt = torch.from_numpy(lat)[None, None].expand(1, hq, L, dk)
    vt = torch.from_numpy(lat[:, :dv].copy())[None, None].expand(1, hq, L, dv)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()
    assert o.shape == (hq, dv)
    assert np.max(np.abs(o - ref)) < 1e-12
    for h in range(hq):
        assert lse[h] == pytest.approx(logsumexp(scale * (lat @ q[h])), abs=1e-11)


# --------------------------------------------------------------------------
# the method's claim: merging the shards reproduces full attention
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L,N", [(512, 1), (512, 2), (513, 3), (512, 4), (100, 8), (37, 16), (5, 8)])
def test_sharded_merge_equals_unsharded(L, N):
    q, K, V = _rand(8, 16, scale=2.0), _rand(L, 2, 16), _rand(L, 2, 12)
    scale = 0.5
    starts = O.shard_starts([L - 1], N)[0]
    o_full, l_full = O.attention(q, K, V, scale)
    o, lse, parts, lses = O.sharded_attention(q, K, V, scale, starts, L)
    assert np.max(np.abs(o - o_full)) < 1e-12
    assert np.max(np.abs(lse - l_full)) < 1e-12
    # LSE identity against scipy: full LSE = log-sum-exp of the shard LSEs
    assert np.allclose(logsumexp(lses, axis=0), l_full, atol=1e-12)
    # every shard's partial is plain attention over its own range
    for i in range(N):
        lo, hi = O.shard_token_range(starts, i, L)
        oi, li = O.attention(q, K, V, scale, lo, hi)
        assert np.array_equal(parts[i], oi) and np.array_equal(lses[i], li)


def test_n1_is_plain_attention():
    q, K, V = _rand(4, 8), _rand(50, 1, 8), _rand(50, 1, 8)
    o, lse, _, _ = O.sharded_attention(q, K, V, 0.3, O.shard_starts([49], 1)[0], 50)
    o2, l2 = O.attention(q, K, V, 0.3)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)


def test_merge_empty_shards():
    parts = np.zeros((3, 2, 4))
    lses = np.full((3, 2), -np.inf)
    o, lse = O.merge(parts, lses)
    assert np.all(o == 0) and np.all(np.isneginf(lse)) and not np.isnan(o).any()
    p = _rand(2, 2, 4)
    l = _rand(2, 2)
    o1, l1 = O.merge(p, l)
    o2, l2 = O.merge(np.concatenate([p, np.full((1, 2, 4), 123.0)]),
                     np.concatenate([l, np.full((1, 2), -np.inf)]))
    assert np.allclose(o1, o2, atol=1e-15) and np.allclose(l1, l2, atol=1e-15)


def test_merge_weights_by_lse():
    # two partials with LSE a, b: weights are softmax([a, b]) (closed form)
    p = _rand(2, 1, 3)
    a, b = 1.7, -0.4
    o, lse = O.merge(p, np.array([[a], [b]]))
    wa = 1.0 / (1.0 + math.exp(b - a))
    assert np.allclose(o[0], wa * p[0, 0] + (1 - wa) * p[1, 0], atol=1e-15)
    assert lse[0] == pytest.approx(logsumexp([a, b]), abs=1e-15)


def test_needle_dominates():
    # a key aligned with the query far above the rest: O -> v_needle, within
    # the bound that follows from the score gap
    L, d = 2000, 64
    q, K, V = _rand(1, d), _rand(L, 1, d), _rand(L, 1, d)
    t_star = 1234
    K[t_star, 0] = 4.0 * q[0]
    scale = 1.0 / math.sqrt(d)
    o, _ = O.attention(q, K, V, scale)
    s = scale * (K[:, 0] @ q[0])
    gap = s[t_star] - np.max(np.delete(s, t_star))
    p_rest = (L - 1) * math.exp(-gap) / (1 + (L - 1) * math.exp(-gap))
    bound = p_rest * 2 * np.max(np.abs(V))
    assert np.max(np.abs(o[0] - V[t_star, 0])) <= bound + 1e-15
    assert gap > 10


def test_bf16_widening_matches_torch():
    x = torch.randn(4096, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits_to_f64(bits), x.to(torch.float64).numpy())
    special = torch.tensor([0.0, -0.0, 1.0, -2.5, 3.0e38, 1e-40], dtype=torch.bfloat16)
    sb = special.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits_to_f64(sb), special.to(torch.float64).numpy())


# --------------------------------------------------------------------------
# planted mistakes: copies of the definition with one plausible bug each must
# fail the pins above (so the pins can tell a wrong oracle from a right one)
# --------------------------------------------------------------------------
def _mutant(kind):
    def att(q, K, V, scale, lo=0, hi=None):
        hq, hkv = q.shape[0], K.shape[1]
        g = hq // hkv
        hi = K.shape[0] if hi is None else hi
        o = np.zeros((hq, V.shape[2]))
        lse = np.zeros(hq)
        for h in range(hq):
            kv = (h % hkv) if kind == "head_map" else h // g
            sc = 1.0 if kind == "no_scale" else scale
            s = sc * (K[lo:hi, kv] @ q[h])
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            o[h] = (e @ V[lo:hi, kv]) / (1.0 if kind == "no_norm" else l)
            lse[h] = (np.log(l) if kind == "lse_no_max" else m + np.log(l))
        return o, lse
    return att


@pytest.mark.parametrize("kind", ["head_map", "no_scale", "no_norm", "lse_no_max"])
def test_pins_catch_planted_mistakes(kind):
    q, K, V = _rand(4, 3), _rand(6, 2, 3), _rand(6, 2, 2)
    o, lse = _mutant(kind)(q, K, V, 0.6, 0, 6)
    ob, lb = _brute(q, K, V, 0.6, 0, 6)
    assert max(np.max(np.abs(o - ob)), np.max(np.abs(lse - lb))) > 1e-6
