"""Pins for the oracle's 8-bit (FP8 E4M3) cache decoding (CPU only): every
code against torch's float8_e4m3fn, closed-form values of the format, and
attention over a decoded cache against attention over the same values."""
import math

import numpy as np
import torch

import oracle as O


def test_every_code_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                                  # 0x7F and 0xFF only
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_closed_form_codes():
    v = lambda c: float(O.e4m3_to_f64(np.array([c], dtype=np.uint8))[0])
    assert v(0x7E) == 448.0                                # largest finite: 1.75 * 2^8
    assert v(0x38) == 1.0                                  # exponent field 7 = bias
    assert v(0x08) == 2.0 ** -6                            # smallest normal
    assert v(0x07) == 7 / 8 * 2.0 ** -6                    # largest subnormal
    assert v(0x01) == 2.0 ** -9                            # smallest subnormal
    assert v(0x00) == 0.0 and v(0x80) == 0.0 and math.copysign(1, v(0x80)) < 0
    assert v(0xB8) == -1.0 and v(0xFE) == -448.0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))


def test_positive_codes_are_increasing_and_symmetric():
    pos = O.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    neg = O.e4m3_to_f64(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)


def test_scaled_cache_attention_equals_attention_on_values():
    rng = np.random.default_rng(5)
    kc = rng.integers(0, 0x7F, size=(40, 2, 16)).astype(np.uint8) | (rng.integers(0, 2, (40, 2, 16)) << 7).astype(np.uint8)
    vc = rng.integers(0, 0x7F, size=(40, 2, 16)).astype(np.uint8)
    K, V = O.fp8_kv(kc, vc, 0.25, 3.0)
    assert np.array_equal(K, 0.25 * O.e4m3_to_f64(kc)) and np.array_equal(V, 3.0 * O.e4m3_to_f64(vc))
    q = rng.standard_normal((8, 16))
    o, lse = O.attention(q, K, V, 0.1)
    # by hand for one head: softmax over the decoded, scaled keys
    s = 0.1 * (K[:, 0, :] @ q[0])
    w = np.exp(s - s.max())
    assert np.allclose(o[0], (w[:, None] * V[:, 0, :]).sum(0) / w.sum(), atol=1e-12)
