"""The seeded input module: counter-based draws are a pure function of the
logical coordinates (so the GPU fill and the CPU oracle see the same bits),
with the intended first moments; needles replace exactly the planned rows."""
import numpy as np
import torch

from sequence_sharded_decode_gb300 import configs, inputs


def test_draw_depends_only_on_coordinates():
    a = inputs.kv_tokens(0, inputs.STREAM_K, [3, 3, 5], [10, 11, 7], 4, 128)
    b = inputs.sequence_kv(0, inputs.STREAM_K, 3, 9, 12, 4, 128)
    c = inputs.sequence_kv(0, inputs.STREAM_K, 5, 7, 8, 4, 128)
    assert torch.equal(a[0], b[1]) and torch.equal(a[1], b[2]) and torch.equal(a[2], c[0])
    # chunking does not matter
    d = inputs.kv_tokens(0, inputs.STREAM_V, [1] * 50, list(range(50)), 2, 64, chunk=7)
    e = inputs.kv_tokens(0, inputs.STREAM_V, [1] * 50, list(range(50)), 2, 64)
    assert torch.equal(d, e)


def test_streams_and_seeds_differ():
    k = inputs.sequence_kv(0, inputs.STREAM_K, 0, 0, 64, 2, 64).float()
    v = inputs.sequence_kv(0, inputs.STREAM_V, 0, 0, 64, 2, 64).float()
    k1 = inputs.sequence_kv(1, inputs.STREAM_K, 0, 0, 64, 2, 64).float()
    assert abs(float((k * v).mean())) < 0.05 and abs(float((k * k1).mean())) < 0.05


def test_moments_of_the_normal_stand_in():
    x = inputs.sequence_kv(0, inputs.STREAM_LATENT, 2, 0, 4096, 1, 576).float()
    assert abs(float(x.mean())) < 0.01
    assert abs(float(x.std()) - 1.0) < 0.01
    assert float(x.abs().max()) <= 3.47


def test_lognormal_lengths_of_the_presets():
    ctx = configs.get("mla_decode").ctx_lens()
    assert ctx.shape == (64,) and ctx.min() >= 4096 and ctx.max() <= 262144
    assert int(ctx.sum()) == 5651643
    assert int(configs.get("mla_high_concurrency").ctx_lens().sum()) == 43050767
    assert abs(np.median(configs.get("mla_high_concurrency").ctx_lens()) / 67000 - 1) < 0.1


def test_block_tables_are_permutations():
    counts = np.array([[3, 0], [2, 5], [0, 1]])
    tabs = inputs.block_tables(4, counts, 1.25)
    for i, (cap, tab) in enumerate(tabs):
        used = np.concatenate([tab[b, :counts[b, i]] for b in range(3)])
        assert len(set(used.tolist())) == len(used) == counts[:, i].sum()
        assert used.min() >= 0 and used.max() < cap
        assert cap == int(np.ceil(counts[:, i].sum() * 1.25)) or cap == 1


def test_plant_needles_replaces_only_planned_rows():
    wl = configs.get("gqa_tiny").with_(needles=3)
    plan = wl.needle_plan()
    q = inputs.query(wl.seed, [0], wl.q_heads, wl.dk)
    L = 512
    k = inputs.sequence_kv(wl.seed, inputs.STREAM_K, 0, 0, L, wl.kv_heads, wl.dk)
    k2 = inputs.plant_needles(k.clone(), np.zeros(L), np.arange(L), q, plan, wl.q_heads)
    changed = (k2 != k).any(dim=2).nonzero().tolist()
    want = sorted((t, h // 4) for t, h in plan[0])
    assert sorted(tuple(x) for x in changed) == want
    for t, h in plan[0]:
        assert torch.equal(k2[t, h // 4].float(), 4.0 * q[0, h].float())


def test_e4m3_codes_match_torch_rounding_for_every_bf16_in_range():
    # every bf16 bit pattern whose value is finite and at most 448 in magnitude
    bits = torch.arange(65536, dtype=torch.int64).to(torch.int16)
    x = bits.view(torch.bfloat16)
    f = x.to(torch.float32)
    ok = torch.isfinite(f) & (f.abs() <= 448)
    ours = inputs.e4m3_codes(x[ok])
    ref = f[ok].to(torch.float8_e4m3fn).view(torch.uint8)
    # torch keeps the sign of values that round to zero; so do we
    assert torch.equal(ours, ref)


def test_e4m3_codes_saturate_and_clear_nan():
    x = torch.tensor([1000.0, -1e30, float("inf"), float("-inf"), float("nan"), 449.0], dtype=torch.bfloat16)
    c = inputs.e4m3_codes(x).tolist()
    assert c[:4] == [0x7E, 0xFE, 0x7E, 0xFE]
    assert c[4] & 0x7F == 0
    assert c[5] == 0x7E
