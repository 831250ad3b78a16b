"""dcp_merge against the oracle's merge, and the work plan's invariants."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,B,H,D", [(1, 3, 4, 8), (2, 5, 16, 128), (8, 7, 128, 512), (16, 2, 8, 64),
                                     (32, 3, 5, 12), (40, 2, 3, 4)])
def test_merge_matches_oracle(N, B, H, D):
    g = torch.Generator().manual_seed(N * 1000 + B)
    parts = torch.randn((N, B, H, D), generator=g, dtype=torch.float32)
    lses = torch.randn((N, B, H), generator=g, dtype=torch.float32) * 20
    # empty shards (-inf) in places, and one row empty everywhere
    mask = torch.rand((N, B, H), generator=g) < 0.3
    lses[mask] = -float("inf")
    lses[:, 0, 0] = -float("inf")
    o = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    dcp.dcp_merge(parts.cuda(), lses.cuda(), o, lse)
    torch.cuda.synchronize()
    ro, rl = O.merge(parts.double().numpy(), lses.double().numpy())
    assert_close(o.cpu().numpy(), ro, "merged O", atol=1e-5)
    got = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(got[fin] - rl[fin]).max() < 1e-5
    assert np.all(o.cpu().numpy()[0, 0] == 0)


def _plan(st):
    ws = st.workspace.cpu().numpy()
    hdr = ws[:256].view(np.int32)
    n_items, n_lanes, n_ctas, total = (int(x) for x in hdr[:4])
    return ws, n_items, n_lanes, n_ctas, total


@pytest.mark.parametrize("name,over", [
    ("gqa_mid", dict(batch=5, ctx_kind="lognormal", median=2000, sigma=1.5, ctx_lo=0, ctx_hi=40000, shards=7)),
    ("gqa_tiny", dict(batch=1, ctx_fixed=20, shards=4)),        # fewer tiles than CTAs
    ("gqa_mid", {}),
])
def test_plan_covers_every_tile_once_and_balances(name, over):
    wl = configs.get(name).with_(**over)
    st = DecodeState(wl)
    st.step()
    torch.cuda.synchronize()
    ws, n_items, n_lanes, n_ctas, total = _plan(st)
    # mirror of the layout in the library's workspace header
    lanes_off = 256
    lanes = ws[lanes_off:lanes_off + 32 * n_lanes].view(np.int32).reshape(n_lanes, 8)
    items_off = (lanes_off + 32 * n_lanes + 255) // 256 * 256
    items = ws[items_off:items_off + 16 * n_items].view(np.int32).reshape(n_items, 4)
    max_items = n_lanes + n_ctas
    cta_off = (items_off + 16 * max_items + 255) // 256 * 256
    cta_begin = ws[cta_off:cta_off + 4 * (n_ctas + 1)].view(np.int32)
    tiles = lanes[:, 3]
    assert tiles.sum() == total
    tile = 16
    assert np.array_equal(tiles, (lanes[:, 1] - lanes[:, 0] + tile - 1) // tile)
    covered = [np.zeros(t, dtype=np.int32) for t in tiles]
    per_cta = np.zeros(n_ctas, dtype=np.int64)
    assert cta_begin[0] == 0 and cta_begin[n_ctas] == n_items
    assert np.all(np.diff(cta_begin) >= 0)
    for c in range(n_ctas):
        for k in range(cta_begin[c], cta_begin[c + 1]):
            lane, t0, t1, _ = items[k]
            assert 0 <= t0 < t1 <= tiles[lane]
            covered[lane][t0:t1] += 1
            per_cta[c] += t1 - t0
    assert all((cv == 1).all() for cv in covered)
    busy = per_cta[per_cta > 0]
    assert busy.max() - busy.min() <= 1
    # a lane is written directly iff one item covers it
    for lane in range(n_lanes):
        n = lanes[lane, 5]
        ks = [k for k in range(n_items) if items[k, 0] == lane]
        assert len(ks) == n
        assert all((items[k, 3] == -1) == (n == 1) for k in ks)
