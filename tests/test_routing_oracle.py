"""Pins for the oracle's routing and paged scatter (CPU only, bit-exact)."""
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_routing_golden(name):
    ctx = shards = None
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "ctx_len":
                ctx = int(parts[1])
            elif parts[0] == "shards":
                shards = int(parts[1])
            else:
                rows.append(tuple(int(x) for x in parts))
    return ctx, shards, rows


def test_page_example_200k_on_4():
    ctx, n, rows = _read_routing_golden("routing_200k_4.txt")
    starts = O.shard_starts([ctx], n)[0]
    for i, lo, hi in rows:
        assert O.shard_token_range(starts, i, ctx) == (lo, hi)
    # every token of the page's example routes to the shard the page names
    for t in (0, 1, 49999, 50000, 99999, 100000, 149999, 150000, 199999):
        i, p = O.owner(t, starts)
        lo, hi = [(r[1], r[2]) for r in rows if r[0] == i][0]
        assert lo <= t < hi and p == t - lo


@pytest.mark.parametrize("L0,N,reserve", [(0, 1, 3), (1, 4, 2), (5, 4, 3), (16, 4, 0), (17, 4, 5),
                                          (511, 4, 1), (100, 7, 10), (3, 16, 20), (64, 8, 64)])
def test_routing_partition_brute_force(L0, N, reserve):
    starts = O.shard_starts([L0], N)[0]
    C = O.shard_chunk(L0, N)
    assert C == max(1, -(-L0 // N))
    total = L0 + reserve
    cap = O.shard_capacity_tokens(L0, N, reserve)
    assert cap.sum() == total
    seen = {}
    for t in range(total):
        i, p = O.owner(t, starts)
        assert 0 <= i < N and 0 <= p < cap[i]
        assert (i, p) not in seen
        seen[(i, p)] = t
        # contiguous ranges: shard i's tokens are exactly starts[i] + 0..cap-1
        assert t == i * C + p
        # the owner is the only shard whose range holds t (last one open-ended)
        for j in range(N):
            lo = j * C
            hi = None if j == N - 1 else (j + 1) * C
            inside = lo <= t and (hi is None or t < hi)
            assert inside == (j == i)
    assert len(seen) == total
    # attended ranges tile [0, L) for any L
    for L in (0, L0, total):
        covered = []
        for i in range(N):
            lo, hi = O.shard_token_range(starts, i, L)
            covered.extend(range(lo, hi))
        assert covered == list(range(L))


def test_blocks_needed():
    bn = O.blocks_needed([511, 0, 100], 4, 16, 1)
    # 512 tokens -> 4 shards of 128 -> 8 blocks each
    assert bn[0].tolist() == [8, 8, 8, 8]
    # empty context: C = 1, one appended token lands in shard 0
    assert bn[1].tolist() == [1, 0, 0, 0]
    # 101 tokens, C = 25: 25, 25, 25, 26 tokens
    assert bn[2].tolist() == [2, 2, 2, 2]


def test_scatter_gather_roundtrip():
    # every token written by the scatter is read back from exactly the slot
    # that routing names, and nothing else in the pools changes
    rng = np.random.default_rng(5)
    B, N, Bs, hkv, d = 3, 3, 4, 2, 5
    ctx = [10, 3, 17]
    reserve = 2
    starts = O.shard_starts(ctx, N)
    counts = O.blocks_needed(ctx, N, Bs, reserve)
    tables, pools_k, pools_v = [], [], []
    for i in range(N):
        need = int(counts[:, i].sum())
        perm = rng.permutation(need + 3)
        t = np.full((B, max(1, counts[:, i].max())), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            t[b, :counts[b, i]] = perm[off:off + counts[b, i]]
            off += counts[b, i]
        tables.append(t)
        pools_k.append(np.full((need + 3, hkv, Bs, d), 0xAB, dtype=np.uint16))
        pools_v.append(np.full((need + 3, hkv, Bs, d), 0xCD, dtype=np.uint16))
    seq, pos = [], []
    for b in range(B):
        for t in range(ctx[b] + reserve):
            seq.append(b)
            pos.append(t)
    T = len(pos)
    k = rng.integers(0, 60000, size=(T, hkv, d)).astype(np.uint16)
    v = rng.integers(0, 60000, size=(T, hkv, d)).astype(np.uint16)
    O.scatter_gqa(pools_k, pools_v, starts, tables, Bs, seq, pos, k, v)
    written = [np.zeros(p.shape[0:1] + p.shape[2:3], dtype=bool) for p in pools_k]
    for j in range(T):
        b, t = seq[j], pos[j]
        i, p = O.owner(t, starts[b])
        phys = tables[i][b, p // Bs]
        assert np.array_equal(pools_k[i][phys, :, p % Bs], k[j])
        assert np.array_equal(pools_v[i][phys, :, p % Bs], v[j])
        assert not written[i][phys, p % Bs]
        written[i][phys, p % Bs] = True
    for i in range(N):
        assert np.all(pools_k[i].transpose(0, 2, 1, 3)[~written[i]] == 0xAB)
        assert np.all(pools_v[i].transpose(0, 2, 1, 3)[~written[i]] == 0xCD)


def test_planted_routing_mistakes_fail():
    # floor instead of ceiling for C, or a closed last shard, break the pins
    L0, N = 17, 4
    bad_c = max(1, L0 // N)
    good = O.shard_starts([L0], N)[0]
    assert list(good) != [i * bad_c for i in range(N)]
    starts = good
    t_append = L0
    i, _ = O.owner(t_append, starts)
    assert i == N - 1  # open-ended last shard takes the appended token


def _mla_scatter_case(scatter):
    """Scatter latent rows of three sequences into fragmented MLA pools with
    `scatter` and check every row against the layout [num_blocks, block_size,
    Dk] written out independently: row j of sequence b at global position t
    goes to shard i = min(t // C, N - 1) with C = max(1, ceil(ctx / N)), local
    position p = t - i * C, physical block tables[i][b, p // Bs] and slot
    p % Bs, i.e. flat row phys * Bs + slot of the pool viewed as [rows, Dk]
    (the view the kernels' TMA maps use). Canary values stay everywhere else."""
    rng = np.random.default_rng(11)
    B, N, Bs, dk = 3, 4, 8, 6
    ctx = [37, 5, 64]
    reserve = 3
    starts = O.shard_starts(ctx, N)
    counts = O.blocks_needed(ctx, N, Bs, reserve)
    tables, pools = [], []
    for i in range(N):
        need = int(counts[:, i].sum())
        cap = need + 5                       # holes: a fragmented pool
        perm = rng.permutation(cap)
        t = np.full((B, max(1, counts[:, i].max())), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            t[b, :counts[b, i]] = perm[off:off + counts[b, i]]
            off += counts[b, i]
        tables.append(t)
        pools.append(np.full((cap, Bs, dk), 0xBEEF, dtype=np.uint16))
    seq = [b for b in range(B) for _ in range(ctx[b] + reserve)]
    pos = [t for b in range(B) for t in range(ctx[b] + reserve)]
    lat = rng.integers(0, 60000, size=(len(pos), dk)).astype(np.uint16)
    scatter(pools, starts, tables, Bs, seq, pos, lat)
    written = [np.zeros(p.shape[0] * Bs, dtype=bool) for p in pools]
    for j, (b, t) in enumerate(zip(seq, pos)):
        C = max(1, -(-ctx[b] // N))
        i = min(t // C, N - 1)
        p = t - i * C
        phys = int(tables[i][b, p // Bs])
        row = phys * Bs + p % Bs
        flat = pools[i].reshape(-1, dk)
        if not np.array_equal(flat[row], lat[j]) or written[i][row]:
            return False
        written[i][row] = True
    return all(np.all(pools[i].reshape(-1, dk)[~written[i]] == 0xBEEF) for i in range(N))


def test_scatter_mla_layout_roundtrip():
    assert _mla_scatter_case(O.scatter_mla)


def test_scatter_mla_planted_mistakes_fail():
    # block and slot swapped in the write, or the slot taken from the global
    # position instead of the shard-local one: each must fail the pin above
    def swapped(pools, starts, tables, block_size, seq_ids, positions, latent_new):
        for j in range(len(positions)):
            b = int(seq_ids[j])
            i, phys, slot = O.paged_slot(int(positions[j]), starts[b], tables, b, block_size)
            pools[i][slot % pools[i].shape[0], phys % block_size, :] = latent_new[j]

    def global_slot(pools, starts, tables, block_size, seq_ids, positions, latent_new):
        for j in range(len(positions)):
            b, t = int(seq_ids[j]), int(positions[j])
            i, phys, _ = O.paged_slot(t, starts[b], tables, b, block_size)
            pools[i][phys, t % block_size, :] = latent_new[j]

    assert not _mla_scatter_case(swapped)
    assert not _mla_scatter_case(global_slot)
