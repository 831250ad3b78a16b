"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the attention method: no routing, no
softmax, no merge. It only draws numbers. Both sides call the same functions
here, each on its own device, and get identical values:

* Every KV / query element is a pure function of (seed, stream, logical
  coordinates) -- a counter-based draw -- so the GPU can generate the full
  pools chunk by chunk while the CPU regenerates only the rows it checks.
* The draw is integer-only up to one float32 multiply and the bf16 rounding,
  both of which round identically on CPU and GPU: four 16-bit uniforms from
  two 32-bit integer hashes (Thomas Mueller's 32-bit mixing function, with
  the published 0x45d9f3b multiplier), summed (an Irwin-Hall(4) variate:
  mean 0 and variance 1 after centring and scaling, tails cut at +-3.46),
  scaled in float32 and rounded to bf16. This stands in for N(0, 1).
* Context lengths and block-table permutations come from numpy's
  default_rng(seed); they are plain integers.
"""
from __future__ import annotations

import math

import numpy as np
import torch

MASK32 = 0xFFFFFFFF
_MUL = 0x45D9F3B                       # < 2**27, so x * _MUL < 2**59: no int64 overflow
_IH4_MEAN = 4 * 65535 // 2             # 131070
_IH4_INV_STD = 1.0 / math.sqrt((2.0 ** 32 - 1.0) / 3.0)

# Counter streams: one per logical tensor.
STREAM_Q = 1
STREAM_K = 2
STREAM_V = 3
STREAM_LATENT = 4
STREAM_Q_MLA = 5

# Field widths of the logical coordinates packed into one int64 counter.
T_BITS = 20          # positions < 2**20 = 1,048,576
H_BITS = 8           # heads < 256
D_BITS = 10          # feature index < 1024


def _mix32_int(x: int) -> int:
    x &= MASK32
    x = (((x >> 16) ^ x) * _MUL) & MASK32
    x = (((x >> 16) ^ x) * _MUL) & MASK32
    return ((x >> 16) ^ x) & MASK32


def _mix32_(x: torch.Tensor) -> torch.Tensor:
    """In-place 32-bit mix of an int64 tensor holding values in [0, 2**32)."""
    x ^= x >> 16
    x *= _MUL
    x &= MASK32
    x ^= x >> 16
    x *= _MUL
    x &= MASK32
    x ^= x >> 16
    return x


def _keys(seed: int, stream: int) -> tuple[int, int]:
    k0 = _mix32_int(_mix32_int(seed * 0x9E37 + 0x85EB) ^ (stream * 0x27D4EB2F))
    k1 = _mix32_int(k0 ^ 0x165667B1)
    return k0, k1


def _row_key(rows: torch.Tensor, k: int) -> torch.Tensor:
    lo = rows & MASK32
    inner = _mix32_((rows >> 32) ^ k)
    return _mix32_(lo ^ inner)


def counter_normal_bf16(rows: torch.Tensor, cols: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """bf16 draws (approximately N(0,1)) for every (row, col) counter pair.

    rows: int64 [R] (< 2**62), cols: int64 [C] (< 2**32); returns [R, C] bf16
    on the rows' device. Each element hashes (row key XOR col) twice.
    """
    if rows.dtype != torch.int64 or cols.dtype != torch.int64:
        raise TypeError("counters must be int64")
    k0, k1 = _keys(seed, stream)
    x = _mix32_(_row_key(rows, k0)[:, None] ^ cols[None, :])
    y = _mix32_(_row_key(rows, k1)[:, None] ^ cols[None, :])
    s = x & 0xFFFF
    s += x >> 16
    s += y & 0xFFFF
    s += y >> 16
    del x, y
    s -= _IH4_MEAN
    f = s.to(torch.float32)
    del s
    f *= torch.tensor(_IH4_INV_STD, dtype=torch.float32, device=rows.device)
    return f.to(torch.bfloat16)


def _hd_index(n_heads: int, width: int, device) -> torch.Tensor:
    if n_heads > (1 << H_BITS) or width > (1 << D_BITS):
        raise ValueError("head/feature index out of the counter's field")
    h = torch.arange(n_heads, dtype=torch.int64, device=device)
    d = torch.arange(width, dtype=torch.int64, device=device)
    return ((h[:, None] << D_BITS) | d[None, :]).reshape(-1)


def query(seed: int, batch_ids, n_heads: int, width: int, device="cpu", stream: int = STREAM_Q):
    """Decode queries [len(batch_ids), n_heads, width] bf16 for the given sequences."""
    b = torch.as_tensor(batch_ids, dtype=torch.int64, device=device).reshape(-1)
    out = counter_normal_bf16(b, _hd_index(n_heads, width, device), seed, stream)
    return out.view(b.numel(), n_heads, width)


def query_tokens(seed: int, batch_ids, q_len: int, n_heads: int, width: int, device="cpu",
                 stream: int = STREAM_Q):
    """Queries of q_len new tokens per sequence: [len(batch_ids), q_len, n_heads, width] bf16.

    Query token j of sequence b draws from counter row b + j * 2**32, so token 0
    is the one-token query of sequence b (query(seed, [b], ...))."""
    b = torch.as_tensor(batch_ids, dtype=torch.int64, device=device).reshape(-1)
    j = torch.arange(q_len, dtype=torch.int64, device=device)
    rows = (b[:, None] + (j[None, :] << 32)).reshape(-1)
    out = counter_normal_bf16(rows, _hd_index(n_heads, width, device), seed, stream)
    return out.view(b.numel(), q_len, n_heads, width)


def kv_tokens(seed: int, stream: int, batch_ids, positions, n_heads: int, width: int,
              device="cpu", chunk: int = 1 << 14) -> torch.Tensor:
    """Per-token KV rows [T, n_heads, width] bf16 for (batch_ids[j], positions[j])."""
    b = torch.as_tensor(batch_ids, dtype=torch.int64, device=device).reshape(-1)
    t = torch.as_tensor(positions, dtype=torch.int64, device=device).reshape(-1)
    if b.numel() != t.numel():
        raise ValueError("batch_ids and positions differ in length")
    if t.numel() and (int(t.max()) >= (1 << T_BITS) or int(t.min()) < 0):
        raise ValueError("position outside the counter's field")
    hd = _hd_index(n_heads, width, device)
    out = torch.empty((t.numel(), n_heads, width), dtype=torch.bfloat16, device=device)
    flat = out.view(t.numel(), n_heads * width)
    for s in range(0, t.numel(), chunk):
        rows = (b[s:s + chunk] << T_BITS) | t[s:s + chunk]
        flat[s:s + chunk] = counter_normal_bf16(rows, hd, seed, stream)
    return out


def sequence_kv(seed: int, stream: int, b: int, lo: int, hi: int, n_heads: int, width: int,
                device="cpu") -> torch.Tensor:
    """KV rows of sequence b at positions [lo, hi): [hi - lo, n_heads, width] bf16."""
    pos = torch.arange(lo, hi, dtype=torch.int64, device=device)
    return kv_tokens(seed, stream, torch.full_like(pos, b), pos, n_heads, width, device)


def e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """FP8 E4M3 codes (uint8) of bf16 values, rounded to nearest even, with
    magnitudes above 448 saturated to +-448 and NaN mapped to 0.

    Integer operations only on the bf16 bit patterns, so CPU and GPU give the
    same codes for the same draws (an 8-bit cache is filled on the device
    while the checker decodes the same codes on the host)."""
    if x.dtype != torch.bfloat16:
        raise TypeError("bf16 input expected")
    b = x.contiguous().view(torch.int16).to(torch.int64) & 0xFFFF
    sign = (b >> 8) & 0x80
    e = (b >> 7) & 0xFF                    # bf16 exponent field (bias 127)
    m = b & 0x7F                           # 7 mantissa bits
    E = e - 127                            # unbiased exponent
    # normal results: exponent field E + 7 in [1, 15], 3 mantissa bits
    keep = m >> 4
    rem = m & 0xF
    up = (rem > 8) | ((rem == 8) & ((keep & 1) == 1))
    normal = ((E + 7) << 3) + keep + up.to(torch.int64)      # a mantissa carry bumps the exponent
    # subnormal results (E < -6): round (1.m) * 2^E / 2^-9 = (128 + m) >> (-E - 2)
    sh = (-E - 2).clamp(min=5, max=40)
    full = 128 + m
    q = full >> sh
    r = full - (q << sh)
    half = torch.ones_like(sh) << (sh - 1)
    q = q + ((r > half) | ((r == half) & ((q & 1) == 1))).to(torch.int64)
    mag = torch.where(E >= -6, normal, q)
    mag = torch.where(e == 0, torch.zeros_like(mag), mag)    # zeros and bf16 subnormals (< 2^-126) -> 0
    mag = torch.where(mag > 0x7E, torch.full_like(mag, 0x7E), mag)   # saturate at 448 (0x7F is NaN)
    mag = torch.where(e == 0xFF, torch.where(m == 0, torch.full_like(mag, 0x7E), torch.zeros_like(mag)), mag)
    return (sign | mag).to(torch.uint8)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (as numpy, on the host)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# Integers: lengths and block-table permutations
# ---------------------------------------------------------------------------
def lognormal_lengths(seed: int, batch: int, median: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    """Context lengths: clip(rint(median * exp(sigma * z)), lo, hi), z ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(batch)
    return np.clip(np.rint(median * np.exp(sigma * z)), lo, hi).astype(np.int64)


def block_tables(seed: int, counts: np.ndarray, capacity_factor: float = 1.0):
    """Random physical block assignment for every (sequence, shard).

    counts: int [B, N], the number of logical blocks each sequence needs in
    each shard (computed by the caller). Shard i's pool gets
    ceil(capacity_factor * sum_b counts[b, i]) blocks (at least 1); its blocks
    are handed out from a random permutation of the pool, so a factor above 1
    leaves holes (a fragmented pool). Returns a list over shards of
    (num_blocks, table) with table int32 [B, max(1, max_b counts[b, i])],
    unused entries -1.
    """
    counts = np.asarray(counts, dtype=np.int64)
    if counts.ndim != 2 or (counts < 0).any():
        raise ValueError("counts must be a non-negative [B, N] array")
    rng = np.random.default_rng(seed)
    out = []
    B, N = counts.shape
    for i in range(N):
        need = int(counts[:, i].sum())
        cap = max(1, int(math.ceil(need * capacity_factor)))
        perm = rng.permutation(cap)[:need].astype(np.int32)
        width = max(1, int(counts[:, i].max()) if B else 1)
        table = np.full((B, width), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            n = int(counts[b, i])
            table[b, :n] = perm[off:off + n]
            off += n
        out.append((cap, table))
    return out


def needle_plan(seed: int, seq_lens, per_seq: int, q_heads: int) -> dict:
    """Planted "needle" keys: for each sequence, `per_seq` (position, query
    head) pairs drawn uniformly from [0, seq_len) x [0, q_heads)."""
    rng = np.random.default_rng(seed + 7919)
    plan = {}
    for b, L in enumerate(seq_lens):
        L = int(L)
        if L <= 0:
            continue
        n = min(per_seq, L)
        pos = rng.choice(L, size=n, replace=False)
        heads = rng.integers(0, q_heads, size=n)
        plan[b] = sorted((int(t), int(h)) for t, h in zip(pos, heads))
    return plan


def plant_needles(rows: torch.Tensor, batch_ids, positions, q: torch.Tensor, plan: dict, q_heads: int,
                  alpha: float = 4.0) -> torch.Tensor:
    """Replace the key rows of planted positions by alpha * q[b, h] (bf16).

    rows: [T, Hkv, Dk] (GQA keys) or [T, Dk] (MLA latent); q: [B, Hq, Dk] on
    the rows' device. GQA puts the needle in KV head h // (Hq / Hkv). alpha is
    a power of two, so the product is exact in bf16 on every device.
    """
    if not plan:
        return rows
    b = torch.as_tensor(batch_ids, dtype=torch.int64, device=rows.device).reshape(-1)
    t = torch.as_tensor(positions, dtype=torch.int64, device=rows.device).reshape(-1)
    for bb, needles in plan.items():
        for tt, h in needles:
            idx = torch.nonzero((b == bb) & (t == tt)).reshape(-1)
            if idx.numel() == 0:
                continue
            val = (q[bb, h].to(torch.float32) * alpha).to(torch.bfloat16)
            if rows.dim() == 3:
                kvh = h // (q_heads // rows.shape[1])
                rows[idx, kvh, :] = val
            else:
                rows[idx, :] = val
    return rows
