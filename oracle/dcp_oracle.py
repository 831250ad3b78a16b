"""Float64 CPU oracle for sequence-sharded decode attention (DCP).

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module:
only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may call it. It shares no code with the CUDA library or its Python
binding; it reads plain numpy arrays (bf16 data arrives as raw uint16 bit
patterns and is widened here, exactly, to float64).

What the method computes, and the passages each function follows:

* Contiguous token ranges per shard -- Qiita write-up "vLLMの-dcpが長文脈の
  KVキャッシュ重複を消して3倍速くする", section "トークンの区間でGPUに割り振る"
  (a 200K-token request on 4 GPUs: GPU0 holds tokens 0-50K, GPU1 50K-100K,
  each GPU one contiguous interval); "Inference Systems Infrastructure Notes
  (7): DCP", section 2 (every GPU holds only its [start:end] slice).
* Per-shard partial attention over the local KV slice, then an exact merge of
  the partials by online-softmax reweighting -- the same Qiita section (the
  three steps: gather the one-token query, partial attention on the local
  slice, combine the partial results with online-softmax reweighting) and
  "Inference Systems Infrastructure Notes (7): DCP", section 2 (slices
  processed in parallel, then reassembled into the full attention result).
* The whole point of the merge is that it is exact: the sharded result is the
  plain full-context softmax attention. So `attention` below is that plain
  definition, and `sharded_attention` + `merge` are the method's steps,
  checked against it.
* MLA: one latent KV head ("effectively one KV head" -- Qiita section
  "なぜテンソル並列だとKVキャッシュが二重に載るのか"). Reading taken where the
  pages are silent: the key is the whole cached latent row (576 wide), the
  value is its first 512 entries, and the query is already absorbed (576 wide
  per head).

Readings where the pages are silent (each also listed in the design notes):
  chunk C = max(1, ceil(L0 / N)); shard i < N-1 owns [i*C, (i+1)*C); the last
  shard is open-ended and receives every later token; the appended token is
  attended in its own step; natural-log LSE; an empty shard has LSE = -inf
  and O = 0; GQA head h reads KV head floor(h / g) with g = Hq / Hkv.

Parity pins for every function here live in tests/test_oracle.py and
tests/test_routing_oracle.py; none of the functions is unpinned.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -math.inf


# ---------------------------------------------------------------------------
# bf16 widening (exact)
# ---------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) to float64 exactly.

    A bf16 value is the upper half of the IEEE binary32 with the same bits, so
    shifting the pattern left by 16 gives the float32 exactly; float32 ->
    float64 is exact as well.
    """
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Step a1: contiguous sharding of the token axis (routing)
# ---------------------------------------------------------------------------
def shard_chunk(ctx_len: int, n_shards: int) -> int:
    """Tokens per shard for a sequence whose context before decoding is L0.

    The pages show equal contiguous ranges (200K tokens on 4 GPUs -> 50K each);
    where N does not divide L0 the plainest reading is the ceiling, so every
    shard but the last holds exactly C tokens. C >= 1 keeps the routing
    defined for an empty context.
    """
    if n_shards < 1:
        raise ValueError("n_shards must be >= 1")
    if ctx_len < 0:
        raise ValueError("ctx_len must be >= 0")
    return max(1, -(-ctx_len // n_shards))


def shard_starts(ctx_lens, n_shards: int) -> np.ndarray:
    """Global start position of every shard, int32 [B, N]: start_i = i * C."""
    ctx = [int(x) for x in ctx_lens]
    out = np.zeros((len(ctx), n_shards), dtype=np.int32)
    for b, L0 in enumerate(ctx):
        c = shard_chunk(L0, n_shards)
        for i in range(n_shards):
            out[b, i] = i * c
    return out


def owner(t: int, starts_b) -> tuple[int, int]:
    """Shard that owns global position t, and t's position inside that shard.

    The owner is the last shard whose start is <= t: shards before the last
    hold [start_i, start_{i+1}); the last shard is open-ended, so a token
    appended after the prefill lands there (reading: the pages do not say
    where new decode tokens go).
    """
    if t < 0:
        raise ValueError("negative position")
    i_own = 0
    for i, s in enumerate(starts_b):
        if int(s) <= t:
            i_own = i
    return i_own, t - int(starts_b[i_own])


def shard_capacity_tokens(ctx_len: int, n_shards: int, reserve: int) -> np.ndarray:
    """Tokens each shard must hold for L0 context tokens plus `reserve` appends.

    Shard i < N-1 holds positions [i*C, (i+1)*C) that fall below L0 + reserve;
    the last shard holds everything from (N-1)*C up to L0 + reserve.
    """
    c = shard_chunk(ctx_len, n_shards)
    total = ctx_len + reserve
    cap = np.zeros(n_shards, dtype=np.int64)
    for i in range(n_shards):
        lo = i * c
        hi = total if i == n_shards - 1 else min((i + 1) * c, total)
        cap[i] = max(0, hi - lo)
    return cap


def blocks_needed(ctx_lens, n_shards: int, block_size: int, reserve: int) -> np.ndarray:
    """Paged blocks per (sequence, shard): ceil(capacity / block_size), int32 [B, N]."""
    ctx = [int(x) for x in ctx_lens]
    out = np.zeros((len(ctx), n_shards), dtype=np.int32)
    for b, L0 in enumerate(ctx):
        cap = shard_capacity_tokens(L0, n_shards, reserve)
        out[b] = [-(-int(x) // block_size) for x in cap]
    return out


def shard_token_range(starts_b, i: int, seq_len: int) -> tuple[int, int]:
    """Global [lo, hi) of the tokens shard i attends for a sequence of length L."""
    n = len(starts_b)
    lo = int(starts_b[i])
    hi = seq_len if i == n - 1 else int(starts_b[i + 1])
    lo = min(lo, seq_len)
    hi = min(hi, seq_len)
    return lo, max(lo, hi)


# ---------------------------------------------------------------------------
# Step a2: where a token's K/V lands in the paged pools (CPU scatter)
# ---------------------------------------------------------------------------
def paged_slot(t: int, starts_b, tables, b: int, block_size: int) -> tuple[int, int, int]:
    """(shard, physical block, slot) of global position t of sequence b.

    `tables[i]` is shard i's block table, int32 [B, max_blocks], mapping the
    shard-local logical block index to a physical block of shard i's pool.
    """
    i, p = owner(t, starts_b)
    logical = p // block_size
    slot = p % block_size
    phys = int(tables[i][b, logical])
    return i, phys, slot


def scatter_gqa(pools_k, pools_v, starts, tables, block_size, seq_ids, positions, k_new, v_new):
    """Write tokens into GQA pools laid out [num_blocks, Hkv, block_size, D].

    pools_* are lists (one per shard) of arrays of any dtype (bit patterns are
    copied as they are). k_new/v_new are [T, Hkv, D] in the pools' dtype.
    """
    for j in range(len(positions)):
        b = int(seq_ids[j])
        i, phys, slot = paged_slot(int(positions[j]), starts[b], tables, b, block_size)
        pools_k[i][phys, :, slot, :] = k_new[j]
        pools_v[i][phys, :, slot, :] = v_new[j]


def scatter_mla(pools, starts, tables, block_size, seq_ids, positions, latent_new):
    """Write latent rows into MLA pools laid out [num_blocks, block_size, Dk]."""
    for j in range(len(positions)):
        b = int(seq_ids[j])
        i, phys, slot = paged_slot(int(positions[j]), starts[b], tables, b, block_size)
        pools[i][phys, slot, :] = latent_new[j]


# ---------------------------------------------------------------------------
# Steps a4/a5 (and the unsharded definition they must reproduce)
# ---------------------------------------------------------------------------
def attention(q, K, V, scale: float, lo: int = 0, hi: int | None = None):
    """Plain softmax attention of one decode query over tokens [lo, hi).

    q: [Hq, Dk]; K: [L, Hkv, Dk]; V: [L, Hkv, Dv] (float64). Head h uses KV head
    floor(h / g), g = Hq / Hkv (consecutive grouping). Returns O [Hq, Dv] and
    the natural-log LSE [Hq]:

        s_t = scale * <q_h, k_t>,  m = max_t s_t,  l = sum_t exp(s_t - m)
        O_h = sum_t exp(s_t - m) v_t / l,  LSE_h = m + ln l.

    An empty range gives O = 0 and LSE = -inf (an empty shard contributes
    nothing to the merge).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, dk = q.shape
    L, hkv, dk2 = K.shape
    if dk2 != dk:
        raise ValueError("q and K widths differ")
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    dv = V.shape[2]
    hi = L if hi is None else hi
    lo = max(0, min(lo, L))
    hi = max(lo, min(hi, L))
    g = hq // hkv
    O = np.zeros((hq, dv), dtype=np.float64)
    lse = np.full(hq, NEG_INF, dtype=np.float64)
    if hi == lo:
        return O, lse
    for kv in range(hkv):
        qh = q[kv * g:(kv + 1) * g]                      # [g, Dk]
        s = scale * (qh @ K[lo:hi, kv, :].T)             # [g, n]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        O[kv * g:(kv + 1) * g] = (e @ V[lo:hi, kv, :]) / l
        lse[kv * g:(kv + 1) * g] = (m + np.log(l))[:, 0]
    return O, lse


def mla_attention(q, latent, scale: float, dv: int = 512, lo: int = 0, hi: int | None = None):
    """MLA-absorbed decode attention: one latent KV head.

    q: [Hq, Dk] (absorbed query, Dk = latent width); latent: [L, Dk]. The key
    is the whole latent row; the value is its first `dv` entries.
    """
    latent = np.asarray(latent, dtype=np.float64)
    K = latent[:, None, :]
    V = latent[:, None, :dv]
    return attention(q, K, V, scale, lo, hi)


# ---------------------------------------------------------------------------
# Step a6: the merge of per-shard partials
# ---------------------------------------------------------------------------
def merge(o_parts, lses):
    """Combine N partial results by LSE reweighting.

    o_parts: [N, ..., Dv]; lses: [N, ...]. For each row:
        M = max_i LSE_i,  w_i = exp(LSE_i - M),
        O = sum_i w_i O_i / sum_i w_i,  LSE = M + ln sum_i w_i.
    Rows where every shard is empty (all LSE = -inf) give O = 0, LSE = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    M = lses.max(axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - Ms[None]), 0.0)
    wsum = w.sum(axis=0)
    safe = np.where(wsum > 0, wsum, 1.0)
    O = (w[..., None] * o_parts).sum(axis=0) / safe[..., None]
    O = np.where(finite[..., None], O, 0.0)
    lse = np.where(finite, Ms + np.log(safe), NEG_INF)
    return O, lse


def sharded_attention(q, K, V, scale: float, starts_b, seq_len: int):
    """The method end to end for one sequence: partial per shard, then merge.

    Returns (O, LSE, per-shard O_i, per-shard LSE_i).
    """
    parts, lses = [], []
    for i in range(len(starts_b)):
        lo, hi = shard_token_range(starts_b, i, seq_len)
        o_i, l_i = attention(q, K, V, scale, lo, hi)
        parts.append(o_i)
        lses.append(l_i)
    O, lse = merge(np.stack(parts), np.stack(lses))
    return O, lse, np.stack(parts), np.stack(lses)


# ---------------------------------------------------------------------------
# Multi-token decode queries (speculative / multi-token-prediction steps)
# ---------------------------------------------------------------------------
# The pages name speculative decoding and MTP as what DCP is to be combined
# with next (Qiita write-up, section "実務でどう見るか"; "Inference Systems
# Infrastructure Notes (7): DCP", section 5) but give no formula. Reading
# taken: a step that verifies q_len new tokens of sequence b appends all of
# them (seq_len counts them), and query token i sits at global position
# seq_len - q_len + i and attends every token at or before its own position
# (causal among the new tokens), exactly as q_len consecutive one-token decode
# steps would. Under sharding each query is routed like a one-token query
# whose sequence ends at its own position; the merge is unchanged.
def mtp_limits(seq_len: int, q_len: int) -> list[int]:
    """Exclusive causal limit of each query token: seq_len - q_len + i + 1,
    floored at 0 (a query before position 0 attends nothing)."""
    if q_len < 1:
        raise ValueError("q_len must be >= 1")
    return [max(0, int(seq_len) - q_len + i + 1) for i in range(q_len)]


def mtp_attention(q, K, V, scale: float, seq_len: int):
    """Unsharded attention of q_len query tokens q [q_len, Hq, Dk] over the
    logical K/V of one sequence, each query causal at its own position.
    Returns O [q_len, Hq, Dv] and LSE [q_len, Hq]."""
    q = np.asarray(q, dtype=np.float64)
    outs, lses = [], []
    for i, hi in enumerate(mtp_limits(seq_len, q.shape[0])):
        o_i, l_i = attention(q[i], K, V, scale, 0, hi)
        outs.append(o_i)
        lses.append(l_i)
    return np.stack(outs), np.stack(lses)


def sharded_mtp_attention(q, K, V, scale: float, starts_b, seq_len: int):
    """The method for q_len query tokens of one sequence: per query token,
    partial attention on every shard's range clipped to the query's causal
    limit, then the LSE merge. Returns (O [q_len, Hq, Dv], LSE [q_len, Hq],
    O_parts [N, q_len, Hq, Dv], LSE_parts [N, q_len, Hq])."""
    q = np.asarray(q, dtype=np.float64)
    res = [sharded_attention(q[i], K, V, scale, starts_b, hi)
           for i, hi in enumerate(mtp_limits(seq_len, q.shape[0]))]
    O = np.stack([r[0] for r in res])
    lse = np.stack([r[1] for r in res])
    parts = np.stack([r[2] for r in res], axis=1)
    part_lses = np.stack([r[3] for r in res], axis=1)
    return O, lse, parts, part_lses


# ---------------------------------------------------------------------------
# 8-bit KV cache (e4m3 codes with one scale per tensor)
# ---------------------------------------------------------------------------
# P1 lists KV cache quantization among the techniques other serving stacks
# pair with context parallelism ("KV cache quantization, offloading ..."); it
# names no format. Reading taken: the cache holds FP8 E4M3 codes (the "fn"
# variant of the OCP 8-bit floating-point formats: no infinities, one NaN
# pattern per sign) and one float scale for all keys and one for all values
# of a layer; a cached key is k_scale * decode(code), a value
# v_scale * decode(code). Attention over the decoded cache is the plain
# definition above.
def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of FP8 E4M3 codes (uint8): sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits. Exponent field 0 holds the subnormals
    (m / 8) * 2**-6; exponent field 15 with mantissa 7 is NaN; there is no
    infinity, so exponent 15 with mantissa 0..6 is an ordinary normal
    (up to 1.75 * 2**8 = 448)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def fp8_kv(k_codes, v_codes, k_scale: float, v_scale: float):
    """Float64 keys and values of an 8-bit cache: scale * decode(code)."""
    return float(k_scale) * e4m3_to_f64(k_codes), float(v_scale) * e4m3_to_f64(v_codes)
