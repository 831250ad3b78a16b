"""Named workload presets (shapes, sizes and seeds only).

Each preset is one decode step of one attention layer: every sequence has
`ctx` tokens before the step, the step appends one token per sequence and
then attends over ctx + 1 tokens, split across `shards` virtual shards.
Values are the seeded draws of `inputs` (stand-ins for N(0,1) bf16 data).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import inputs

GQA = 0
MLA = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: int                 # GQA or MLA
    batch: int
    q_heads: int
    kv_heads: int
    dk: int
    dv: int
    block_size: int
    shards: int
    scale: float
    ctx_kind: str             # "fixed" or "lognormal"
    ctx_fixed: int = 0
    median: float = 67000.0
    sigma: float = 0.75
    ctx_lo: int = 4096
    ctx_hi: int = 262144
    capacity_factor: float = 1.0   # > 1: fragmented pools with holes
    seed: int = 0
    needles: int = 0               # planted q-aligned keys per sequence (structured parity cases)
    kv_dtype: str = "bf16"         # "bf16" or "fp8" (E4M3 codes of the bf16 draws, GQA only)
    k_scale: float = 1.0           # fp8: key = k_scale * decode(code)
    v_scale: float = 1.0           # fp8: value = v_scale * decode(code)

    def ctx_lens(self) -> np.ndarray:
        """Context length of every sequence before the decode step."""
        if self.ctx_kind == "fixed":
            return np.full(self.batch, self.ctx_fixed, dtype=np.int64)
        return inputs.lognormal_lengths(self.seed, self.batch, self.median, self.sigma,
                                        self.ctx_lo, self.ctx_hi)

    def needle_plan(self) -> dict:
        if self.needles <= 0:
            return {}
        return inputs.needle_plan(self.seed, self.ctx_lens() + 1, self.needles, self.q_heads)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def kv_bytes_per_token(self) -> int:
        """Bytes of KV cache read per attended token (2 per element, 1 for fp8)."""
        elem = 1 if self.kv_dtype == "fp8" else 2
        if self.kind == MLA:
            return elem * self.dk                   # one latent row; V aliases its prefix
        return elem * self.kv_heads * (self.dk + self.dv)


def _preset(**kw) -> Workload:
    return Workload(**kw)


PRESETS = {
    # batch 1, 8/2 heads, head_dim 64, 512 attended tokens over 4 shards of 128.
    "gqa_tiny": _preset(name="gqa_tiny", kind=GQA, batch=1, q_heads=8, kv_heads=2, dk=64, dv=64,
                        block_size=16, shards=4, scale=1.0 / math.sqrt(64), ctx_kind="fixed",
                        ctx_fixed=511),
    # batch 32, 64/4 heads, head_dim 128, 32768 attended tokens over 2 shards.
    "gqa_mid": _preset(name="gqa_mid", kind=GQA, batch=32, q_heads=64, kv_heads=4, dk=128, dv=128,
                       block_size=16, shards=2, scale=1.0 / math.sqrt(128), ctx_kind="fixed",
                       ctx_fixed=32767),
    # batch 64, 128 heads on one 576-wide latent (512-wide values), lognormal lengths, 8 shards.
    "mla_decode": _preset(name="mla_decode", kind=MLA, batch=64, q_heads=128, kv_heads=1, dk=576,
                          dv=512, block_size=64, shards=8, scale=1.0 / math.sqrt(576),
                          ctx_kind="lognormal"),
    # batch 8, 200,000 context tokens + 1 appended, 8 shards (16 in the variant below).
    "mla_long": _preset(name="mla_long", kind=MLA, batch=8, q_heads=128, kv_heads=1, dk=576,
                        dv=512, block_size=64, shards=8, scale=1.0 / math.sqrt(576),
                        ctx_kind="fixed", ctx_fixed=200000),
    "mla_long_16": _preset(name="mla_long_16", kind=MLA, batch=8, q_heads=128, kv_heads=1, dk=576,
                           dv=512, block_size=64, shards=16, scale=1.0 / math.sqrt(576),
                           ctx_kind="fixed", ctx_fixed=200000),
    # batch 512, lognormal lengths, 8 shards, fragmented pools (1.25x capacity).
    "mla_high_concurrency": _preset(name="mla_high_concurrency", kind=MLA, batch=512, q_heads=128,
                                    kv_heads=1, dk=576, dv=512, block_size=64, shards=8,
                                    scale=1.0 / math.sqrt(576), ctx_kind="lognormal",
                                    capacity_factor=1.25),
}


def get(name: str) -> Workload:
    try:
        return PRESETS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(PRESETS)}") from None
