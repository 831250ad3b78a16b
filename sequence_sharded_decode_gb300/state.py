"""Device state of one decode step for a workload preset.

Allocates the N shard pools, block tables, queries, the step's new tokens,
the reused workspace and the output buffers with torch, fills the pools
through dcp_kv_append, and runs one step through the C ABI:
append -> partial attention on every shard -> LSE merge.
"""
from __future__ import annotations

import numpy as np
import torch

from . import configs, dcp, inputs


class DecodeState:
    def __init__(self, wl: configs.Workload, device: str = "cuda", fill: bool = True,
                 canary: int | None = None, table_seed: int | None = None, fill_chunk: int = 1 << 18,
                 q_len: int = 1, gen_device: str | None = None):
        """q_len > 1: every sequence brings q_len new tokens per step (a
        speculative / multi-token step); query token j sits at position
        ctx[b] + j and the partial pass is dcp_decode_partial_all_mtp.
        gen_device: where the seeded draws are made before they are copied to
        `device` (default: on `device`; "cpu" for small cases keeps the
        device's launch list to the library's own kernels)."""
        self.wl = wl
        self.device = device
        self.gen = device if gen_device is None else gen_device
        self.q_len = q_len
        self.ctx = wl.ctx_lens().astype(np.int64)
        B, N = wl.batch, wl.shards
        self.f8 = wl.kv_dtype == "fp8"
        self.desc = dcp.AttnDesc(wl.kind, wl.q_heads, wl.kv_heads, wl.dk, wl.dv, wl.block_size, wl.scale,
                                 dcp.DCP_KV_FP8_E4M3 if self.f8 else dcp.DCP_KV_BF16, wl.k_scale, wl.v_scale)
        starts, blocks = dcp.dcp_shard_plan(self.ctx, N, wl.block_size, q_len)
        self.starts_host, self.blocks_host = starts, blocks
        seed_t = wl.seed + 1 if table_seed is None else table_seed
        self.tables_host = inputs.block_tables(seed_t, blocks, wl.capacity_factor)
        self.shards = []
        for cap, tab in self.tables_host:
            if wl.kind == configs.MLA:  # one latent row per token (E4M3 codes for the 8-bit cache)
                k = torch.empty((cap, wl.block_size, wl.dk), dtype=torch.uint8 if self.f8 else torch.bfloat16,
                                device=device)
                v = None
            elif self.f8:  # E4M3 codes; the values of a block stored transposed (dims x tokens)
                k = torch.empty((cap, wl.kv_heads, wl.block_size, wl.dk), dtype=torch.uint8, device=device)
                v = torch.empty((cap, wl.kv_heads, wl.dv, wl.block_size), dtype=torch.uint8, device=device)
            else:
                k = torch.empty((cap, wl.kv_heads, wl.block_size, wl.dk), dtype=torch.bfloat16, device=device)
                v = torch.empty((cap, wl.kv_heads, wl.block_size, wl.dv), dtype=torch.bfloat16, device=device)
            if canary is not None:
                if self.f8:
                    k.fill_(canary & 0xFF)
                    if v is not None:
                        v.fill_(canary & 0xFF)
                else:
                    k.view(torch.int16).fill_(canary)
                    if v is not None:
                        v.view(torch.int16).fill_(canary)
            self.shards.append(dcp.Shard(k, v, torch.from_numpy(tab).to(device)))
        self.starts = torch.from_numpy(starts).to(device)
        qstream = inputs.STREAM_Q_MLA if wl.kind == configs.MLA else inputs.STREAM_Q
        if q_len == 1:
            self.q = inputs.query(wl.seed, np.arange(B), wl.q_heads, wl.dk, self.gen, stream=qstream).to(device)
            self.q0 = self.q
        else:
            self.q = inputs.query_tokens(wl.seed, np.arange(B), q_len, wl.q_heads, wl.dk, self.gen,
                                         stream=qstream).to(device)
            self.q0 = self.q[:, 0].contiguous()  # planted needles copy query token 0
        self.needles = wl.needle_plan()
        new_b = np.repeat(np.arange(B), q_len)
        new_t = (self.ctx[:, None] + np.arange(q_len)[None, :]).reshape(-1)
        self.seq_ids = torch.from_numpy(new_b.astype(np.int32)).to(device) if q_len > 1 else None
        self.positions = torch.from_numpy(new_t.astype(np.int32)).to(device)
        self.seq_lens = torch.from_numpy((self.ctx + q_len).astype(np.int32)).to(device)
        self.k_new, self.v_new = self.token_rows(new_b, new_t)
        ws = dcp.dcp_workspace_size_mtp(self.desc, B, q_len, N)
        if ws <= 0:
            raise RuntimeError("dcp_workspace_size failed")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        rows = (B,) if q_len == 1 else (B, q_len)
        self.o_parts = torch.empty((N, *rows, wl.q_heads, wl.dv), dtype=torch.float32, device=device)
        self.lses = torch.empty((N, *rows, wl.q_heads), dtype=torch.float32, device=device)
        self.o = torch.empty((*rows, wl.q_heads, wl.dv), dtype=torch.float32, device=device)
        self.lse = torch.empty((*rows, wl.q_heads), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        if fill:
            self.fill_context(fill_chunk)

    # -- token rows from the seeded generator -------------------------------
    def token_rows(self, b, t):
        """K/V (or latent) rows of tokens (b[j], t[j]), drawn on the generation
        device and returned on the state's device."""
        wl = self.wl
        g = self.gen
        b = torch.as_tensor(b).to(g)
        t = torch.as_tensor(t).to(g)
        if wl.kind == configs.MLA:
            lat = inputs.kv_tokens(wl.seed, inputs.STREAM_LATENT, b, t, 1, wl.dk, g, chunk=1 << 18)
            lat = inputs.plant_needles(lat.view(-1, wl.dk), b, t, self.q0.to(g), self.needles, wl.q_heads)
            if self.f8:  # the cache holds the E4M3 codes of the same draws
                lat = inputs.e4m3_codes(lat)
            return lat.to(self.device), None
        k = inputs.kv_tokens(wl.seed, inputs.STREAM_K, b, t, wl.kv_heads, wl.dk, g, chunk=1 << 16)
        k = inputs.plant_needles(k, b, t, self.q0.to(g), self.needles, wl.q_heads)
        v = inputs.kv_tokens(wl.seed, inputs.STREAM_V, b, t, wl.kv_heads, wl.dv, g, chunk=1 << 16)
        if self.f8:  # the cache holds the E4M3 codes of the same draws
            k, v = inputs.e4m3_codes(k), inputs.e4m3_codes(v)
        return k.to(self.device), v.to(self.device)

    def fill_context(self, chunk: int = 1 << 18):
        """Write every context token [0, ctx[b]) of every sequence into the pools."""
        ctx = torch.from_numpy(self.ctx).to(self.gen)
        ends = torch.cumsum(ctx, 0)
        begins = ends - ctx
        total = int(ends[-1]) if ctx.numel() else 0
        for s in range(0, total, chunk):
            idx = torch.arange(s, min(total, s + chunk), dtype=torch.int64, device=self.gen)
            b = torch.searchsorted(ends, idx, right=True)
            t = idx - begins[b]
            k, v = self.token_rows(b, t)
            dcp.dcp_kv_append(self.desc, self.shards, self.starts, t.to(torch.int32).to(self.device), k, v,
                              seq_ids=b.to(torch.int32).to(self.device), err=self.err)

    # -- the decode step through the C ABI ------------------------------------
    def append(self, stream=None):
        dcp.dcp_kv_append(self.desc, self.shards, self.starts, self.positions, self.k_new, self.v_new,
                          seq_ids=self.seq_ids, err=self.err, stream=stream)

    def partial(self, stream=None):
        if self.q_len == 1:
            dcp.dcp_decode_partial_all(self.desc, self.q, self.shards, self.seq_lens, self.starts, self.o_parts,
                                       self.lses, self.workspace, err=self.err, stream=stream)
        else:
            dcp.dcp_decode_partial_all_mtp(self.desc, self.q, self.shards, self.seq_lens, self.starts,
                                           self.o_parts, self.lses, self.workspace, err=self.err, stream=stream)

    def attention(self, stream=None):
        """Partial attention of every shard and the merge in one call."""
        dcp.dcp_attention_all(self.desc, self.q, self.shards, self.seq_lens, self.starts, self.o_parts, self.lses,
                              self.o, self.lse, self.workspace, err=self.err, stream=stream)

    def merge(self, stream=None):
        dcp.dcp_merge(self.o_parts, self.lses, self.o, self.lse, stream=stream)

    def step(self, stream=None, fused: bool = False):
        """append -> partial attention of every shard -> merge; fused: the last
        two in one call (dcp_attention_all; the shards' partial rows of split
        ranges -- for MLA, all of them -- are then not written), else
        dcp_decode_partial_all(_mtp) then dcp_merge."""
        self.append(stream)
        if fused:
            self.attention(stream)
        else:
            self.partial(stream)
            self.merge(stream)

    # -- algorithmic bytes ---------------------------------------------------
    def attended_tokens(self) -> int:
        """Distinct tokens the step attends: the context plus the new tokens
        (with several query tokens, each token is still read from HBM once)."""
        return int((self.ctx + self.q_len).sum())

    def attention_flops(self) -> int:
        """Multiply-add flops of the partial pass: for every query token, q.k
        and p.v over each token it attends (2 (Dk + Dv) per head and token)."""
        wl = self.wl
        per_seq = self.q_len * (self.ctx + 1) + self.q_len * (self.q_len - 1) // 2  # sum_j (ctx + j + 1)
        return int(2 * wl.q_heads * (wl.dk + wl.dv) * per_seq.sum())

    def kv_bytes(self) -> int:
        """KV bytes the partial-attention pass must read (each attended token once)."""
        return self.attended_tokens() * self.wl.kv_bytes_per_token

    def step_bytes(self, fused: bool = False) -> dict:
        """Algorithmic HBM bytes of one step, by call. Two calls (and GQA's
        one call): the shards' partial rows are written and read back. MLA's
        one call merges the shards on chip: KV, queries and the merged rows
        only (the pieces of the few row groups a CTA boundary cuts are left
        out: at most two per CTA pair)."""
        wl = self.wl
        B, N, Hq, dv, dk = wl.batch * self.q_len, wl.shards, wl.q_heads, wl.dv, wl.dk
        part = N * B * Hq * (dv + 1) * 4
        out = B * Hq * (dv + 1) * 4
        new_tok = B * (wl.kv_bytes_per_token if wl.kind == configs.GQA else dk * 2)
        if fused and wl.kind == configs.MLA:
            return {
                "append": 2 * new_tok,                  # read the new rows, write them
                "attention": self.kv_bytes() + B * Hq * dk * 2 + out,
            }
        return {
            "append": 2 * new_tok,
            "partial": self.kv_bytes() + B * Hq * dk * 2 + part,
            "merge": part + out,
        }
