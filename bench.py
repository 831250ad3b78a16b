#!/usr/bin/env python3
"""Benchmark of one DCP decode step (append -> partial attention on every
virtual shard -> LSE merge) through the C ABI, on synthetic seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--q-len Q] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is whole-job achieved HBM GB/s: the
step's algorithmic bytes (KV read once, queries, partials written and read,
output, appended rows) over the device-timed step, summed over ranks and
divided by the slowest rank's time. `--q-len Q` (Q > 1) runs a multi-token
step instead: Q new tokens per sequence, query token j at position ctx + j,
causal among the new tokens; each KV token still counts once. With N > 1 each rank runs an independent
replica of the workload (weak scaling; the shards of one step live in one
GPU's memory, so nothing crosses GPUs). `--impl reference` times the float64
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DCP decode attn: achieved HBM GB/s (% of GB300 peak); decode tokens/s per layer"
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _tensor_peak() -> float:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return 1700.0


def _workload_config(wl, st=None, q_len: int = 1) -> dict:
    name = wl.name + (", fp8 KV cache" if wl.kv_dtype == "fp8" else "")
    cfg = {"workload": name if q_len == 1 else f"{name}, {q_len} query tokens per sequence", "batch": wl.batch, "q_heads": wl.q_heads, "kv_heads": wl.kv_heads,
           "head_dim_k": wl.dk, "head_dim_v": wl.dv, "block_size": wl.block_size, "shards": wl.shards,
           "context": (f"{wl.ctx_fixed}+{q_len}" if wl.ctx_kind == "fixed"
                       else f"lognormal(median {wl.median:g}, sigma {wl.sigma}) in [{wl.ctx_lo},{wl.ctx_hi}] +{q_len}"),
           "fragmented_pools": wl.capacity_factor > 1.0,
           "kv_cache": ("fp8 e4m3 codes, k_scale %g, v_scale %g" % (wl.k_scale, wl.v_scale)
                        if wl.kv_dtype == "fp8" else "bf16"),
           "l2": "inputs larger than L2 (KV read per step >> 129 MB); no flush"}
    if st is not None:
        cfg["attended_tokens"] = st.attended_tokens()
        cfg["kv_bytes_per_step"] = st.kv_bytes()
    return cfg


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def _traffic_for(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[workload]
        src = os.path.join(ROOT, "sequence_sharded_decode_gb300", "csrc", kernel_file)
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if ent.get("source_sha256_16") != h:
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# the CPU oracle leg (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def oracle_prepare(wl, seqs, q_len: int = 1):
    """Generate (outside any timing) the bf16 inputs of the sampled sequences."""
    import oracle as O
    from sequence_sharded_decode_gb300 import configs, inputs

    ctx = wl.ctx_lens()
    starts = O.shard_starts(ctx, wl.shards)
    data = []
    for b in seqs:
        L = int(ctx[b]) + q_len
        qs = inputs.STREAM_Q_MLA if wl.kind == configs.MLA else inputs.STREAM_Q
        if q_len == 1:
            q = inputs.bf16_bits(inputs.query(wl.seed, [b], wl.q_heads, wl.dk, stream=qs))[0]
        else:
            q = inputs.bf16_bits(inputs.query_tokens(wl.seed, [b], q_len, wl.q_heads, wl.dk, stream=qs))[0]
        if wl.kind == configs.MLA and wl.kv_dtype == "fp8":  # one row of E4M3 codes per token
            kb = inputs.e4m3_codes(inputs.sequence_kv(wl.seed, inputs.STREAM_LATENT, b, 0, L, 1, wl.dk)).numpy()
            vb = kb[:, :, :wl.dv]
        elif wl.kind == configs.MLA:
            kb = inputs.bf16_bits(inputs.sequence_kv(wl.seed, inputs.STREAM_LATENT, b, 0, L, 1, wl.dk))
            vb = None
        elif wl.kv_dtype == "fp8":  # E4M3 codes (uint8) of the same draws
            kb = inputs.e4m3_codes(inputs.sequence_kv(wl.seed, inputs.STREAM_K, b, 0, L, wl.kv_heads, wl.dk)).numpy()
            vb = inputs.e4m3_codes(inputs.sequence_kv(wl.seed, inputs.STREAM_V, b, 0, L, wl.kv_heads, wl.dv)).numpy()
        else:
            kb = inputs.bf16_bits(inputs.sequence_kv(wl.seed, inputs.STREAM_K, b, 0, L, wl.kv_heads, wl.dk))
            vb = inputs.bf16_bits(inputs.sequence_kv(wl.seed, inputs.STREAM_V, b, 0, L, wl.kv_heads, wl.dv))
        data.append((b, L, q, kb, vb, starts[b]))
    return data


def oracle_pass(wl, data):
    """One timed oracle pass (bf16 widening + per-shard partials + merge) over
    the prepared sequences; returns (seconds, KV bytes covered)."""
    import oracle as O

    t0 = time.perf_counter()
    nbytes = 0
    for b, L, q, kb, vb, starts_b in data:
        qf = O.bf16_bits_to_f64(q)
        if kb.dtype == np.uint8:
            K, V = O.fp8_kv(kb, vb, wl.k_scale, wl.v_scale)
        else:
            K = O.bf16_bits_to_f64(kb)
            V = K[:, :, :wl.dv] if vb is None else O.bf16_bits_to_f64(vb)
        if qf.ndim == 2:
            O.sharded_attention(qf, K, V, wl.scale, starts_b, L)
        else:
            O.sharded_mtp_attention(qf, K, V, wl.scale, starts_b, L)
        nbytes += L * wl.kv_bytes_per_token
    return time.perf_counter() - t0, nbytes


def _cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_sample(wl, seqs, budget_s: float, q_len: int = 1):
    """Oracle throughput over a bounded sample: repeat passes until budget_s."""
    data = oracle_prepare(wl, seqs, q_len)
    t_total, nbytes, runs = 0.0, 0, 0
    while runs == 0 or t_total < budget_s:
        t, n = oracle_pass(wl, data)
        t_total += t
        nbytes += n
        runs += 1
    desc = (f"sequence(s) {list(seqs)} of {wl.name} over their full contexts; {runs} oracle pass(es) of "
            f"float64 per-shard partials + merge; input generation excluded")
    return nbytes / t_total / 1e9, t_total, desc, _cores()


_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def oracle_leg(args, threads: int):
    """The oracle sample in a fresh interpreter whose BLAS pool is pinned to
    `threads` threads (the thread count must be fixed before numpy loads).
    Returns the leg's JSON dict, or None if it failed."""
    env = dict(os.environ)
    for v in _THREAD_VARS:
        env[v] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-leg", "--workload", args.workload,
           "--cpu-seconds", str(args.cpu_seconds), "--q-len", str(args.q_len), "--kv-dtype", args.kv_dtype]
    if args.batch is not None:
        cmd += ["--batch", str(args.batch)]
    if args.shards is not None:
        cmd += ["--shards", str(args.shards)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        for line in reversed(r.stdout.strip().splitlines()):
            if line.startswith("{"):
                d = json.loads(line)
                d["cores"] = threads
                return d
    except Exception:
        pass
    return None


def run_oracle_leg(args, wl):
    """Child side of oracle_leg: print the sample's throughput as one JSON line."""
    seqs = [0, min(1, wl.batch - 1)] if wl.batch > 1 else [0]
    gbs, secs, desc, _ = oracle_sample(wl, seqs, args.cpu_seconds, args.q_len)
    print(json.dumps({"value": round(gbs, 4), "unit": "GB/s", "kind": "oracle", "sample": desc,
                      "seconds": round(secs, 2)}), flush=True)
    return 0


def run_reference(args, wl):
    """Reference arm: the float64 CPU oracle, K timed passes over one sampled
    sequence of the workload after W untimed ones (rank 0 only)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    seqs = [0]
    data = oracle_prepare(wl, seqs, args.q_len)
    times, nbytes = [], 0
    for i in range(args.warmup + args.steps):
        t, n = oracle_pass(wl, data)
        if i >= args.warmup:
            times.append(t)
            nbytes = n
    value = nbytes / float(np.mean(times)) / 1e9
    desc = (f"sequence 0 of {wl.name} over its full context per step; float64 per-shard partials + merge; "
            f"input generation excluded")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * float(np.mean(times)), 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": _workload_config(wl, q_len=args.q_len),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": _cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# cross-rank aggregation (host side; replicas share no data)
# ---------------------------------------------------------------------------
def max_over_ranks(vals, device="cpu"):
    """Element-wise max of per-rank timings (all ranks get the result)."""
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_gbs(world: int, bytes_per_step_per_rank: int, ms_slowest: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return world * bytes_per_step_per_rank / (ms_slowest * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------
def run_ours(args, wl):
    import torch

    from sequence_sharded_decode_gb300 import dcp
    from sequence_sharded_decode_gb300.state import DecodeState

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dcp.load()
    st = DecodeState(wl, device=f"cuda:{local}", q_len=args.q_len)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    fused = not args.two_calls
    bytes_ = st.step_bytes(fused)
    step_bytes = sum(bytes_.values())
    # the dominant kernel's call, timed alone for the roofline: MLA's one call
    # (plan + attention with the shards merged on chip) where the step uses it,
    # else the partial call (plan + attention + combine of split ranges)
    one_call_mla = fused and wl.kind == 1
    call_bytes = bytes_["attention"] if one_call_mla else st.step_bytes(False)["partial"]
    call_name = ("dcp_attention_all (plan + attention, shards merged in the kernel), timed alone" if one_call_mla
                 else "dcp_decode_partial_all (plan + attention + combine), timed alone")
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            st.step(stream, fused)
    barrier()
    K = args.steps
    ev_p0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_p1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(K):
                st.step(stream, fused)
            end.record(stream)
            # the dominant kernel's call alone, on the same stream
            for i in range(K):
                ev_p0[i].record(stream)
                if one_call_mla:
                    st.attention(stream)
                else:
                    st.partial(stream)
                ev_p1[i].record(stream)
        stream.synchronize()
    barrier()
    clocks = clk.summary()
    ms = start.elapsed_time(end) / K
    partial_ms = sum(a.elapsed_time(b) for a, b in zip(ev_p0, ev_p1)) / K
    err = int(st.err.item())
    if err:
        raise RuntimeError(f"device error flag set: {err}")

    # End to end through the public API: every step copies its inputs in from
    # pinned host memory and its result (O, LSE) back out, as a serving loop
    # does. Copies run on their own stream, double-buffered on the device, so
    # step i+1's inputs come in and step i's result goes out while the GPU
    # computes: the timed region spans the first input copy to the last
    # result copy.
    names_in = [n for n in ("q", "k_new", "v_new", "seq_ids", "positions", "seq_lens") if getattr(st, n) is not None]
    host_in = {n: getattr(st, n).cpu().pin_memory() for n in names_in}
    host_out = {n: torch.empty(getattr(st, n).shape, dtype=getattr(st, n).dtype).pin_memory() for n in ("o", "lse")}
    dev = [{n: torch.empty_like(getattr(st, n)) for n in names_in + ["o", "lse"]} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    copy_stream = torch.cuda.Stream()  # host -> device
    out_stream = torch.cuda.Stream()   # device -> host

    def e2e_run(n_steps):
        in_free = [None, None]    # compute done reading input set b
        out_free = [None, None]   # result of set b copied out
        last = None
        for i in range(n_steps):
            b = i & 1
            d = dev[b]
            with torch.cuda.stream(copy_stream):
                if in_free[b] is not None:
                    copy_stream.wait_event(in_free[b])
                for n in names_in:
                    d[n].copy_(host_in[n], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(copy_stream)
            stream.wait_event(ready)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            for n in names_in + ["o", "lse"]:
                setattr(st, n, d[n])
            st.step(stream, fused)
            done = torch.cuda.Event()
            done.record(stream)
            in_free[b] = done
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(done)
                for n in ("o", "lse"):
                    host_out[n].copy_(d[n], non_blocking=True)
                out = torch.cuda.Event()
                out.record(out_stream)
            out_free[b] = out
            last = out
        return last

    e2e_run(max(3, args.warmup))
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(copy_stream)
    stream.wait_event(e0)
    last = e2e_run(K)
    out_stream.wait_event(last)
    e1.record(out_stream)
    out_stream.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / K
    err = int(st.err.item())
    if err:
        raise RuntimeError(f"device error flag set in the end-to-end run: {err}")

    ms, partial_ms, e2e_ms = max_over_ranks([ms, partial_ms, e2e_ms], device=f"cuda:{local}")

    if rank == 0:
        peak, peak_kind = _peaks()
        value = whole_job_gbs(world, step_bytes, ms)
        achieved = call_bytes / (partial_ms * 1e-3) / 1e9
        kern = "dcp_mla.cu" if wl.kind == 1 else "dcp_gqa.cu"
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp8 e4m3 KV (fp16 MMA, fp32 accumulate)" if wl.kv_dtype == "fp8" else "bf16",
            "data": "synthetic",
            "config": _workload_config(wl, st, args.q_len) | {"parallelism": f"replicas x{world}"},
            "hbm_frac_of_peak": round(value / world / peak, 4),
            "tokens_per_s_per_layer": round(world * wl.batch * args.q_len / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "kernel": call_name,
                         "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": (_traffic_for(kern, wl.name + ("_fp8" if wl.kv_dtype == "fp8" else ""))
                                     if args.q_len == 1 else None),
                         "algorithmic_bytes_per_launch": call_bytes},
            "step_bytes": bytes_,
            "step_calls": ("dcp_kv_append, dcp_attention_all (partial attention, shards merged in the kernel)"
                           if one_call_mla else
                           "dcp_kv_append, dcp_attention_all (partial attention + one-pass merge)" if fused
                           else "dcp_kv_append, dcp_decode_partial_all, dcp_merge"),
            "e2e": {"value": round(whole_job_gbs(world, step_bytes, e2e_ms), 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            # per step: append, plan, attention and, one call: the finishing
            # kernel (MLA) or the one-pass merge (GQA); two calls: combine and merge
            "gpu_launches": (4 if (one_call_mla or fused) else 5) * K,
            "clocks": clocks,
        }
        if args.q_len > 1:
            # with many query tokens per step the pass is a dense contraction:
            # its tensor roofline against the measured bf16 peak
            flops = st.attention_flops()
            tf_peak = _tensor_peak()
            line["tensor_roofline"] = {"bound": "tensor", "achieved": round(flops / (partial_ms * 1e-3) / 1e12, 2),
                                       "peak": tf_peak, "unit": "TFLOP/s",
                                       "frac": round(flops / (partial_ms * 1e-3) / 1e12 / tf_peak, 4),
                                       "flops_per_launch": flops,
                                       "note": "mma.sync / tcgen05 kernels of the decode path; peak = measured "
                                               "cuBLAS bf16, sustained"}
        if world == 1 and not args.no_cpu_baseline:
            # the oracle on every host core (its BLAS pool pinned to the
            # affinity count), and once on a single thread
            allc = oracle_leg(args, _cores())
            one = oracle_leg(args, 1)
            if allc is not None:
                line["cpu_baseline"] = allc
                if one is not None:
                    line["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "seconds")}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mla_high_concurrency")
    ap.add_argument("--oracle-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override the preset's batch (profiling cases)")
    ap.add_argument("--shards", type=int, default=None, help="override the preset's shard count")
    ap.add_argument("--two-calls", action="store_true",
                    help="partial attention and merge as two calls (default: one dcp_attention_all call)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="KV cache element type (fp8: E4M3 codes with per-tensor scales)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence per step (speculative step, or a prefill chunk)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not 1 <= args.q_len <= 8192:
        ap.error("--q-len must be in [1, 8192]")
    from sequence_sharded_decode_gb300 import configs
    wl = configs.get(args.workload)
    if args.batch is not None:
        wl = wl.with_(batch=args.batch)
    if args.shards is not None:
        wl = wl.with_(shards=args.shards)
    if args.kv_dtype == "fp8":
        wl = wl.with_(kv_dtype="fp8")
    if args.oracle_leg:
        return run_oracle_leg(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
