"""Benchmark: quantized-KV decode attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: encode/append of the
new token(s) of every sequence, then decode attention (split-K kernel +
combine / inverse-rotation kernel) over the grown cache.  The default workload
is the batched turbo4 decode at Llama-3-8B attention shape (B=32, Hq=32,
Hkv=8, ragged contexts U[16384, 32768], 1 appended token per sequence), whose
per-step inputs (about 0.83 GB) are larger than L2, so no flush is needed
between steps.

Printed: one JSON line (rank 0) with value = effective GB/s over the
algorithmic bytes of the step (packed K/V + norms over every visible token,
q, o, and the append's fp16 inputs and packed outputs), tokens/s, the decode
kernel's roofline (its own duration from 12 launches timed with the library's
event pair right after the timed steps), the oracle's CPU baseline, an
end-to-end figure through the C ABI with host buffers, clocks sampled during
the timed region, and the number of kernel launches; besides, the step
captured once into a CUDA graph and replayed 50 times, each replay timed on
its own (median, p10, p90 under `graph`).  The default run (one
GPU, workload 4) also times workloads 2, 3 and 5 (with the 4096-token
prefill-chunk encode of workload 5) the same way and reports each under
`other_workloads`.

--impl reference times the fp64 CPU oracle (the correctness reference of this
library; nothing else implements the pages' method here) on a bounded sample
of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quantized_kv_cache_flash_gb300 import workloads as wl  # noqa: E402

METRIC = "quantized-KV decode attention: effective HBM GB/s (% of peak), tokens/s"
PROMPT_METRIC = "chunked-prefill attention over the packed cache: TFLOP/s (causal FLOPs), tokens/s"
# bytes per token per kv head (K, V): packed record + fp16 norm, or fp16 K, or
# a table record (codes + centroid x norm table, no norm)
REC = {"turbo4_asym": (256, 66), "turbo3": (50, 50), "turbo4": (66, 66),
       "turbo3_asym": (256, 50), "turbo4k_3v": (66, 50), "turbo3_table": (64, 64)}
L2_BYTES = 129 * 1024 * 1024
KERNEL_STEPS = 12   # decode launches timed on their own, after the timed steps
GRAPH_REPLAYS = 50  # replays of the step's CUDA graph, each timed on its own (median, p10, p90)
PREFILL_REPS = 5    # prefill-chunk appends per timed run (distinct inputs, together above 2 x L2)
PIPELINE_MIN_MS = 0.1   # e2e: device step time above which the host copies overlap compute


def prompt_flops(w: wl.Workload) -> float:
    """Algorithmic FLOPs of the causal attention of a Tq-token prompt into an
    empty cache: query j sees j + 1 tokens; QK^T and PV are 2 * 128 FLOPs per
    (row, visible token) each."""
    vis = w.tq * (w.tq + 1) / 2
    return 4.0 * 128 * w.batch * w.num_q_heads * vis


def load_tensor_peak():
    """Dense fp16 tensor peak: the measured bf16 cuBLAS figure (burst) --
    fp16 and bf16 share the same nominal dense rate on this part."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured bf16_tflops (cuBLAS, burst) x 1.0 fp16/bf16"
    except Exception:
        return 1900.0, "fallback"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def decode_bytes(w: wl.Workload, lens: np.ndarray) -> int:
    """Algorithmic bytes of one decode: packed K/V + norms of every visible
    token of every KV head, plus q read and o written (fp16)."""
    rk, rv = REC[w.mode]
    kv = int(np.sum(lens.astype(np.int64))) * w.num_kv_heads * (rk + rv)
    qo = 2 * w.batch * w.num_q_heads * w.tq * 128 * 2
    return kv + qo


def decode_kernel_bytes(w: wl.Workload, lens: np.ndarray) -> int:
    """Algorithmic bytes of the split-K kernel alone: packed K/V + norms and q."""
    rk, rv = REC[w.mode]
    return (int(np.sum(lens.astype(np.int64))) * w.num_kv_heads * (rk + rv)
            + w.batch * w.num_q_heads * w.tq * 128 * 2)


def append_bytes(w: wl.Workload, t_new: int) -> int:
    """fp16 K and V read, packed records + norms written."""
    rk, rv = REC[w.mode]
    n = w.batch * w.num_kv_heads * t_new
    return n * (2 * 128 * 2) + n * (rk + rv)


def nominal_step_bytes(w: wl.Workload) -> float:
    """The bytes one step of the workload reads and writes, as the GPU arms
    count them for the config's L2 note: the prompt's fp16 q, K and V for a
    prompt workload, else the first timed step's decode and append bytes."""
    if w.prompt:
        return float(w.batch * w.tq * 128 * 2 * (w.num_q_heads + 2 * w.num_kv_heads))
    lens0 = wl.lengths(w).astype(np.int64)[:w.batch]
    return float(decode_bytes(w, lens0) + append_bytes(w, max(w.append, 0)))


def config_dict(w: wl.Workload):
    """The workload's config, the same for both arms.  The L2 note follows the
    decode arm's rule: steps under 2 x L2 flush L2 between steps (the prompt
    arm always does)."""
    ctx = (f"U[{w.context_min},{w.context}]" if w.ragged else str(w.context))
    step_bytes = nominal_step_bytes(w)
    return {"workload": w.name, "mode": w.mode, "batch": w.batch, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": 128, "context": ctx, "tq": w.tq,
            "append_per_step": max(w.append, 0), "rot_seed": w.rot_seed,
            "l2": ("inputs larger than L2 (%.0f MB per step > 2 x 129 MB), no flush" % (step_bytes / 1e6)
                   if step_bytes >= 2 * L2_BYTES and not w.prompt
                   else "L2 flushed between steps (%.0f MB per step)" % (step_bytes / 1e6))}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle sample (run in a child process with one BLAS thread)
# ---------------------------------------------------------------------------
def oracle_prompt_sample(w: wl.Workload, budget_s: float, seed: int = 0):
    """The oracle on prompt prefixes of one kv head at a time until budget_s is
    spent: encode a 256-token prefix of K and V, then the causal attention of
    all its G * 256 query rows.  Returns (FLOPs, seconds, units, description)."""
    from oracle import tq_oracle as o
    kb, vb = o.MODES[w.mode]
    cbk, cbv = (o.codebook(kb) if kb else None), o.codebook(vb)
    s = o.sign_vector(w.rot_seed)
    G, T = w.group, 256
    flops, units, t_spent, u = 0.0, 0, 0.0, 0
    while t_spent < budget_s:
        h = (u * 3 + seed) % w.num_kv_heads
        u += 1
        kx = wl.keys(w, 0, h, 0, T)
        vx = wl.values(w, 0, h, 0, T)
        q = wl.random_fp16(95000 + h + seed, (G, T, 128))
        t0 = time.perf_counter()
        vi, vn, _, _ = o.encode(vx, cbv, s)
        unit = {"v_idx": vi, "v_norm": vn}
        if kb is None:
            unit["k"] = kx
        else:
            unit["k_idx"], unit["k_norm"], _, _ = o.encode(kx, cbk, s)
        o.decode_unit(w.mode, q, unit, T, T, G, cbk, cbv, s, 1 / math.sqrt(128), 1.0)
        t_spent += time.perf_counter() - t0
        flops += 4.0 * 128 * G * T * (T + 1) / 2
        units += 1
    desc = (f"{units} kv heads, each: encode of a {T}-token prompt prefix (K and V) + causal "
            f"attention of its {G * T} query rows, fp64 NumPy, 1 BLAS thread")
    return flops, t_spent, units, desc


def oracle_sample(wnum: int, budget_s: float, seed: int = 0, mode=None):
    """Run the oracle on (b, kv-head) units of the workload until budget_s is
    spent: append of the step's new token (encode) + decode over the unit's
    visible context, on a packed cache of random records.  Returns
    (bytes, seconds, units, description); for a prompt workload FLOPs in place
    of bytes."""
    import dataclasses
    from oracle import tq_oracle as o
    w = wl.by_number(wnum)
    if mode:
        w = dataclasses.replace(w, mode=mode)
    if w.prompt:
        return oracle_prompt_sample(w, budget_s, seed)
    lens = wl.lengths(w)
    kb, vb = o.MODES[w.mode]
    table = w.mode in o.TABLE_MODES
    cbk = o.codebook(kb) if kb else None
    cbv = o.codebook(vb)
    s = o.sign_vector(w.rot_seed)
    G = w.group
    rk, rv = REC[w.mode]
    total_b, units, t_spent = 0, 0, 0.0
    u = 0
    while t_spent < budget_s:
        b, h = (u * 7 + seed) % w.batch, (u * 3 + seed) % w.num_kv_heads
        u += 1
        L = int(lens[b])
        key = 90000 + 131 * b + h
        rows = L
        if kb is None:
            kdat = wl.random_fp16(key, (rows, 128))
        else:
            kdat = wl.random_codes(key, rows, 16 * kb)
            knorm = wl.random_norms(key, rows)
        vdat = wl.random_codes(key + 1, rows, 16 * vb)
        vnorm = wl.random_norms(key + 1, rows)
        q = wl.random_fp16(key + 2, (G, w.tq, 128))
        knew = wl.random_fp16(key + 3, (max(w.append, 1), 128))
        t0 = time.perf_counter()
        # append (encode the new token's K and V)
        if kb is not None:
            o.encode(knew, cbk, s)
        o.encode(knew, cbv, s)
        unit = {"v_idx": o.unpack_codes(vdat, vb), "v_norm": vnorm}
        if table:
            o.centroid_norm_table(o.encode(knew, cbv, s)[1], cbv)  # the records' tables
            unit = {"k_idx": o.unpack_codes(kdat, kb), "k_table": o.centroid_norm_table(knorm, cbk),
                    "v_idx": unit["v_idx"], "v_table": o.centroid_norm_table(vnorm, cbv)}
        elif kb is None:
            unit["k"] = kdat
        else:
            unit["k_idx"] = o.unpack_codes(kdat, kb)
            unit["k_norm"] = knorm
        o.decode_unit(w.mode, q, unit, L, w.tq, G, cbk, cbv, s, 1 / math.sqrt(128), 1.0)
        t_spent += time.perf_counter() - t0
        total_b += L * (rk + rv) + 2 * G * w.tq * 128 * 2 + max(w.append, 1) * (512 + rk + rv)
        units += 1
    desc = (f"{units} (batch, kv-head) units of the workload, each: encode of the appended "
            f"token + decode of its {G * w.tq} query rows over the full visible context "
            f"(random packed records), fp64 NumPy, 1 BLAS thread")
    return total_b, t_spent, units, desc


def _oracle_worker(job):
    """One process of the oracle pool: (workload, budget, seed, mode) -> oracle_sample."""
    wnum, budget, seed, mode = job
    return oracle_sample(wnum, budget, seed=seed, mode=mode)


class OraclePool:
    """The oracle on every host core: one single-threaded process per core,
    started with spawn (never forked: the parent may hold a CUDA context), each
    taking its own (batch, kv head) units of the workload for the same budget;
    throughput = the bytes (FLOPs) of all of them / the longest one's time."""

    def __init__(self, nproc=None):
        import multiprocessing as mp
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"   # inherited by the workers
        self.n = nproc or os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.n)

    def sample(self, wnum, budget_s, seed0, mode=None):
        jobs = [(wnum, budget_s, seed0 + 7919 * i, mode) for i in range(self.n)]
        res = self.pool.map(_oracle_worker, jobs)
        self.last_rates = [r[0] / r[1] for r in res if r[1] > 0]   # each single-threaded process
        return (sum(r[0] for r in res), max(r[1] for r in res), sum(r[2] for r in res), res[0][3])

    def close(self):
        self.pool.close()
        self.pool.join()


def run_cpu_baseline(wnum: int, budget_s: float, mode=None):
    pool = OraclePool()
    try:
        b, s, u, desc = pool.sample(wnum, budget_s, 0, mode)
    finally:
        pool.close()
    prompt = wl.by_number(wnum).prompt
    scale = 1e12 if prompt else 1e9
    return {"value": b / s / scale, "unit": "TFLOP/s" if prompt else "GB/s",
            "cores": pool.n, "kind": "oracle",
            "sample": f"{pool.n} single-threaded processes x ({desc}); {u} units in all",
            "seconds": round(s, 2),
            # one core alone (the median single-threaded process)
            "per_core_value": statistics.median(pool.last_rates) / scale if pool.last_rates else None}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def prompt_arm(args, rank, world, device_index):
    """One step = append a Tq-token prompt to an empty cache (encode) and run
    the causal attention of its Tq queries over it (tcgen05 prefill kernel)."""
    import torch
    import quantized_kv_cache_flash_gb300 as tqf
    from quantized_kv_cache_flash_gb300 import build as tqbuild

    tqbuild.build()
    dev = torch.device("cuda", device_index)
    torch.cuda.set_device(dev)
    w = workload(args)
    B, Hq, Hkv, T = w.batch, w.num_q_heads, w.num_kv_heads, w.tq
    cap = int(math.ceil(T / 16) * 16)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + rank)
    ch = torch.tensor(wl.outlier_channels(w), device=dev, dtype=torch.long)

    def randn(shape, outl=False):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        if outl and ch.numel():
            x[..., ch] *= 8.0
        return x.to(torch.float16)

    ctx = tqf.Context()
    cache = tqf.Cache(tqf.MODES[w.mode], B, Hkv, cap, dev, rot_seed=w.rot_seed)
    k, v, q = randn((B, Hkv, T, 128), True), randn((B, Hkv, T, 128)), randn((B, Hq, T, 128))
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step():
        tqf.tq_encode_append(ctx, cache, k, v, stream)
        tqf.tq_prefill_attention(ctx, cache, q, out, T, 0.0, stream)

    steps, warm = args.steps, args.warmup
    for _ in range(warm):
        cache.lengths.zero_()
        step()
    torch.cuda.synchronize()
    if tqf.tq_get_status(ctx) != 0:
        raise RuntimeError("device status after the warm-up")
    barrier(world)
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    clocks = ClockSampler(device_index)
    clocks.start()
    tqf.tq_set_kernel_timing(ctx, True)
    tqf.tq_get_kernel_time(ctx)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    evs = []
    for i in range(steps):
        cache.lengths.zero_()
        scratch.fill_(float(i))          # L2 flush between steps, outside the timed intervals
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs)
    kern_ms, kern_n = tqf.tq_get_kernel_time(ctx)
    tqf.tq_set_kernel_timing(ctx, False)
    if tqf.tq_get_status(ctx) != 0:
        raise RuntimeError("device status after the timed steps")
    ms_max = reduce_max(world, ms)
    flops = prompt_flops(w)
    value = flops * steps * world / (ms_max * 1e-3) / 1e12
    peak, peak_kind = load_tensor_peak()
    achieved = flops / (kern_ms / kern_n * 1e-3) / 1e12 if kern_n else None

    # end to end with host buffers: prompt K/V and q in, the output back
    # Every step uploads its prompt's fp16 K, V and q from pinned host memory
    # and reads the output back, on a second stream, double-buffered: step
    # i+1's upload runs while step i computes, step i's read-back while step
    # i+1 computes.
    kh, vh, qh = k.cpu().pin_memory(), v.cpu().pin_memory(), q.cpu().pin_memory()
    kd = [torch.empty_like(k) for _ in range(2)]
    vd = [torch.empty_like(v) for _ in range(2)]
    qd = [torch.empty_like(q) for _ in range(2)]
    od = [torch.empty_like(out) for _ in range(2)]
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    copy_stream = torch.cuda.Stream(device=dev)
    h2d_ev = [torch.cuda.Event() for _ in range(2)]
    comp_ev = [torch.cuda.Event() for _ in range(2)]
    d2h_ev = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()

    def upload(sl):
        copy_stream.wait_event(comp_ev[sl])      # the step that last read buffer sl is done
        with torch.cuda.stream(copy_stream):
            kd[sl].copy_(kh, non_blocking=True)
            vd[sl].copy_(vh, non_blocking=True)
            qd[sl].copy_(qh, non_blocking=True)
        h2d_ev[sl].record(copy_stream)

    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    copy_stream.wait_event(f0)
    upload(0)
    for i in range(steps):
        sl = i % 2
        if i + 1 < steps:
            upload((i + 1) % 2)
        stream.wait_event(h2d_ev[sl])
        stream.wait_event(d2h_ev[sl])              # od[sl] has been read back
        cache.lengths.zero_()
        tqf.tq_encode_append(ctx, cache, kd[sl], vd[sl], stream)
        tqf.tq_prefill_attention(ctx, cache, qd[sl], od[sl], T, 0.0, stream)
        comp_ev[sl].record(stream)
        copy_stream.wait_event(comp_ev[sl])
        with torch.cuda.stream(copy_stream):
            oh.copy_(od[sl], non_blocking=True)
        d2h_ev[sl].record(copy_stream)
    done = torch.cuda.Event()
    done.record(copy_stream)
    stream.wait_event(done)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(world, f0.elapsed_time(f1))
    h2d = k.numel() * 2 * 2 + q.numel() * 2
    return {
        "w": w, "value": value, "unit": "TFLOP/s", "prefill_encode": None, "ms": ms_max,
        "tokens_per_s": B * T * steps * world / (ms_max * 1e-3), "step_bytes": float(h2d),
        "clocks": clk,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": (achieved / peak) if achieved else None, "traffic": None,
                     "kernel": "tq_prefill_kernel (tcgen05)",
                     "kernel_ms": kern_ms / kern_n if kern_n else None,
                     "kernel_flops": flops, "peak_kind": peak_kind},
        "e2e": {"value": flops * steps * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(out.numel() * 2),
                "ms_per_step": e2e_ms / steps},
        "launches": 2 * steps,
    }


def gpu_arm(args, rank, world, device_index):
    import torch
    import quantized_kv_cache_flash_gb300 as tqf
    from quantized_kv_cache_flash_gb300 import build as tqbuild

    tqbuild.build()
    dev = torch.device("cuda", device_index)
    torch.cuda.set_device(dev)
    w = workload(args)
    lens0 = wl.lengths(wl.by_number(args.workload)).astype(np.int64)[:w.batch]
    t_new = max(w.append, 0)
    steps, warm = args.steps, args.warmup
    kt = KERNEL_STEPS
    grow = t_new * (max(steps, GRAPH_REPLAYS) + warm + kt + 2)
    cap = int(math.ceil((int(lens0.max()) + grow + 16) / 16) * 16)
    B, Hq, Hkv, Tq = w.batch, w.num_q_heads, w.num_kv_heads, w.tq
    mode = tqf.MODES[w.mode]
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + rank)
    ch = torch.tensor(wl.outlier_channels(w), device=dev, dtype=torch.long)

    def randn(shape, outl=False):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        if outl and ch.numel():
            x[..., ch] *= 8.0
        return x.to(torch.float16)

    ctx = tqf.Context()
    cache = tqf.Cache(mode, B, Hkv, cap, dev, rot_seed=w.rot_seed)
    # prefill (untimed): encode max(L)-t_new tokens for every sequence, then trim
    pre = int(lens0.max()) - t_new
    CH = 4096
    done = 0
    while done < pre:
        n = min(CH, pre - done)
        tqf.tq_encode_append(ctx, cache, randn((B, Hkv, n, 128), True),
                             randn((B, Hkv, n, 128)))
        done += n
    cache.lengths.copy_(torch.from_numpy((lens0 - t_new).astype(np.int32)))
    torch.cuda.synchronize()
    assert tqf.tq_get_status(ctx) == 0

    nstep = steps + warm
    qs = [randn((B, Hq, Tq, 128)) for _ in range(nstep + kt)]
    kn = [randn((B, Hkv, t_new, 128), True) for _ in range(nstep + kt)] if t_new else []
    vn = [randn((B, Hkv, t_new, 128)) for _ in range(nstep + kt)] if t_new else []
    out = torch.empty((B, Hq, Tq, 128), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, max_len):
        if t_new:
            tqf.tq_encode_append(ctx, cache, kn[i], vn[i], stream)
        tqf.tq_decode_attention(ctx, cache, qs[i], out, max_len, 0.0, stream)

    # lengths seen by decode at step i: lens0 + i*t_new (append first)
    def lens_at(i):
        return lens0 + i * t_new

    max_len_hint = int(lens0.max()) + grow
    for i in range(warm):
        step(i, max_len_hint)
    torch.cuda.synchronize()
    barrier(world)

    est_bytes = decode_bytes(w, lens0) + append_bytes(w, t_new)
    flush = est_bytes < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    clocks = ClockSampler(device_index)
    clocks.start()
    tqf.tq_set_kernel_timing(ctx, False)
    tqf.tq_get_kernel_time(ctx)   # reset
    torch.cuda.synchronize()

    # The timed steps carry no event between their launches (an event there
    # stops programmatic dependent launch from overlapping them); the decode
    # kernel's own duration comes from KERNEL_STEPS further steps right after
    # them, each decode launch bracketed by the library's event pair.
    def timed_step(i):
        step(i, max_len_hint)

    torch.cuda.nvtx.range_push("timed")   # ncu --nvtx --nvtx-include timed/ selects these launches
    if not flush:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(warm, nstep):
            timed_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
    else:
        # the step's inputs fit in L2: write a 2 x L2 buffer between steps,
        # outside the timed intervals
        evs = []
        for i in range(warm, nstep):
            scratch.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            timed_step(i)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs)
    torch.cuda.nvtx.range_pop()
    # the decode kernel alone (same stream, inputs flushed from L2 when they fit)
    sampled = list(range(nstep, nstep + kt))
    tqf.tq_set_kernel_timing(ctx, True)
    for i in sampled:
        if flush:
            scratch.fill_(float(i))
        step(i, max_len_hint)
    torch.cuda.synchronize()
    clk = clocks.stop()
    kern_ms, kern_n = tqf.tq_get_kernel_time(ctx)
    tqf.tq_set_kernel_timing(ctx, False)
    ms_max = reduce_max(world, ms)
    status = tqf.tq_get_status(ctx)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed steps")

    step_bytes = [decode_bytes(w, lens_at(i)) + append_bytes(w, t_new) for i in range(warm, nstep)]
    kern_bytes = [decode_kernel_bytes(w, lens_at(i)) for i in sampled]
    total_bytes = float(sum(step_bytes)) * world
    value = total_bytes / (ms_max * 1e-3) / 1e9
    tokens = B * Tq * steps * world
    peak, peak_kind = load_peaks()
    achieved = (sum(kern_bytes) / kern_n) / (kern_ms / kern_n * 1e-3) / 1e9 if kern_n else None

    # ---- the same steps back to back with L2 warm (reported separately, as
    # the hot-L2 figure, for workloads whose step fits in L2) ----
    hot = None
    if flush:
        cache.lengths.copy_(torch.from_numpy((lens0 - t_new + warm * t_new).astype(np.int32)))
        torch.cuda.synchronize()
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for i in range(warm, nstep):
            step(i, max_len_hint)
        h1.record(stream)
        torch.cuda.synchronize()
        hot_ms = reduce_max(world, h0.elapsed_time(h1))
        hot = {"value": total_bytes / (hot_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": hot_ms / steps,
               "note": "L2 not flushed: the step's inputs stay in L2 between steps"}

    # ---- the step replayed from one CUDA graph (reported separately): its
    # launches captured once; GRAPH_REPLAYS replays, each reading the inputs of
    # one of the timed steps from static buffers and bracketed by its own
    # events (L2 flushed before each when the step fits in L2) ----
    q_st = torch.empty_like(qs[0])
    k_st = torch.empty_like(kn[0]) if t_new else None
    v_st = torch.empty_like(vn[0]) if t_new else None
    gs = torch.cuda.Stream(device=dev)
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        with torch.cuda.graph(g, stream=gs):
            if t_new:
                tqf.tq_encode_append(ctx, cache, k_st, v_st, gs)
            tqf.tq_decode_attention(ctx, cache, q_st, out, max_len_hint, 0.0, gs)
    torch.cuda.synchronize()
    cache.lengths.copy_(torch.from_numpy((lens0 - t_new + warm * t_new).astype(np.int32)))
    evs = []
    for r in range(GRAPH_REPLAYS):
        i = warm + r % steps
        q_st.copy_(qs[i])
        if t_new:
            k_st.copy_(kn[i])
            v_st.copy_(vn[i])
        if flush:
            scratch.fill_(float(r))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    if tqf.tq_get_status(ctx) != 0:
        raise RuntimeError("device status after the graph-replay leg")
    g_ms = sorted(a.elapsed_time(b) for a, b in evs)
    pct = {q: reduce_max(world, float(np.percentile(g_ms, q))) for q in (10, 50, 90)}
    graph = {"value": total_bytes / steps / (pct[50] * 1e-3) / 1e9, "unit": "GB/s",
             "replays": GRAPH_REPLAYS, "ms_p10": pct[10], "ms_p50": pct[50], "ms_p90": pct[90],
             "note": "one CUDA graph per step (append + decode), each replay timed on its own; value at the "
                     "median" + ("; L2 flushed before each replay" if flush else "; inputs larger than L2")}
    del g

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its q (and new K/V) from pinned host memory and reads
    # its output back.  Steps long enough to hide the extra host calls
    # (> PIPELINE_MIN_MS on the device) run their copies on a second stream,
    # double-buffered: step i+1's inputs go up while step i computes, and step
    # i's output comes down while step i+1 computes.  Shorter steps are bound
    # by the host's calls, so their copies stay on the compute stream.
    qh = [q.cpu().pin_memory() for q in qs]
    knh = [k.cpu().pin_memory() for k in kn]
    vnh = [v.cpu().pin_memory() for v in vn]
    pipelined = ms_max / steps > PIPELINE_MIN_MS
    nbuf = 2 if pipelined else 1
    q_dev = [torch.empty_like(qs[0]) for _ in range(nbuf)]
    k_dev = [torch.empty_like(kn[0]) for _ in range(nbuf)] if t_new else None
    v_dev = [torch.empty_like(vn[0]) for _ in range(nbuf)] if t_new else None
    out_dev = [torch.empty_like(out) for _ in range(nbuf)]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    copy_stream = torch.cuda.Stream(device=dev)
    h2d_ev = [torch.cuda.Event() for _ in range(nbuf)]
    comp_ev = [torch.cuda.Event() for _ in range(nbuf)]
    d2h_ev = [torch.cuda.Event() for _ in range(nbuf)]
    # rewind the cache lengths so the e2e steps see the same contexts
    cache.lengths.copy_(torch.from_numpy((lens0 - t_new + warm * t_new).astype(np.int32)))
    torch.cuda.synchronize()
    barrier(world)

    def upload(i, sl):
        copy_stream.wait_event(comp_ev[sl])      # the step that last read buffer sl is done
        with torch.cuda.stream(copy_stream):
            q_dev[sl].copy_(qh[i], non_blocking=True)
            if t_new:
                k_dev[sl].copy_(knh[i], non_blocking=True)
                v_dev[sl].copy_(vnh[i], non_blocking=True)
        h2d_ev[sl].record(copy_stream)

    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    order = list(range(warm, nstep))
    if pipelined:
        copy_stream.wait_event(f0)
        upload(order[0], 0)
        for j, i in enumerate(order):
            sl = j % nbuf
            if j + 1 < len(order):
                upload(order[j + 1], (j + 1) % nbuf)
            stream.wait_event(h2d_ev[sl])
            stream.wait_event(d2h_ev[sl])              # out_dev[sl] has been read back
            if t_new:
                tqf.tq_encode_append(ctx, cache, k_dev[sl], v_dev[sl], stream)
            tqf.tq_decode_attention(ctx, cache, q_dev[sl], out_dev[sl], max_len_hint, 0.0, stream)
            comp_ev[sl].record(stream)
            copy_stream.wait_event(comp_ev[sl])
            with torch.cuda.stream(copy_stream):
                out_h.copy_(out_dev[sl], non_blocking=True)
            d2h_ev[sl].record(copy_stream)
        done = torch.cuda.Event()
        done.record(copy_stream)
        stream.wait_event(done)
    else:
        for i in order:
            q_dev[0].copy_(qh[i], non_blocking=True)
            if t_new:
                k_dev[0].copy_(knh[i], non_blocking=True)
                v_dev[0].copy_(vnh[i], non_blocking=True)
                tqf.tq_encode_append(ctx, cache, k_dev[0], v_dev[0], stream)
            tqf.tq_decode_attention(ctx, cache, q_dev[0], out_dev[0], max_len_hint, 0.0, stream)
            out_h.copy_(out_dev[0], non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(world, f0.elapsed_time(f1))
    h2d = qs[0].numel() * 2 + (2 * kn[0].numel() * 2 if t_new else 0)
    d2h = out.numel() * 2

    prefill = None
    if w.prefill_chunk:
        T = w.prefill_chunk
        chunks = [(randn((B, Hkv, T, 128), True), randn((B, Hkv, T, 128))) for _ in range(PREFILL_REPS)]
        # PREFILL_REPS chunk appends back to back (the stream never waits on
        # the host; each reads its own inputs), from PREFILL_REPS chunks below
        # the workload's lengths
        times = []
        base = torch.from_numpy((lens0 - PREFILL_REPS * T).astype(np.int32)).to(dev)
        for rep in range(4):
            cache.lengths.copy_(base)
            if flush:
                scratch.fill_(float(rep))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for kc, vc in chunks:
                tqf.tq_encode_append(ctx, cache, kc, vc, stream)
            b.record(stream)
            torch.cuda.synchronize()
            if rep:
                times.append(a.elapsed_time(b) / PREFILL_REPS)
        rk, rv = REC[w.mode]
        pb = B * Hkv * T * (2 * 256 + rk + rv)
        pm = statistics.median(times)
        prefill = {"tokens_per_seq": T, "ms": pm, "GB/s": pb / (pm * 1e-3) / 1e9, "bytes": pb,
                   "vectors": 2 * B * Hkv * T}
        if tqf.tq_get_status(ctx) != 0:
            raise RuntimeError("device status after the prefill encode")

    # sparse V (the V skip of tokens whose softmax weight is below tau) against
    # the plain decode on the same cache, decode kernel alone, for the
    # workload's own queries and for sharper ones (q x 8: most weights tiny)
    sparse = None
    if getattr(args, "sparse_leg", False):
        sparse = []
        L_now = int(cache.lengths.max().item())
        for qscale in (1.0, 8.0):
            q = (qs[0].float() * qscale).to(torch.float16)
            res = {"q_scale": qscale, "tau": SPARSE_TAU}
            for name, tau in (("plain", 0.0), ("sparse_v", SPARSE_TAU)):
                tqf.tq_get_kernel_time(ctx)
                tqf.tq_set_kernel_timing(ctx, True)
                for rep in range(KERNEL_STEPS + 2):
                    if rep == 2:  # two untimed warm-up launches
                        torch.cuda.synchronize()
                        tqf.tq_get_kernel_time(ctx)
                    if tau > 0:
                        tqf.tq_decode_attention_sparse_v(ctx, cache, q, out, L_now, tau, 0.0, stream)
                    else:
                        tqf.tq_decode_attention(ctx, cache, q, out, L_now, 0.0, stream)
                torch.cuda.synchronize()
                kms, kn_ = tqf.tq_get_kernel_time(ctx)
                tqf.tq_set_kernel_timing(ctx, False)
                res[name + "_kernel_us"] = kms / kn_ * 1e3
            skipped, judged = tqf.tq_get_sparse_v_tiles(ctx)
            res["tiles_skipped_fraction"] = skipped / max(judged, 1)
            res["speedup"] = res["plain_kernel_us"] / res["sparse_v_kernel_us"]
            sparse.append(res)
        if tqf.tq_get_status(ctx) != 0:
            raise RuntimeError("device status after the sparse-V leg")

    return {
        "w": w, "value": value, "prefill_encode": prefill, "ms": ms_max, "tokens_per_s": tokens / (ms_max * 1e-3),
        "step_bytes": sum(step_bytes) / steps, "clocks": clk,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None,
                     "traffic": load_traffic(w, sum(kern_bytes) / max(kern_n, 1)),
                     "kernel": "tq_decode_kernel (split-K)",
                     "kernel_ms": kern_ms / kern_n if kern_n else None,
                     "kernel_bytes": sum(kern_bytes) / max(kern_n, 1),
                     "kernel_launches_timed": kern_n,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy), kernel timed inside the step"},
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms / steps,
                "copies": "second stream, double-buffered" if pipelined else "compute stream"},
        "launches": (3 if t_new else 2) * steps,
        "hot_l2": hot,
        "graph": graph,
        "sparse_v": sparse,
    }


EXTRA_WORKLOADS = (2, 3, 5)   # timed besides the headline (4) by the default run
SPARSE_TAU = 1e-6             # the threshold the mlxcel ADR 0002 commit calls exact
EXTRA_STEPS = 30


def workload_summary(r, args):
    """The JSON entry of one more workload: the headline's keys that describe it."""
    d = {"value": r["value"], "unit": r.get("unit", "GB/s"), "steps": args.steps,
         "ms_per_step": r["ms"] / args.steps, "tokens_per_s": r["tokens_per_s"],
         "pct_of_peak": 100.0 * r["value"] / r["roofline"]["peak"], "roofline": r["roofline"],
         "e2e": r["e2e"], "clocks": r["clocks"], "config": config_dict(r["w"]),
         "gpu_launches": r["launches"]}
    if r.get("hot_l2"):
        d["hot_l2"] = r["hot_l2"]
    if r.get("graph"):
        d["graph"] = r["graph"]
    if r.get("prefill_encode"):
        d["prefill_encode"] = r["prefill_encode"]
    return d


def workload(args) -> wl.Workload:
    import dataclasses
    w = wl.by_number(args.workload)
    if args.batch and args.batch != w.batch:
        if args.batch > w.batch:
            raise SystemExit("--batch can only shrink a workload")
        w = dataclasses.replace(w, batch=args.batch, name=f"{w.name}__batch{args.batch}")
    if args.mode and args.mode != w.mode:
        w = dataclasses.replace(w, mode=args.mode, name=f"{w.name}__{args.mode}")
    return w


TRAFFIC_SOURCES = ["quantized_kv_cache_flash_gb300/csrc/tq_decode_kernel.cuh",
                   "quantized_kv_cache_flash_gb300/csrc/tq_decode_q.cu",
                   "quantized_kv_cache_flash_gb300/csrc/tq_device.cuh",
                   "quantized_kv_cache_flash_gb300/csrc/tq_internal.h",
                   "quantized_kv_cache_flash_gb300/csrc/tq_api.cu"]   # (the grid plan)


def decode_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(w, kernel_bytes):
    """DRAM bytes (read + write) per decode launch: the committed ncu capture's
    DRAM bytes per algorithmic byte (profiles/traffic.json, taken on a smaller
    batch of the same workload, traffic growing with the units processed)
    times this launch's algorithmic bytes.  None when the capture does not
    cover this workload or the decode kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p)).get(w.name)
        if not d or d.get("source_hash") != decode_source_hash():
            return None
        return float(d["dram_bytes_per_algorithmic_byte"]) * kernel_bytes
    except Exception:
        return None


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(world, v):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"   # gloo: host tensors
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (small profiling cases only)")
    ap.add_argument("--mode", default=None, choices=sorted(REC),
                    help="run the workload's shapes in another cache mode (format and mode A/B)")
    ap.add_argument("--no-extra", action="store_false", dest="extra",
                    help="time only the chosen workload (the default run of workload 4 also "
                         "times workloads 2, 3 and 5)")
    ap.add_argument("--_oracle-sample", type=int, default=None, dest="oracle_sample")
    ap.add_argument("--_budget", type=float, default=10.0, dest="budget")
    args = ap.parse_args()

    if args.oracle_sample is not None:
        b, s, u, desc = oracle_sample(args.oracle_sample, args.budget, mode=args.mode)
        print(json.dumps({"bytes": b, "seconds": s, "units": u, "desc": desc}))
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workload(args)

    if args.impl == "reference":
        if rank != 0:
            return
        # each step: the oracle on every host core, a bounded sample of the
        # workload per core
        per_step = max(0.5, min(10.0, 100.0 / max(args.steps + args.warmup, 1)))
        pool = OraclePool()
        try:
            for i in range(args.warmup):
                pool.sample(args.workload, per_step / 4, i, args.mode)
            tb, ts = 0, 0.0
            desc = ""
            for i in range(args.steps):
                b, s, u, desc = pool.sample(args.workload, per_step, 1000 + i, args.mode)
                tb += b
                ts += s
        finally:
            pool.close()
        v = tb / ts / (1e12 if w.prompt else 1e9)
        unit = "TFLOP/s" if w.prompt else "GB/s"
        line = {"impl": "reference", "metric": PROMPT_METRIC if w.prompt else METRIC, "value": v,
                "unit": unit,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ts / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_dict(w),
                "cpu_baseline": {"value": v, "unit": unit, "cores": pool.n, "kind": "oracle",
                                 "sample": f"per step: {pool.n} single-threaded processes x ({desc})"},
                "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    args.sparse_leg = (world == 1 and args.extra and args.workload == 4 and not args.batch
                       and not args.mode)
    r = (prompt_arm if w.prompt else gpu_arm)(args, rank, world, local)
    # the other decode configurations of the benchmark, each timed the same
    # way (one GPU, the default run only)
    extra = {}
    if (world == 1 and args.extra and args.workload == 4 and not args.batch and not args.mode):
        import copy
        for n in EXTRA_WORKLOADS:
            a2 = copy.copy(args)
            a2.workload, a2.steps, a2.sparse_leg = n, min(args.steps, EXTRA_STEPS), False
            x = gpu_arm(a2, rank, world, local)
            extra[x["w"].name] = workload_summary(x, a2)
    cpu = (run_cpu_baseline(args.workload, args.cpu_budget, args.mode)
           if (rank == 0 and world == 1) else None)
    if rank == 0:
        rf = r["roofline"]
        line = {
            "metric": PROMPT_METRIC if w.prompt else METRIC, "value": r["value"],
            "unit": r.get("unit", "GB/s"), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16xf16->f32 (mma), fp32 softmax", "data": "synthetic",
            "config": config_dict(w),
            "tokens_per_s": r["tokens_per_s"],
            "pct_of_peak": 100.0 * r["value"] / rf["peak"],
            "roofline": rf, "cpu_baseline": cpu, "e2e": r["e2e"], "clocks": r["clocks"],
            "gpu_launches": r["launches"], "impl": "ours",
            "prefill_encode": r["prefill_encode"],
        }
        if r.get("hot_l2"):
            line["hot_l2"] = r["hot_l2"]
        if r.get("graph"):
            line["graph"] = r["graph"]
        if extra:
            line["other_workloads"] = extra
        if r.get("sparse_v"):
            line["sparse_v"] = r["sparse_v"]
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
