#!/usr/bin/env python
"""Benchmark of the NVFP4 paged KV cache decode step on GB300.

Workload (one GPU; N GPUs run N independent replicas): batch 64, every
sequence 32,768 cached tokens, 64 query heads over 8 KV heads (GQA 8),
head_dim 128, 64-token pages under a randomly permuted block table, K/V/Q
drawn N(0,1) -- the 32K iso-concurrency shape of "Accelerating Long-Context
and Agentic Inference with NVFP4 KV Cache" (A4, decode performance).

One step = the whole hot path of a decode step: quantise-append of the new
token of every sequence (64 tokens x 8 KV heads) into the paged cache, then
paged GQA decode attention over all 32,768 tokens (plan, decode, split
reduction).  The cache (2.42 GB) is far larger than L2, so no flush is needed
between steps.

value = HBM GB/s on algorithmic bytes (packed KV + scales + block table + Q +
out, plus the append's BF16 reads and packed writes) / device time per step.
roofline = the decode kernel alone, timed with CUDA events recorded around its
launch on the launching stream, against the measured HBM copy bandwidth.

`--impl reference` times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload and prints the same JSON line with
"impl": "reference".
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 paged decode-attn: HBM GB/s (% of GB300 peak), KV-tokens/s, µs/step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PROFILE_EVERY = 8   # decode-kernel events on every 8th timed step (events between launches cost overlap)
ROOFLINE_LAUNCHES = 256   # decode launches timed one by one after the timed region, whatever --steps is


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-comparisons", action="store_true")
    p.add_argument("--num-splits", type=int, default=0)
    p.add_argument("--batch", type=int, default=64,
                   help="sequences of the 32K workload (64 = the benchmark; smaller = a profiling case)")
    p.add_argument("--comparison", choices=["extend", "agent_decode", "agent_step", "append", "calibrate"], default=None,
                   help="run only this comparison (its own JSON line; a profiling case) and exit")
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers

def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_bf16_peak():
    """Measured dense BF16 TFLOP/s (burst, for a kernel timed alone), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def decode_bytes(batch, seq_len, hq, hkv, max_pages, dtype_bytes_per_token_head):
    """Algorithmic bytes of one decode call: KV (+ scales) + block table + Q + out."""
    kv = batch * seq_len * hkv * dtype_bytes_per_token_head
    return kv + batch * max_pages * 4 + 2 * batch * hq * 128 * 2 + batch * 4


def append_bytes(tokens, hkv, packed_bytes_per_token_head):
    """Algorithmic bytes of one quantise-append: BF16 K/V in, packed rows out, slots."""
    return tokens * hkv * 2 * 128 * 2 + tokens * hkv * packed_bytes_per_token_head + tokens * 8


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        try:
            cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if gpu_id:
                cmd += ["-i", gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1 and len(s) == len(self.FIELDS)]
        note = "samples inside the timed region"
        if not rows:  # timed region shorter than the sampling period: take the nearest samples
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))
            rows = [s for (_, s) in near[:3] if len(s) == len(self.FIELDS)]
            note = "nearest samples (timed region shorter than the 50 ms sampling period)"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(r[0]) for r in rows) if v is not None)
        mx = [v for v in (num(r[1]) for r in rows) if v is not None]
        reasons = set()
        for r in rows:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"],
                                 r[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "note": note}


def decode_kernel_traffic(batch, num_splits):
    """DRAM bytes per decode-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source and covers this batch of the 32K
    workload with the automatic split (else None)."""
    if num_splits:
        return None
    key = {64: "dram_bytes_per_launch_full_size", 8: "dram_bytes_per_launch_batch8"}.get(batch)
    if key is None:
        return None
    src = os.path.join(ROOT, "nvfp4_quantised_paged_gb300", "csrc", "decode_attention.cu")
    summ = os.path.join(ROOT, "profiles", "decode_kernel_dram.txt")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        kv = {}
        for line in open(summ):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") == h:
            return float(kv[key])
    except Exception:
        pass
    return None


def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return world, rank, local, dist
    return 1, 0, 0, None


def max_over_ranks(dist, x):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle leg

def oracle_decode_sample(w, nseq, seed_device="cpu"):
    """Builds the oracle's own pool for the first `nseq` sequences of the
    workload (untimed) and returns a callable running one oracle decode over
    them, plus the algorithmic bytes that call covers."""
    import numpy as np
    import torch

    import oracle

    seqs = list(range(nseq))
    pages = sorted({int(p) for b in seqs for p in w.block_table[b].tolist() if p >= 0})
    remap = {p: i for i, p in enumerate(pages)}
    bt = w.block_table[seqs].clone()
    bt = torch.tensor([[remap[int(p)] if p >= 0 else -1 for p in row] for row in bt.tolist()], dtype=torch.int32)
    pool = oracle.OraclePool(len(pages), w.page_size, w.num_kv_heads)

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    for b in seqs:
        k, v = w.seq_kv(b, seed_device)
        t = torch.arange(int(w.seq_lens[b]))
        slots = bt[b].to(torch.int64)[t // w.page_size] * w.page_size + t % w.page_size
        oracle.quantize_append(pool, bits(k), bits(v), slots.numpy())
    q = bits(w.q(seed_device)[:nseq])
    sl = w.seq_lens[:nseq].numpy()
    cores = os.cpu_count() or 1

    def run(nthreads=cores):
        return oracle.decode_attention(pool, q, bt.numpy(), sl, w.sm_scale, nthreads=nthreads)

    nbytes = decode_bytes(nseq, int(w.seq_lens[0]), w.num_q_heads, w.num_kv_heads, w.max_pages, 144)
    return run, nbytes, cores


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86 'model name', Arm implementer / part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model"):
        for ln in info.splitlines():
            if ln.startswith(key):
                return ln.split(":", 1)[1].strip()
    impl = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")]
    part = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")]
    return "Arm implementer %s part %s" % (impl[0] if impl else "?", part[0] if part else "?")


def cpu_baseline(w, seed_device):
    cores = os.cpu_count() or 1
    nseq = max(1, min(w.batch, math.ceil(cores / w.num_kv_heads)))
    run, nbytes, cores = oracle_decode_sample(w, nseq, seed_device)
    run()  # warm
    t0 = time.perf_counter()
    reps = 0
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 > 10.0:
            break
    dt = (time.perf_counter() - t0) / reps
    # one thread on one sequence (all its kv heads), a few seconds of work
    run1, nbytes1, _ = oracle_decode_sample(w, 1, seed_device)
    t1 = time.perf_counter()
    reps1 = 0
    while True:
        run1(nthreads=1)
        reps1 += 1
        if time.perf_counter() - t1 > 3.0:
            break
    dt1 = (time.perf_counter() - t1) / reps1
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d of %d sequences (%d (seq, kv_head) units of %d tokens), fp64 decode over the oracle's "
                      "own NVFP4 pool, %d repetitions" % (nseq, w.batch, nseq * w.num_kv_heads,
                                                          int(w.seq_lens[0]), reps),
            "ms_per_sample": dt * 1e3, "cpu_model": cpu_model(),
            "single_thread": {"value": nbytes1 / dt1 / 1e9, "unit": "GB/s", "ms_per_sample": dt1 * 1e3,
                              "sample": "1 sequence x %d kv heads, %d repetitions" % (w.num_kv_heads, reps1)}}


def workload_config(w, world):
    """The workload keys of the reference arm's "config" (the GPU arm reports
    the same keys, plus its step and split count)."""
    return {"workload": w.name, "batch": w.batch, "seq_len": int(w.seq_lens[0]), "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": 128, "page_size": w.page_size,
            "kv_cache": "nvfp4 (e2m1 + e4m3 per 16, tensor scale 1.0)",
            "l2": "inputs larger than L2 (2.42 GB cache vs 129 MB L2), no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args):
    import workloads
    world, rank, local, dist = init_dist()
    if rank != 0:
        return
    w = workloads.decode_32k()
    cores = os.cpu_count() or 1
    nseq = max(1, min(w.batch, math.ceil(cores / w.num_kv_heads)))
    run, nbytes, cores = oracle_decode_sample(w, nseq, "cpu")
    for _ in range(max(0, args.warmup)):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = nbytes / dt / 1e9
    sample = "%d of %d sequences x %d KV heads per step (%d tokens each), fp64 oracle decode on %d host threads" % (
        nseq, w.batch, w.num_kv_heads, int(w.seq_lens[0]), cores)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w, world), step="paged decode attention of the sampled sequences",
                           sample=sample),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU leg

def fill_cache(m, w, cache, device):
    for b in range(w.batch):
        k, v = w.seq_kv(b, device)
        m.quantize_append(cache, k, v, w.slots(b).to(device))
        del k, v


def time_decode_only(m, w, dtype, device, steps, warmup):
    """Decode-kernel time and whole-call time (µs; plan + decode + reduce, calls
    back to back) for workload w over a cache of `dtype` (used for the FP8
    byte-ratio comparison and the long-context workload)."""
    import torch
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, dtype=dtype, device=device)
    fill_cache(m, w, cache, device)
    q = w.q(device)
    bt, sl = w.block_table.to(device), w.seq_lens.to(device)
    ws = m.alloc_decode_workspace(cache, w.batch, w.num_q_heads)
    out = torch.empty_like(q)
    for _ in range(warmup):
        m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws)
    before = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    after = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    m.profile_decode(before, after)
    torch.cuda.synchronize()
    for _ in range(steps):
        m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    m.profile_decode([], [])
    us = sum(b.elapsed_time(a) for b, a in zip(before, after)) / steps * 1e3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    call_us = e0.elapsed_time(e1) / steps * 1e3
    assert m.check_device_errors() == 0
    del cache
    torch.cuda.empty_cache()
    return us, call_us


def time_append(m, device, steps, warmup):
    import torch

    import workloads
    w = workloads.append_65k()
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, device=device)
    k, v = w.kv(device)
    slots = w.slot_mapping().to(device)
    for _ in range(warmup):
        m.quantize_append(cache, k, v, slots)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(steps):
        m.quantize_append(cache, k, v, slots)
    e.record()
    torch.cuda.synchronize()
    us = s.elapsed_time(e) / steps * 1e3
    nbytes = append_bytes(w.num_tokens, w.num_kv_heads, 144)
    # the same tokens written page by page (a prefill's layout: pages in a seeded
    # order, rows of a page in order) instead of to random slots
    g = torch.Generator().manual_seed(5)
    P = w.page_size
    paged = (torch.randperm(w.num_pages, generator=g)[:w.num_tokens // P].repeat_interleave(P) * P
             + torch.arange(w.num_tokens) % P).to(torch.int64).to(device)
    for _ in range(warmup):
        m.quantize_append(cache, k, v, paged)
    torch.cuda.synchronize()
    s.record()
    for _ in range(steps):
        m.quantize_append(cache, k, v, paged)
    e.record()
    torch.cuda.synchronize()
    us_paged = s.elapsed_time(e) / steps * 1e3
    return {"workload": w.name, "us_per_call": us, "gb_per_s": nbytes / us / 1e3, "algorithmic_bytes": nbytes,
            "page_ordered_us_per_call": us_paged, "page_ordered_gb_per_s": nbytes / us_paged / 1e3,
            "note": "back-to-back calls; 268 MB of BF16 input per call exceeds the 129 MB L2; the workload's slots "
                    "are a random permutation, page_ordered writes the same tokens page by page"}


def time_calibrate(m, device, steps, warmup):
    """Tensor-scale calibration (amax of K and V) over the 65,536-token append input."""
    import torch

    import workloads
    w = workloads.append_65k()
    k, v = w.kv(device)
    for _ in range(warmup):
        m.calibrate_global_scales(k, v, w.num_kv_heads)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(steps):
        m.calibrate_global_scales(k, v, w.num_kv_heads)
    e.record()
    torch.cuda.synchronize()
    us = s.elapsed_time(e) / steps * 1e3
    nbytes = 2 * w.num_tokens * w.num_kv_heads * 128 * 2
    return {"workload": w.name, "us_per_call": us, "gb_per_s": nbytes / us / 1e3, "algorithmic_bytes": nbytes,
            "note": "reads K and V once (BF16); back-to-back calls over 268 MB, beyond the 129 MB L2"}


def extend_flops(prefix_lens, chunk, G, Hkv):
    """Algorithmic FLOPs of extend attention: 2 * 2 * 128 per (query row, visible key)."""
    return sum(Hkv * G * (chunk * p + chunk * (chunk + 1) // 2) for p in prefix_lens) * 4 * 128


def time_extend(m, device, steps, warmup, peak_tflops):
    """Path 2 on the agent mix's 8 extend requests: prefix dequant of their cached
    prefixes (NVFP4 pages -> BF16 workspace), then extend attention of each
    512-token chunk over [prefix || chunk]; and the same in one call with the
    prefix expanded from the pages inside the kernel (paged_us)."""
    import torch

    import workloads
    mix = workloads.agent_mix()
    w = mix.decode
    rows = mix.extend_rows()
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, device=device)
    for row in rows:
        k, v = w.seq_kv(row, device)
        m.quantize_append(cache, k, v, w.slots(row).to(device))
        del k, v
    pl = w.seq_lens[rows].contiguous()
    cu_p = torch.zeros(len(rows) + 1, dtype=torch.int32)
    cu_p[1:] = torch.cumsum(pl, 0)
    bt, pl_d, cu_p_d = w.block_table[rows].contiguous().to(device), pl.to(device), cu_p.to(device)
    total = int(cu_p[-1])
    L = mix.chunk_tokens
    q = torch.cat([mix.chunk_q(r, device) for r in range(len(rows))])
    kn = torch.cat([mix.chunk_kv(r, device)[0] for r in range(len(rows))])
    vn = torch.cat([mix.chunk_kv(r, device)[1] for r in range(len(rows))])
    cu_q = torch.arange(0, L * (len(rows) + 1), L, dtype=torch.int32, device=device)
    kw, vw = m.prefix_dequant(cache, bt, pl_d, cu_p_d, total)
    out = torch.empty_like(q)

    def run(with_dequant):
        if with_dequant:
            m.prefix_dequant(cache, bt, pl_d, cu_p_d, total, k_ws=kw, v_ws=vw)
        m.extend_attention(q, kw, vw, cu_p_d, kn, vn, cu_q, L, w.sm_scale, out=out)

    res = {"workload": "agent-mix extends: 8 x 512-token chunks over prefixes of %s tokens, q32kv8"
           % "/".join(str(int(x)) for x in pl)}
    def dequant_only():
        m.prefix_dequant(cache, bt, pl_d, cu_p_d, total, k_ws=kw, v_ws=vw)

    def paged():  # path 2 in one call: the prefix expanded from the NVFP4 pages inside the kernel
        m.extend_attention_paged(cache, q, bt, pl_d, kn, vn, cu_q, L, w.sm_scale, out=out)

    for key, fn in (("extend_us", lambda: run(False)), ("path2_us", lambda: run(True)), ("dequant_us", dequant_only),
                    ("paged_us", paged)):
        for _ in range(warmup):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        res[key] = s.elapsed_time(e) / steps * 1e3
    assert m.check_device_errors() == 0
    dq_bytes = total * w.num_kv_heads * (144 + 2 * 2 * 128)  # NVFP4 in, BF16 K and V out
    res["dequant_gb_per_s"] = dq_bytes / res["dequant_us"] / 1e3
    res["dequant_algorithmic_bytes"] = dq_bytes
    flops = extend_flops([int(x) for x in pl], L, w.num_q_heads // w.num_kv_heads, w.num_kv_heads)
    res.update({"paged_tflops": flops / res["paged_us"] / 1e6, "paged_over_path2_time": res["paged_us"] / res["path2_us"],
                "workspace_bytes_saved": total * w.num_kv_heads * 2 * 2 * 128})
    res.update({"algorithmic_flops": flops, "extend_tflops": flops / res["extend_us"] / 1e6,
                "extend_frac_of_bf16_peak": flops / res["extend_us"] / 1e6 / peak_tflops,
                "bf16_peak_tflops": peak_tflops,
                "note": "tcgen05 (TMEM accumulators) BF16 kernel; peak = measured cuBLAS BF16 burst"})
    del cache
    torch.cuda.empty_cache()
    return res


def time_agent_decode(m, device, steps, warmup):
    """Decode of the agent mix's 128 sequences (shared 3,200-token prefix): the plain
    decode call against the cascade call that attends the shared pages once per kv head."""
    import torch

    import workloads
    mix = workloads.agent_mix()
    w = mix.decode
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, device=device)
    fill_cache(m, w, cache, device)
    dec = list(range(mix.num_decode))
    q = w.q(device)[dec].contiguous()
    bt = w.block_table[dec].contiguous().to(device)
    sl = w.seq_lens[dec].contiguous().to(device)
    shared = w.shared_prefix_tokens
    sp = w.block_table[0, :shared // w.page_size].contiguous().to(device)
    out = torch.empty_like(q)
    ws = torch.empty(max(m.cascade_workspace_bytes(cache, len(dec), w.num_q_heads, shared), 256),
                     dtype=torch.uint8, device=device)
    res = {"workload": "agent-mix decode: 128 sequences of %d-%d tokens sharing %d, q32kv8 p64"
           % (int(sl.min()), int(sl.max()), shared)}
    calls = {"plain_us": lambda: m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws),
             "cascade_us": lambda: m.cascade_decode_attention(cache, q, sp, shared, bt, sl, w.sm_scale, out=out,
                                                              workspace=ws)}
    for key, fn in calls.items():
        for _ in range(warmup):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        res[key] = s.elapsed_time(e) / steps * 1e3
    assert m.check_device_errors() == 0
    logical = int(sl.sum()) * w.num_kv_heads * 144
    unique = (int(sl.sum()) - (len(dec) - 1) * shared) * w.num_kv_heads * 144
    res.update({"logical_kv_bytes": logical, "unique_kv_bytes": unique,
                "plain_logical_gb_per_s": logical / res["plain_us"] / 1e3,
                "cascade_logical_gb_per_s": logical / res["cascade_us"] / 1e3,
                "cascade_speedup": res["plain_us"] / res["cascade_us"]})
    del cache
    torch.cuda.empty_cache()
    return res


def time_agent_step(m, device, steps, warmup):
    """One step of the whole agent mix: cascade decode of the 128 sequences, then
    path 2 of the 8 extends (prefix dequant, extend attention, quantise-append of
    their chunks)."""
    import torch

    import workloads
    mix = workloads.agent_mix()
    w = mix.decode
    P = w.page_size
    cache = m.PagedCache(w.num_pages, P, w.num_kv_heads, device=device)
    fill_cache(m, w, cache, device)  # decode rows, and the extend rows' prefixes
    dec, rows = list(range(mix.num_decode)), mix.extend_rows()
    q = w.q(device)[dec].contiguous()
    bt_d, sl_d = w.block_table[dec].contiguous().to(device), w.seq_lens[dec].contiguous().to(device)
    shared = w.shared_prefix_tokens
    sp = w.block_table[0, :shared // P].contiguous().to(device)
    ws = torch.empty(max(m.cascade_workspace_bytes(cache, len(dec), w.num_q_heads, shared), 256), dtype=torch.uint8,
                     device=device)
    pl = w.seq_lens[rows].contiguous()
    cu_p = torch.zeros(len(rows) + 1, dtype=torch.int32)
    cu_p[1:] = torch.cumsum(pl, 0)
    total = int(cu_p[-1])
    bt_e, pl_d, cu_p_d = w.block_table[rows].contiguous().to(device), pl.to(device), cu_p.to(device)
    L = mix.chunk_tokens
    qc = torch.cat([mix.chunk_q(r, device) for r in range(len(rows))])
    kn = torch.cat([mix.chunk_kv(r, device)[0] for r in range(len(rows))])
    vn = torch.cat([mix.chunk_kv(r, device)[1] for r in range(len(rows))])
    cu_q = torch.arange(0, L * (len(rows) + 1), L, dtype=torch.int32, device=device)
    slots_c = torch.cat([mix.chunk_slots(r) for r in range(len(rows))]).to(device)
    kw, vw = m.prefix_dequant(cache, bt_e, pl_d, cu_p_d, total)
    out_d, out_e = torch.empty_like(q), torch.empty_like(qc)

    def step():
        m.cascade_decode_attention(cache, q, sp, shared, bt_d, sl_d, w.sm_scale, out=out_d, workspace=ws)
        m.prefix_dequant(cache, bt_e, pl_d, cu_p_d, total, k_ws=kw, v_ws=vw)
        m.extend_attention(qc, kw, vw, cu_p_d, kn, vn, cu_q, L, w.sm_scale, out=out_e)
        m.quantize_append(cache, kn, vn, slots_c)

    for _ in range(warmup):
        step()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    us = s.elapsed_time(e) / steps * 1e3
    Hkv = w.num_kv_heads
    unique = (int(sl_d.sum()) - (len(dec) - 1) * shared) * Hkv * 144   # decode: the shared pages counted once
    extend_bytes = total * Hkv * (144 + 4 * 128) + len(rows) * L * Hkv * (512 + 144)
    flops = extend_flops([int(x) for x in pl], L, w.num_q_heads // Hkv, Hkv)
    del cache
    torch.cuda.empty_cache()
    return {"workload": "agent mix step: cascade decode of 128 sequences + path 2 of 8 extends of 512 tokens",
            "us_per_step": us, "unique_bytes_per_step": unique + extend_bytes,
            "unique_gb_per_s": (unique + extend_bytes) / us / 1e3, "extend_flops_per_step": flops}


def run_ours(args):
    import torch

    import nvfp4_quantised_paged_gb300 as m
    import workloads

    world, rank, local, dist = init_dist()
    torch.cuda.set_device(local)
    device = "cuda:%d" % local
    w = workloads.decode_32k() if args.batch == 64 else workloads.make_decode(
        "decode b%d s32768 q64kv8 p64" % args.batch, 1003, [32_768] * args.batch, 64, 8, 64)
    B, S, Hq, Hkv, P = w.batch, int(w.seq_lens[0]), w.num_q_heads, w.num_kv_heads, w.page_size

    cache = m.PagedCache(w.num_pages, P, Hkv, device=device)
    fill_cache(m, w, cache, device)
    q = w.q(device)
    bt, sl = w.block_table.to(device), w.seq_lens.to(device)
    # the step's new token of every sequence goes to position S-1
    g = torch.Generator(device=device)
    g.manual_seed(4242)
    new_k = torch.randn((B, Hkv, 128), generator=g, device=device).to(torch.bfloat16)
    new_v = torch.randn((B, Hkv, 128), generator=g, device=device).to(torch.bfloat16)
    new_slots = torch.cat([w.slots(b, S - 1, S) for b in range(B)]).to(device)
    ws = m.alloc_decode_workspace(cache, B, Hq, args.num_splits)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def step():   # one call: plan, decode with the new token appended in-kernel (and the reduction, or a reduction kernel)
        m.paged_decode_attention_append(cache, new_k, new_v, q, bt, sl, w.sm_scale, out=out, workspace=ws,
                                        num_splits=args.num_splits)

    def two_call_step():   # the same work as a quantise-append call followed by a decode call
        m.quantize_append(cache, new_k, new_v, new_slots)
        m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws, num_splits=args.num_splits)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0

    K = args.steps
    # the decode kernel is timed on every PROFILE_EVERY-th step of the timed region
    n_prof = (K + PROFILE_EVERY - 1) // PROFILE_EVERY
    before = [torch.cuda.Event(enable_timing=True) for _ in range(n_prof)]
    after = [torch.cuda.Event(enable_timing=True) for _ in range(n_prof)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    m.profile_decode(before, after, PROFILE_EVERY)
    barrier(dist)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(K):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(dist)
    m.profile_decode([], [])
    assert m.check_device_errors() == 0
    ms_step = max_over_ranks(dist, ev0.elapsed_time(ev1) / K)
    region_samples = sorted(b.elapsed_time(a) * 1e3 for b, a in zip(before, after))
    region_us = max_over_ranks(dist, sum(region_samples) / n_prof)

    # the roofline kernel on its own: ROOFLINE_LAUNCHES more steps, each with its
    # decode-kernel launch bracketed by events (the step's other launches run too)
    nr = ROOFLINE_LAUNCHES
    rb = [torch.cuda.Event(enable_timing=True) for _ in range(nr)]
    ra = [torch.cuda.Event(enable_timing=True) for _ in range(nr)]
    m.profile_decode(rb, ra, 1)
    torch.cuda.synchronize()
    t_roof0 = time.time()
    for _ in range(nr):
        step()
    torch.cuda.synchronize()
    t_roof1 = time.time()
    m.profile_decode([], [])
    assert m.check_device_errors() == 0
    dec_samples = sorted(b.elapsed_time(a) * 1e3 for b, a in zip(rb, ra))
    dec_us = max_over_ranks(dist, sum(dec_samples) / nr)
    dec_median_us = max_over_ranks(dist, dec_samples[nr // 2])

    time.sleep(0.1)
    sampler.stop()

    dbytes = decode_bytes(B, S, Hq, Hkv, w.max_pages, 144)
    abytes = append_bytes(B, Hkv, 144)
    step_bytes = dbytes + abytes
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    kv_tokens_per_s = world * B * S / (ms_step * 1e-3)

    # the same step as two calls (quantise-append, then decode), for comparison
    for _ in range(3):
        two_call_step()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(K):
        two_call_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    two_call_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / K)

    # ---- end to end through the public API with host buffers
    q_h = q.cpu().pin_memory()
    k_h, v_h = new_k.cpu().pin_memory(), new_v.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, k_d, v_d = torch.empty_like(q), torch.empty_like(new_k), torch.empty_like(new_v)

    def e2e_step():
        q_d.copy_(q_h, non_blocking=True)
        k_d.copy_(k_h, non_blocking=True)
        v_d.copy_(v_h, non_blocking=True)
        m.paged_decode_attention_append(cache, k_d, v_d, q_d, bt, sl, w.sm_scale, out=out, workspace=ws,
                                        num_splits=args.num_splits)
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier(dist)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(K):
        e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / K)

    # The same with the copies on a second stream, double-buffered: the inputs of
    # step i + 1 go up and the output of step i comes back while step i + 1's
    # kernels run (as a serving loop overlaps them); every step's copies stay
    # inside the timed region.
    copy = torch.cuda.Stream()
    sets = [(torch.empty_like(q), torch.empty_like(new_k), torch.empty_like(new_v), torch.empty_like(out))
            for _ in range(2)]
    up = [torch.cuda.Event() for _ in range(2)]      # inputs of the set landed
    done = [torch.cuda.Event() for _ in range(2)]    # the set's kernels finished
    down = [torch.cuda.Event() for _ in range(2)]    # the set's output read back

    def h2d_issue(i):
        qs, ks, vs, _ = sets[i & 1]
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(done[i & 1])  # step i - 2 has read this set
            qs.copy_(q_h, non_blocking=True)
            ks.copy_(k_h, non_blocking=True)
            vs.copy_(v_h, non_blocking=True)
            up[i & 1].record(copy)

    def compute_issue(i):
        qs, ks, vs, os_ = sets[i & 1]
        stream.wait_event(up[i & 1])
        if i >= 2:
            stream.wait_event(down[i & 1])  # step i - 2's output has been read back
        m.paged_decode_attention_append(cache, ks, vs, qs, bt, sl, w.sm_scale, out=os_, workspace=ws,
                                        num_splits=args.num_splits)
        done[i & 1].record(stream)

    def d2h_issue(i):
        with torch.cuda.stream(copy):
            copy.wait_event(done[i & 1])
            out_h.copy_(sets[i & 1][3], non_blocking=True)
            down[i & 1].record(copy)

    def pipelined(n):
        h2d_issue(0)
        for i in range(n):
            if i + 1 < n:
                h2d_issue(i + 1)
            compute_issue(i)
            d2h_issue(i)
        stream.wait_event(down[(n - 1) & 1])

    pipelined(3)
    torch.cuda.synchronize()
    barrier(dist)
    ev0.record(stream)
    copy.wait_stream(stream)
    pipelined(K)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / K)
    assert m.check_device_errors() == 0
    h2d = q.numel() * 2 + new_k.numel() * 2 * 2
    d2h = out.numel() * 2

    peak, peak_kind = peak_hbm()
    achieved = dbytes / (dec_us * 1e-6) / 1e9
    traffic = decode_kernel_traffic(B, args.num_splits)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16->f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": B, "seq_len": S, "num_q_heads": Hq, "num_kv_heads": Hkv,
                   "head_dim": 128, "page_size": P, "kv_cache": "nvfp4 (e2m1 + e4m3 per 16, tensor scale 1.0)",
                   "step": "quantize-append of 1 new token per sequence + paged decode attention, one fused call",
                   "l2": "inputs larger than L2 (2.42 GB cache vs 129 MB L2), no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "num_splits": args.num_splits or m.decode_auto_splits(cache, Hq)},
        "us_per_step": ms_step * 1e3, "kv_tokens_per_s": kv_tokens_per_s,
        "pct_of_nominal_8tbps": 100.0 * (value / world) / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": 100.0 * (value / world) / peak,
        "algorithmic_bytes_per_step": step_bytes,
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "pinned host buffers; each step's inputs up and output back on a second stream, "
                          "double-buffered, overlapping the neighbouring steps' kernels",
                "serial_ms_per_step": e2e_serial_ms,
                "serial_value": world * step_bytes / (e2e_serial_ms * 1e-3) / 1e9},
        "gpu_launches": m.decode_launch_count(cache, B, Hq, args.num_splits) * K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "decode_kernel<nvfp4>", "us_per_launch": dec_us, "median_us_per_launch": dec_median_us,
                     "min_us_per_launch": dec_samples[0], "max_us_per_launch": dec_samples[-1],
                     "timed_launches": nr, "algorithmic_bytes_per_launch": dbytes,
                     "timing": "%d fused steps after the timed region, the decode-kernel launch of each bracketed by "
                               "CUDA events on its stream" % nr,
                     "clocks": sampler.summary(t_roof0, t_roof1),
                     "in_timed_region": {"us_per_launch": region_us, "timed_launches": n_prof,
                                         "every": PROFILE_EVERY}},
        "clocks": sampler.summary(t_wall0, t_wall1),
    }

    # single-GPU comparisons: reported at N = 1 only (under torchrun the other GPUs would wait idle)
    if not args.no_comparisons and rank == 0 and world == 1:
        comp = {"two_call_step": {"ms_per_step": two_call_ms, "value": world * step_bytes / (two_call_ms * 1e-3) / 1e9,
                                  "unit": "GB/s", "note": "quantize_append then paged_decode_attention (4 launches)"}}
        del cache
        torch.cuda.empty_cache()
        fp8_us, fp8_call = time_decode_only(m, w, 1, device, 100, 5)
        comp["fp8_e4m3_cache_same_workload"] = {
            "decode_us": fp8_us, "call_us": fp8_call, "nvfp4_decode_us": dec_us, "nvfp4_over_fp8_time": dec_us / fp8_us,
            "fp8_gb_per_s": decode_bytes(B, S, Hq, Hkv, w.max_pages, 256) / fp8_us / 1e3,
            "pct_of_nominal_8tbps": 100.0 * decode_bytes(B, S, Hq, Hkv, w.max_pages, 256) / fp8_us / 1e3 /
            NOMINAL_HBM_GBS, "kv_byte_ratio": 144 / 256}
        w4 = workloads.decode_1m()
        us4, call4 = time_decode_only(m, w4, 0, device, 50, 5)
        b4 = decode_bytes(w4.batch, int(w4.seq_lens[0]), w4.num_q_heads, w4.num_kv_heads, w4.max_pages, 144)
        fp8_us4, fp8_call4 = time_decode_only(m, w4, 1, device, 50, 5)
        b4_fp8 = decode_bytes(w4.batch, int(w4.seq_lens[0]), w4.num_q_heads, w4.num_kv_heads, w4.max_pages, 256)
        comp["decode_1m"] = {"workload": w4.name, "decode_us": us4, "gb_per_s": b4 / us4 / 1e3,
                             "pct_of_measured_hbm": 100.0 * b4 / us4 / 1e3 / peak,
                             "pct_of_nominal_8tbps": 100.0 * b4 / us4 / 1e3 / NOMINAL_HBM_GBS,
                             "call_us": call4, "call_gb_per_s": b4 / call4 / 1e3,
                             "kv_tokens_per_s": 2 * 1048576 / (call4 * 1e-6),
                             "fp8_e4m3_cache": {"decode_us": fp8_us4, "call_us": fp8_call4,
                                                "fp8_gb_per_s": b4_fp8 / fp8_us4 / 1e3,
                                                "nvfp4_over_fp8_time": us4 / fp8_us4, "kv_byte_ratio": 144 / 256}}
        comp["append_65k"] = time_append(m, device, 50, 5)
        comp["calibrate_65k"] = time_calibrate(m, device, 50, 5)
        comp["extend_agent_mix"] = time_extend(m, device, 10, 2, load_bf16_peak())
        comp["decode_agent_mix"] = time_agent_decode(m, device, 20, 3)
        comp["agent_mix_step"] = time_agent_step(m, device, 10, 2)
        line["comparisons"] = comp

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, device)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_comparison(args):
    """One comparison on its own, for a profiler to capture its kernels."""
    import torch

    import nvfp4_quantised_paged_gb300 as m
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    if args.comparison == "extend":
        res = time_extend(m, device, args.steps, args.warmup, load_bf16_peak())
    elif args.comparison == "append":
        res = time_append(m, device, args.steps, args.warmup)
    elif args.comparison == "calibrate":
        res = time_calibrate(m, device, args.steps, args.warmup)
    elif args.comparison == "agent_step":
        res = time_agent_step(m, device, args.steps, args.warmup)
    else:
        res = time_agent_decode(m, device, args.steps, args.warmup)
    print(json.dumps({"comparison": args.comparison, **res}), flush=True)


def main():
    args = parse_args()
    if args.comparison:
        run_comparison(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
