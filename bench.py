#!/usr/bin/env python3
"""Paged-attention decode benchmark on GB300 (one JSON line on rank 0).

A step is one pass of the hot path over one batch: for every layer pool, the cache write
of the newest tokens (pa_cache_write) and the paged decode (pa_decode: decode kernel plus
the partition merge). Default workload: Llama-3-70B-shaped decode, 64 sequences x 8192
tokens, Hq 64 / Hkv 8 / d 128, block size 16, fp16, 80 independent layer pools (172 GB of
KV, far larger than L2, so no flush is needed between steps). The same run then times the
long-context split decode (4 sequences x 131072 tokens, 512-token partitions) and reports it
in the line's `secondary` object (`--no-secondary` skips it).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload cfg3|cfg5|cfg2|cfg4|cfg1|verify70b]
    python bench.py --impl reference      # the fp64 CPU oracle as the reference arm
    python bench.py --workload prefill    # chunked prefill (pa_prefill), tensor-core bound: TFLOP/s
    python bench.py --workload cow        # copy-on-write block copies (pa_copy_blocks): GB/s
    python bench.py --workload spec       # speculative rejection sampling (pa_spec_verify): GB/s

Under torchrun each rank runs the same workload on its own GPU (weak scaling, no collective
on the data path); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import synth  # noqa: E402

WORKLOADS = {"cfg1": 1, "cfg2": 2, "cfg3": 3, "cfg4": 4, "cfg5": 5, "verify70b": 6, "prefill": 0, "cow": -1,
             "spec": -2}
DESCR = {
    1: "tiny paged decode (B4, lens 17/64/100/200, Hq8 Hkv2 d64 bs16, fp16)",
    2: "Llama-3-8B-shaped decode layer (B64, lens U[512,4096], Hq32 Hkv8 d128 bs16, bf16)",
    3: "Llama-3-70B-shaped decode, 80 layer pools (B64, ctx 8192, Hq64 Hkv8 d128 bs16, fp16)",
    4: "shared 1024-token prefix + 5-token causal verify (B128, suffix U[64,512], Hq32 Hkv8 d128 bs16, bf16)",
    5: "long-context split decode (B4, ctx 131072, Hq32 Hkv8 d128 bs32, fp16, 512-token partitions)",
    6: "Llama-3-70B-shaped speculative verify: 64 sequences x 8192 tokens, 4 draft tokens each (q_len 4; Hq64 Hkv8: "
       "32 query rows per KV head, the tensor-core decode kernel), d128 bs16, fp16, one layer pool",
    0: "chunked prefill, Llama-3-70B-shaped: 8 sequences each attending with a 512-token chunk that ends at "
       "context 4608 (the 9th chunk of the prompt), Hq64 Hkv8 d128 bs16, 8 layer pools",
}
PREFILL = dict(batch=8, chunk=512, context=4608, layers=8)
DESCR[-1] = ("copy-on-write block copies in a Llama-3-70B-shaped layer pool (32768 blocks of 16 tokens, Hkv 8, "
             "d 128, fp16): 4096 shared blocks copied to private ones, K and V")
DESCR[-2] = ("speculative rejection sampling: 128 sequences x 5 drafts over a 128256-token vocabulary (fp32 "
             "target and draft distributions, seeded)")
COW = dict(num_blocks=32768, Hkv=8, bs=16, d=128, pairs=4096)
SPEC = dict(B=128, K=5, V=128256)


def make_workload(k: int, layers=None, batch=None) -> synth.Workload:
    """The decode workloads: the five of synth.workload, and the 70B-shaped 4-draft verify (k = 6)."""
    if k == 6:
        return synth.custom_workload([8192] * (batch or 64), 64, 8, 128, 16, 4, synth.FP16, tag=600)
    return synth.workload(k, layers=layers, batch=batch)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# sources that decide a kernel's DRAM traffic: the kernel, its helpers and, where the host picks the
# launch shape (partitions per CTA, row tiles), the entry points
TRAFFIC_SOURCES = {
    "decode": ("decode.cu", "pa_device.cuh", "pa_internal.h", "pa_api.cu"),
    "verify": ("verify.cu", "decode.cu", "pa_device.cuh", "pa_internal.h", "pa_api.cu"),
    "spec": ("spec_verify.cu", "pa_device.cuh", "pa_internal.h"),
    "cow": ("copy_blocks.cu", "pa_device.cuh", "pa_internal.h"),
    "prefill": ("prefill.cu", "pa_device.cuh", "pa_internal.h", "pa_api.cu"),
}


def source_sha(kernel: str = "decode") -> str:
    h = hashlib.sha256()
    for fn in TRAFFIC_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_cache_223_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str = "decode"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "kernel_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == source_sha(kernel):
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------ GPU arm

class GpuWorkload:
    """Every layer's pool filled through pa_cache_write; per-layer inputs resident on the device."""

    def __init__(self, wl: synth.Workload, dev, kv_format: int = 0, shared_prefix: bool = False):
        import torch
        import gpu_harness as H
        import synth.device as sdev
        self.wl = wl
        self.layers = []
        kc0, vc0 = H.alloc_caches(wl, kv_format)
        self.pool = H.make_pool(wl, 0, kc0, vc0, kv_format=kv_format)
        for layer in range(wl.layers):
            kc, vc = (kc0, vc0) if layer == 0 else H.alloc_caches(wl, kv_format)
            H.fill(self.pool, wl, layer, kc, vc, new_only=False)
            lw = synth.with_layer(wl, layer)
            (kind, rows, slots), = lw.write_plan(new_only=True)
            r = torch.from_numpy(rows).to(dev)
            kn, vn = sdev.kv_rows(lw, layer, kind, r, dev)
            q, tables, lens = H.device_inputs(wl, layer)
            self.layers.append(dict(kc=kc, vc=vc, kn=kn, vn=vn, slots=torch.from_numpy(slots).to(dev), q=q,
                                    tables=tables, lens=lens, out=torch.empty_like(q)))
        torch.cuda.synchronize()
        self.shared_prefix = shared_prefix and wl.prefix_tokens > 0
        # pa_decode_shared_prefix: prefix kernel + suffix decode + merge
        self.decode_launches = 3 if self.shared_prefix else self.pool.launches(wl.stride, wl.B, wl.Hq, wl.q_len)

    def decode(self, L):
        wl = self.wl
        if self.shared_prefix:
            self.pool.decode_shared_prefix(L["q"], L["tables"], L["lens"], wl.scale, wl.prefix_tokens, out=L["out"],
                                           k_cache=L["kc"], v_cache=L["vc"])
        else:
            self.pool.decode(L["q"], L["tables"], L["lens"], wl.scale, out=L["out"], k_cache=L["kc"], v_cache=L["vc"])

    def step(self, events=None):
        wl = self.wl
        for i, L in enumerate(self.layers):
            self.pool.cache_write(L["kn"], L["vn"], L["slots"], L["kc"], L["vc"])
            if events is not None:
                events[i][0].record()
            self.decode(L)
            if events is not None:
                events[i][1].record()

    def launches_per_step(self):
        return len(self.layers) * (1 + self.decode_launches)


def reduce_max(value: float, device=None) -> float:
    """Maximum of a per-rank value over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_rank_step: int, steps: int, elapsed_ms: float, world_size: int) -> float:
    """Whole-job GB/s: the bytes all ranks processed over the slowest rank's time."""
    return world_size * bytes_per_rank_step * steps / (elapsed_ms * 1e-3) / 1e9


def step_bytes(wl: synth.Workload, kv_format: int = 0):
    """Algorithmic bytes of one step: per layer, the decode's (q + unique valid K/V + used table entries + lens + out)
    and the cache write's (new k/v read + slot map + the rows written). FP8 pools store d code bytes plus a
    4-byte scale per (token, head) row instead of 2*d bytes."""
    n_new = wl.B * wl.q_len
    row16 = wl.d * 2
    row = wl.d + 4 if kv_format else row16
    dec = wl.algorithmic_bytes() - wl.kv_bytes_unique() + wl.kv_bytes_unique() // row16 * row
    cw = n_new * wl.Hkv * 2 * (row16 + row) + 8 * n_new
    return wl.layers * (dec + cw), dec


def time_decode_steps(G: "GpuWorkload", steps: int, warmup: int, dev, barrier):
    """Warm-up, then `steps` timed steps with CUDA events around the whole region and around each decode call.
    Returns (elapsed ms of the region on this rank, per-call ms list, clock summary)."""
    import torch
    for _ in range(warmup):
        G.step()
    barrier()
    nl = len(G.layers)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nl)]
           for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        time.sleep(0.3)
        barrier()
        start.record()
        for s in range(steps):
            G.step(evs[s])
        stop.record()
        barrier()
    dec_ms = [evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(steps) for i in range(nl)]
    return start.elapsed_time(stop), dec_ms, clk.summary()


def decode_roofline(decode_bytes: int, dec_ms, traffic, kernel: str):
    """Roofline of the decode call: algorithmic bytes over the mean call time (CUDA events on the launching
    stream), against the measured HBM copy rate; median and minimum call times beside the mean."""
    peak, peak_kind = peaks()
    avg = float(np.mean(dec_ms))
    achieved = decode_bytes / (avg * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel,
            "algorithmic_bytes_per_launch": decode_bytes, "avg_launch_ms": round(avg, 5),
            "median_launch_ms": round(float(np.median(dec_ms)), 5), "min_launch_ms": round(float(np.min(dec_ms)), 5),
            "frac_at_median": round(decode_bytes / (float(np.median(dec_ms)) * 1e-3) / 1e9 / peak, 4),
            "peak_kind": peak_kind}


def run_gpu(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    k = WORKLOADS[args.workload]
    wl = make_workload(k, layers=args.layers, batch=args.batch)
    kv_format = 1 if args.kv == "fp8" else 0
    G = GpuWorkload(wl, dev, kv_format, args.shared_prefix)
    total_bytes, decode_bytes = step_bytes(wl, kv_format)
    kv_tokens = int(wl.context_lens.sum()) * wl.layers

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()

    elapsed_ms, dec_ms, clocks = time_decode_steps(G, args.steps, args.warmup, dev, barrier)
    elapsed_ms = reduce_max(elapsed_ms, dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_value(total_bytes, args.steps, elapsed_ms, ws)

    # end to end through the public API: pinned host inputs -> device, kernels, result -> host
    e2e = None if args.no_e2e else run_e2e(G, wl, dev, max(3, args.steps // 5), barrier, kv_format)
    launches = G.launches_per_step() * args.steps
    assert G.pool.check() == 0, "device status flagged during the decode benchmark"

    # the long-context workload (graded beside the 70B-shaped one) in the same run, as a secondary object
    secondary = None
    if args.workload == "cfg3" and not kv_format and not args.no_secondary:
        del G
        torch.cuda.empty_cache()
        wl5 = synth.workload(5)
        G5 = GpuWorkload(wl5, dev, 0, False)
        tb5, db5 = step_bytes(wl5, 0)
        el5, dm5, clk5 = time_decode_steps(G5, args.steps, args.warmup, dev, barrier)
        el5 = reduce_max(el5, dev)
        assert G5.pool.check() == 0, "device status flagged during the long-context benchmark"
        secondary = {
            "workload": f"cfg5: {DESCR[5]}", "config": synth.describe(wl5),
            "value": round(job_value(tb5, args.steps, el5, ws), 2), "unit": "GB/s", "steps": args.steps,
            "ms_per_step": round(el5 / args.steps, 4),
            "kv_tokens_per_s": round(ws * int(wl5.context_lens.sum()) * args.steps / (el5 * 1e-3), 1),
            "roofline": decode_roofline(db5, dm5, measured_traffic("cfg5"),
                                        "pa_decode call (decode kernel + partition merge)"),
            "gpu_launches": G5.launches_per_step() * args.steps, "clocks": clk5,
            "l2": "inputs larger than L2 (no flush)"}

    if rank == 0:
        line = {
            "metric": "paged-attn decode KV GB/s & KV tokens/s on 1 GB300 (fraction of HBM peak)",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("fp16" if wl.dtype == synth.FP16 else "bf16") + ("+fp8-kv" if kv_format else ""),
            "data": "synthetic (seeded, N(0,1)-shaped)",
            "config": {**synth.describe(wl), "workload": f"{args.workload}: {DESCR[k]}",
                       "decode_call": "pa_decode_shared_prefix" if args.shared_prefix and wl.prefix_tokens else "pa_decode",
                       "kv_cache": "fp8 e4m3 + fp32 scale per (slot, head)" if kv_format else "16-bit",
                       "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas{ws}"},
            "kv_tokens_per_s": round(ws * kv_tokens * args.steps / (elapsed_ms * 1e-3), 1),
            "fraction_of_hbm_peak": round(value / peaks()[0], 4),
            "roofline": decode_roofline(
                decode_bytes, dec_ms,
                None if kv_format else measured_traffic(args.workload, "verify" if k == 6 else "decode"),
                "pa_decode_shared_prefix call (prefix kernel + suffix decode + merge)"
                if args.shared_prefix and wl.prefix_tokens else "pa_decode call (decode kernel + partition merge)"),
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if secondary:
            line["secondary"] = secondary
        if ws == 1 and not args.no_cpu_baseline and not kv_format:
            line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_e2e(G: GpuWorkload, wl: synth.Workload, dev, steps: int, barrier, kv_format: int = 0):
    """Same step through the Python binding with per-step inputs copied from pinned host memory and the outputs
    read back, all inside the timed region. A layer's six input tensors travel as one copy (they sit side by
    side, 256-byte aligned, in one pinned host buffer and one device buffer that the calls read through views),
    on a copy stream two layers ahead of the compute, and each layer's output returns on a second copy stream
    while later layers compute (every layer has its own buffers); every step ends with the host holding all of
    that step's outputs."""
    import torch
    names = ("kn", "vn", "slots", "q", "tables", "lens")
    stage = []
    for L in G.layers:
        offs, total = [], 0
        for k in names:
            offs.append(total)
            total += (L[k].numel() * L[k].element_size() + 255) // 256 * 256
        hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
        views = dict(L)
        for k, o in zip(names, offs):
            n = L[k].numel() * L[k].element_size()
            hbuf[o:o + n].copy_(L[k].reshape(-1).view(torch.uint8).cpu())
            views[k] = dbuf[o:o + n].view(L[k].dtype).view(L[k].shape)
        hout = torch.empty(L["out"].shape, dtype=L["out"].dtype).pin_memory()
        stage.append((hbuf, dbuf, views, hout))
    h2d = sum(st[0].numel() for st in stage)   # the staging buffers copied (inputs + alignment padding)
    d2h = sum(st[3].numel() * st[3].element_size() for st in stage)
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in G.layers]
    ev_done = [torch.cuda.Event() for _ in G.layers]
    ahead = 2

    def upload(i):
        with torch.cuda.stream(up):
            stage[i][1].copy_(stage[i][0], non_blocking=True)
            ev_in[i].record(up)

    def one():
        up.wait_stream(main)     # the previous step has been read back (synchronised below); nothing in flight
        n = len(stage)
        for i in range(min(ahead, n)):
            upload(i)
        for i, (hbuf, dbuf, V, hout) in enumerate(stage):
            if i + ahead < n:
                upload(i + ahead)
            main.wait_event(ev_in[i])
            G.pool.cache_write(V["kn"], V["vn"], V["slots"], V["kc"], V["vc"])
            G.decode(V)
            ev_done[i].record(main)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[i])
                hout.copy_(V["out"], non_blocking=True)
        down.synchronize()
        main.synchronize()

    one()
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    barrier()
    dt = (time.perf_counter() - t0) / steps
    total_bytes, _ = step_bytes(wl, kv_format)
    ws = dist_env()[0]
    return {"value": round(ws * total_bytes / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 3), "steps": steps}


# ------------------------------------------------------------------------------------- chunked prefill

def prefill_workload(layer: int, dtype: int, batch: int = PREFILL["batch"]) -> synth.Workload:
    """One layer pool of the prefill workload: every sequence's chunk ends at the same context length; each layer
    has its own seed and block placement."""
    return synth.custom_workload([PREFILL["context"]] * batch, 64, 8, 128, 16, PREFILL["chunk"], dtype,
                                 tag=500 + layer)


def prefill_flops(wl: synth.Workload) -> int:
    """Algorithmic FLOPs of one pa_prefill call: QK^T and PV (2 FLOPs per multiply-add each) over the causal
    (row, key) pairs: chunk row qi of sequence b sees L_b - C + qi + 1 keys."""
    C = wl.q_len
    pairs = sum(C * (int(L) - C) + C * (C + 1) // 2 for L in wl.context_lens)
    return 4 * wl.d * wl.Hq * pairs


def tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (bf16 dense burst; fp16 runs at the same nominal rate)"
    except Exception:
        return 1900.0, "fallback"


class PrefillLayers:
    """Per-layer pools with every token but the chunk written; the step writes the chunk and runs pa_prefill."""

    def __init__(self, layers: int, dtype: int, dev, batch: int):
        import torch
        import gpu_harness as H
        import synth.device as sdev
        self.layers = []
        self.pool = None
        for layer in range(layers):
            wl = prefill_workload(layer, dtype, batch)
            kc, vc = H.alloc_caches(wl)
            if self.pool is None:
                self.pool = H.make_pool(wl, 0, kc, vc)
            H.fill(self.pool, wl, 0, kc, vc, new_only=False)
            (kind, rows, slots), = wl.write_plan(new_only=True)
            kn, vn = sdev.kv_rows(wl, 0, kind, torch.from_numpy(rows).to(dev), dev)
            q, tables, lens = H.device_inputs(wl, 0)
            self.layers.append(dict(wl=wl, kc=kc, vc=vc, kn=kn, vn=vn, slots=torch.from_numpy(slots).to(dev), q=q,
                                    tables=tables, lens=lens, out=torch.empty_like(q)))
        torch.cuda.synchronize()

    def step(self, events=None):
        for i, L in enumerate(self.layers):
            self.pool.cache_write(L["kn"], L["vn"], L["slots"], L["kc"], L["vc"])
            if events is not None:
                events[i][0].record()
            self.pool.prefill(L["q"], L["tables"], L["lens"], L["wl"].scale, out=L["out"], k_cache=L["kc"],
                              v_cache=L["vc"])
            if events is not None:
                events[i][1].record()


def prefill_cpu_baseline(wl: synth.Workload, seconds: float):
    """The oracle on sequence prefixes of layer 0: cache write of the chunk + fp64 paged attention with
    q_len = chunk, as many sequences as fit in about `seconds` (at least one)."""
    import oracle
    done, flops, threads, t_total = 0, 0, 0, 0.0
    while done < wl.B and (done == 0 or t_total < seconds):
        hk, hv, news, q = oracle_sample(wl, done + 1)
        t0 = time.perf_counter()
        kn, vn, sl = news[done]
        oracle.cache_write(hk, hv, kn, vn, sl)
        _, threads = oracle.paged_attention(q[done:done + 1], hk, hv, wl.block_tables[done:done + 1],
                                            wl.context_lens[done:done + 1], wl.dtype, wl.scale)
        t_total += time.perf_counter() - t0
        sub = synth.Workload(**{**wl.__dict__, "B": 1, "context_lens": wl.context_lens[done:done + 1]})
        flops += prefill_flops(sub)
        done += 1
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"layer 0, sequences 0..{done - 1} of the prefill workload: chunk cache write + fp64 paged "
                      f"attention with q_len {wl.q_len} ({flops} algorithmic FLOPs) in {t_total:.2f} s"}


def run_prefill(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dtype = synth.DTYPES[args.dtype]
    batch = args.batch or PREFILL["batch"]
    layers = args.layers or PREFILL["layers"]
    P = PrefillLayers(layers, dtype, dev, batch)
    flops_call = prefill_flops(P.layers[0]["wl"])
    flops_step = flops_call * layers

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        P.step()
    barrier()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(layers)]
           for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        time.sleep(0.3)
        barrier()
        start.record()
        for s in range(args.steps):
            P.step(evs[s])
        stop.record()
        barrier()
    elapsed_ms = reduce_max(start.elapsed_time(stop), dev)
    call_ms = [evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps) for i in range(layers)]
    assert P.pool.check() == 0, "device status flagged during the prefill benchmark"
    e2e = None
    if not args.no_e2e:
        host = []
        for L in P.layers:
            host.append({k: L[k].cpu().pin_memory() for k in ("kn", "vn", "slots", "q", "tables", "lens")})
            host[-1]["out"] = torch.empty(L["out"].shape, dtype=L["out"].dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for hl in host for k, t in hl.items() if k != "out")
        d2h = sum(hl["out"].numel() * hl["out"].element_size() for hl in host)

        def one():
            for L, hl in zip(P.layers, host):
                for k in ("kn", "vn", "slots", "q", "tables", "lens"):
                    L[k].copy_(hl[k], non_blocking=True)
                P.pool.cache_write(L["kn"], L["vn"], L["slots"], L["kc"], L["vc"])
                P.pool.prefill(L["q"], L["tables"], L["lens"], L["wl"].scale, out=L["out"], k_cache=L["kc"],
                               v_cache=L["vc"])
                hl["out"].copy_(L["out"], non_blocking=True)
            torch.cuda.current_stream().synchronize()

        one()
        barrier()
        n = max(3, args.steps // 5)
        t0 = time.perf_counter()
        for _ in range(n):
            one()
        barrier()
        dt = (time.perf_counter() - t0) / n
        e2e = {"value": round(ws * flops_step / dt / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 3), "steps": n}
    if rank == 0:
        peak, peak_kind = tensor_peak()
        call_avg = float(np.mean(call_ms))
        achieved = flops_call / (call_avg * 1e-3) / 1e12
        wl0 = P.layers[0]["wl"]
        line = {
            "metric": "chunked-prefill attention TFLOP/s on 1 GB300 (fraction of dense tensor peak)",
            "value": round(ws * flops_step * args.steps / (elapsed_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.dtype, "data": "synthetic (seeded, N(0,1)-shaped)",
            "config": {**synth.describe(wl0), "workload": f"prefill: {DESCR[0]}", "layers": layers,
                       "l2": "8 layer pools (1.2 GB of K/V) cycle through L2 (no flush)",
                       "parallelism": f"replicas{ws}"},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": measured_traffic("prefill", "prefill"),
                         "kernel": "pa_prefill call (prefill kernel)", "algorithmic_flops_per_launch": flops_call,
                         "avg_launch_ms": round(call_avg, 5), "peak_kind": peak_kind},
            "e2e": e2e,
            "gpu_launches": 2 * layers * args.steps,
            "clocks": clk.summary(),
        }
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = prefill_cpu_baseline(prefill_workload(0, dtype, batch), args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------- CoW copy, spec verify

def _timed(fn, steps: int, warmup: int, dev, events_per_step: bool = True):
    """CUDA-event time of `steps` calls (after `warmup`); returns (elapsed ms, per-call ms list, clocks)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        start.record()
        for i in range(steps):
            evs[i][0].record()
            fn()
            evs[i][1].record()
        stop.record()
        torch.cuda.synchronize()
    return start.elapsed_time(stop), [a.elapsed_time(b) for a, b in evs], clk.summary()


def _timed_graph(fn, steps: int, warmup: int, dev, calls: int = 16):
    """`calls` calls of fn captured once in a CUDA graph (as a serving loop issues them, with no host work
    between launches); CUDA-event time of `steps` replays after `warmup`. Returns (elapsed ms over all
    replays, per-call ms list (one entry per replay), clocks)."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                            # first call outside capture (binding set-up)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    elapsed, per, clocks = _timed(g.replay, steps, warmup, dev)
    return elapsed, [x / calls for x in per], clocks


def cow_pairs():
    """4096 (shared source, private destination) block pairs from a seeded permutation of the pool."""
    perm = synth.permutation(0x5EED0100, synth.make_stream(100, 0, 0), COW["num_blocks"])
    n = COW["pairs"]
    return np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int32)


def run_cow(args):
    import torch
    from paged_kv_cache_223_gb300 import pagedattn as pa
    import synth.device as sdev
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    c = COW
    pool = pa.Pool(c["num_blocks"], c["bs"], c["Hkv"], c["d"], torch.float16, 0, max_seqs=1, max_q_heads=c["Hkv"],
                   max_q_len=1, max_context_len=c["bs"])
    for t in (pool.k_cache, pool.v_cache):
        sdev.fill_word(t, 0x3C00)                       # any defined content: the copy moves raw words
    pairs_h = cow_pairs()
    pairs = torch.from_numpy(pairs_h).to(dev)
    block_bytes = c["Hkv"] * c["bs"] * c["d"] * 2
    nbytes = 2 * len(pairs_h) * 2 * block_bytes          # K and V, read + write
    elapsed, per, clocks = _timed(lambda: pa.copy_blocks(pool, pairs), args.steps, args.warmup, dev)
    assert pool.check() == 0
    # end to end: pairs from pinned host memory, the copy, one destination block read back
    e2e = None
    if not args.no_e2e:
        host_pairs = torch.from_numpy(pairs_h).pin_memory()
        back = torch.empty((c["Hkv"], c["bs"], c["d"]), dtype=torch.float16).pin_memory()
        dst0 = int(pairs_h[0, 1])

        def one():
            pairs.copy_(host_pairs, non_blocking=True)
            pa.copy_blocks(pool, pairs)
            back.copy_(pool.k_cache[dst0], non_blocking=True)
            torch.cuda.current_stream().synchronize()
        one()
        n = max(3, args.steps // 5)
        t0 = time.perf_counter()
        for _ in range(n):
            one()
        dt = (time.perf_counter() - t0) / n
        e2e = {"value": round(nbytes / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": int(pairs_h.nbytes),
               "d2h_bytes_per_step": block_bytes, "ms_per_step": round(dt * 1e3, 3), "steps": n}
    peak, peak_kind = peaks()
    call = float(np.mean(per))
    line = {"metric": "copy-on-write block copy GB/s on 1 GB300 (fraction of HBM peak)",
            "value": round(nbytes * args.steps / (elapsed * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16 words (raw copy)",
            "data": "synthetic", "config": {"workload": "cow: " + DESCR[-1], **c,
                                            "l2": "2 x 512 MB moved per step (no flush)"},
            "roofline": {"bound": "hbm", "achieved": round(nbytes / (call * 1e-3) / 1e9, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(nbytes / (call * 1e-3) / 1e9 / peak, 4),
                         "traffic": measured_traffic("cow", "cow"),
                         "kernel": "pa_copy_blocks call", "algorithmic_bytes_per_launch": nbytes,
                         "avg_launch_ms": round(call, 5), "peak_kind": peak_kind},
            "gpu_launches": args.steps, "clocks": clocks}
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        import oracle
        shape = (c["num_blocks"], c["Hkv"], c["bs"], c["d"])
        hk = np.zeros(shape, dtype=np.uint16)
        hv = np.zeros(shape, dtype=np.uint16)
        t0 = time.perf_counter()
        reps = 0
        while reps == 0 or time.perf_counter() - t0 < min(args.cpu_seconds, 5.0):
            oracle.copy_blocks(hk, hv, pairs_h)
            reps += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(reps * nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": f"{reps} passes over the 4096 pairs in {dt:.2f} s"}
    print(json.dumps(line), flush=True)


def spec_inputs(dev):
    """Seeded target/draft distributions (sharpened uniforms, normalised), drafts drawn from the draft
    distributions by inverse CDF, and the uniforms of the accept tests and of the resample."""
    import torch
    c = SPEC
    g = torch.Generator(device=dev)
    g.manual_seed(0x5EED0200)
    def dist(*shape):
        x = torch.rand(*shape, generator=g, device=dev) ** 3
        return x / x.sum(-1, keepdim=True)
    p = dist(c["B"], c["K"] + 1, c["V"])
    q = dist(c["B"], c["K"], c["V"])
    # mix part of the target into the draft so that some drafts are accepted
    q = 0.5 * q + 0.5 * p[:, :c["K"]]
    q = q / q.sum(-1, keepdim=True)
    r = torch.rand(c["B"], c["K"], 1, generator=g, device=dev, dtype=torch.float64)
    draft = torch.searchsorted(torch.cumsum(q.double(), -1), r * q.double().sum(-1, keepdim=True)).squeeze(-1)
    draft = draft.clamp_(max=c["V"] - 1).to(torch.int32)
    u = torch.rand(c["B"], c["K"], generator=g, device=dev)
    v = torch.rand(c["B"], generator=g, device=dev)
    return p.contiguous(), q.contiguous(), draft.contiguous(), u, v


def spec_bytes(n_out: np.ndarray, K: int, V: int) -> int:
    """Bytes a call must move: per sequence the K draft ids, uniforms and the two probabilities of each accept
    test, the rows of the resample (p and q of the rejected position, or p of the bonus position), v, and the
    K+1 output ids and the count."""
    total = 0
    for n in n_out.tolist():
        kept = n - 1
        tests = min(kept + 1, K)
        rows = 2 if kept < K else 1
        total += 4 * K + 4 * K + 8 * tests + rows * 4 * V + 4 + 4 * (K + 1) + 4
    return total


def run_spec(args):
    import torch
    from paged_kv_cache_223_gb300 import pagedattn as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    c = SPEC
    p, q, draft, u, v = spec_inputs(dev)
    out, n_out = pa.spec_verify(p, q, draft, u, v)
    torch.cuda.synchronize()
    nbytes = spec_bytes(n_out.cpu().numpy(), c["K"], c["V"])
    calls = 16
    elapsed, per, clocks = _timed_graph(lambda: pa.spec_verify(p, q, draft, u, v), args.steps, args.warmup, dev,
                                        calls)
    peak, peak_kind = peaks()
    call = float(np.mean(per))
    e2e = None
    if not args.no_e2e:
        hp, hq, hd, hu, hv = (t.cpu().pin_memory() for t in (p, q, draft, u, v))

        def one():
            for d_, h_ in ((p, hp), (q, hq), (draft, hd), (u, hu), (v, hv)):
                d_.copy_(h_, non_blocking=True)
            o, n = pa.spec_verify(p, q, draft, u, v)
            o.cpu(), n.cpu()
        one()
        ne = max(3, args.steps // 5)
        t0 = time.perf_counter()
        for _ in range(ne):
            one()
        dt = (time.perf_counter() - t0) / ne
        h2d = sum(t.numel() * t.element_size() for t in (hp, hq, hd, hu, hv))
        e2e = {"value": round(nbytes / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": int(out.numel() * 4 + n_out.numel() * 4), "ms_per_step": round(dt * 1e3, 3),
               "steps": ne}
    line = {"metric": "speculative rejection sampling GB/s on 1 GB300 (fraction of HBM peak)",
            "value": round(nbytes * args.steps * calls / (elapsed * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps * calls, "warmup": args.warmup * calls,
            "ms_per_step": round(elapsed / (args.steps * calls), 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 probabilities, f32-pair sums",
            "data": "synthetic (seeded)", "config": {"workload": "spec: " + DESCR[-2], **c,
                                                     "accepted_drafts": int(n_out.sum().item() - c["B"]),
                                                     "timing": f"{calls} calls per CUDA graph replay",
                                                     "l2": "720 MB of distributions (no flush)"},
            "sequences_per_s": round(c["B"] / (call * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(nbytes / (call * 1e-3) / 1e9, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(nbytes / (call * 1e-3) / 1e9 / peak, 4),
                         "traffic": measured_traffic("spec", "spec"),
                         "kernel": "pa_spec_verify call", "algorithmic_bytes_per_launch": nbytes,
                         "avg_launch_ms": round(call, 5), "peak_kind": peak_kind},
            "gpu_launches": args.steps * calls, "clocks": clocks}
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        import oracle
        nb = 16
        args_h = [t[:nb].cpu().numpy() for t in (p, q, draft, u, v)]
        t0 = time.perf_counter()
        reps = 0
        while reps == 0 or time.perf_counter() - t0 < min(args.cpu_seconds, 5.0):
            ref, rn = oracle.spec_verify(*args_h)
            reps += 1
        dt = time.perf_counter() - t0
        b2 = spec_bytes(rn, c["K"], c["V"])
        line["cpu_baseline"] = {"value": round(reps * b2 / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{reps} passes over sequences 0..{nb - 1} ({b2} algorithmic bytes each) "
                                          f"in {dt:.2f} s"}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------- CPU oracle arm

def oracle_sample(wl: synth.Workload, nseq: int):
    """Host inputs for the first nseq sequences of layer 0: pools holding their prompt tokens, new tokens, q."""
    import oracle
    shape = (wl.num_blocks, wl.Hkv, wl.bs, wl.d)
    hk = np.zeros(shape, dtype=np.uint16)
    hv = np.zeros(shape, dtype=np.uint16)
    news = []
    for b in range(nseq):
        L = int(wl.context_lens[b])
        t = np.arange(L - wl.q_len, dtype=np.int64)
        oracle.cache_write(hk, hv, wl.kv_values(0, b, t, "k"), wl.kv_values(0, b, t, "v"), wl.slots(b, t))
        tn = np.arange(L - wl.q_len, L, dtype=np.int64)
        news.append((wl.kv_values(0, b, tn, "k"), wl.kv_values(0, b, tn, "v"), wl.slots(b, tn)))
    q = wl.q_values(0, np.arange(nseq))
    return hk, hv, news, q


def oracle_step(wl, hk, hv, news, q, nseq):
    import oracle
    for kn, vn, sl in news:
        oracle.cache_write(hk, hv, kn, vn, sl)
    _, threads = oracle.paged_attention(q, hk, hv, wl.block_tables, wl.context_lens, wl.dtype, wl.scale,
                                        seqs=np.arange(nseq))
    return threads


def sample_bytes(wl, nseq):
    sub = synth.Workload(**{**wl.__dict__, "B": nseq, "context_lens": wl.context_lens[:nseq],
                            "block_tables": wl.block_tables[:nseq], "layers": 1})
    n_new = nseq * wl.q_len
    return sub.algorithmic_bytes() + 2 * n_new * wl.Hkv * wl.d * 2 * 2 + 8 * n_new, int(sub.context_lens.sum())


def pick_nseq(wl, seconds):
    """Sequences per oracle sample so that one sample takes about `seconds`.

    One sequence is timed first; the oracle spreads (sequence, KV head) items over the host threads."""
    import oracle
    hk, hv, news, q = oracle_sample(wl, 1)
    t0 = time.perf_counter()
    threads1 = oracle_step(wl, hk, hv, news, q, 1)
    t1 = time.perf_counter() - t0
    ncpu = oracle.num_cpus()
    per_item = t1 * threads1 / wl.Hkv                     # seconds of one (sequence, KV head) item on one core
    n = int(seconds * ncpu / max(per_item * wl.Hkv, 1e-9))
    return max(1, min(wl.B, n))


def cpu_baseline(wl: synth.Workload, seconds: float):
    import oracle
    nseq = pick_nseq(wl, seconds)
    hk, hv, news, q = oracle_sample(wl, nseq)
    # whole passes over the sample until the time budget is spent (a pass rewrites the same slots)
    t0 = time.perf_counter()
    reps = 0
    while reps == 0 or time.perf_counter() - t0 < seconds:
        threads = oracle_step(wl, hk, hv, news, q, nseq)
        reps += 1
    dt = time.perf_counter() - t0
    nbytes, toks = sample_bytes(wl, nseq)
    return {"value": round(reps * nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"layer 0, sequences 0..{nseq - 1} of {wl.name}: cache write of the newest tokens + fp64 "
                      f"paged attention ({toks} KV tokens, {nbytes} algorithmic bytes per pass), {reps} passes "
                      f"in {dt:.2f} s",
            "kv_tokens_per_s": round(reps * toks / dt, 1)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    k = WORKLOADS[args.workload]
    if k == 0:
        run_prefill_reference(args)
        return
    if k < 0:
        run_aux_reference(args, k)
        return
    wl = make_workload(k, layers=1)
    nseq = pick_nseq(wl, args.ref_step_seconds)
    hk, hv, news, q = oracle_sample(wl, nseq)
    for _ in range(args.warmup):
        oracle_step(wl, hk, hv, news, q, nseq)
    t0 = time.perf_counter()
    threads = 0
    for _ in range(args.steps):
        threads = oracle_step(wl, hk, hv, news, q, nseq)
    dt = (time.perf_counter() - t0) / args.steps
    nbytes, toks = sample_bytes(wl, nseq)
    value = round(nbytes / dt / 1e9, 4)
    wl_full = make_workload(k, layers=1 if k != 3 else 80)
    line = {"impl": "reference",
            "metric": "paged-attn decode KV GB/s & KV tokens/s on 1 GB300 (fraction of HBM peak)",
            "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded, N(0,1)-shaped)",
            "config": {**synth.describe(wl_full), "workload": f"{args.workload}: {DESCR[k]}"},
            "kv_tokens_per_s": round(toks / dt, 1),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: layer 0, sequences 0..{nseq - 1}: cache write of the newest "
                                       f"tokens + fp64 paged attention ({toks} KV tokens)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill_reference(args):
    """The oracle as the prefill reference arm: each step is one bounded sample of the workload."""
    ws = dist_env()[0]
    wl = prefill_workload(0, synth.DTYPES[args.dtype], args.batch or PREFILL["batch"])
    for _ in range(args.warmup):
        prefill_cpu_baseline(wl, 0.0)
    vals = [prefill_cpu_baseline(wl, args.ref_step_seconds) for _ in range(args.steps)]
    value = round(float(np.mean([v["value"] for v in vals])), 6)
    line = {"impl": "reference",
            "metric": "chunked-prefill attention TFLOP/s on 1 GB300 (fraction of dense tensor peak)",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, N(0,1)-shaped)",
            "config": {**synth.describe(wl), "workload": f"prefill: {DESCR[0]}"},
            "cpu_baseline": {**vals[-1], "value": value},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_aux_reference(args, k: int):
    """The oracle as the reference arm of the copy-on-write and rejection-sampling workloads."""
    import oracle
    if k == -1:
        c = COW
        shape = (c["num_blocks"], c["Hkv"], c["bs"], c["d"])
        hk = np.zeros(shape, dtype=np.uint16)
        hv = np.zeros(shape, dtype=np.uint16)
        pairs = cow_pairs()
        nbytes = 2 * len(pairs) * 2 * c["Hkv"] * c["bs"] * c["d"] * 2
        step = lambda: oracle.copy_blocks(hk, hv, pairs)
        metric, unit, sample = ("copy-on-write block copy GB/s on 1 GB300 (fraction of HBM peak)", "GB/s",
                                "each step: the 4096 block pairs, K and V")
    else:
        import torch
        c = SPEC
        nb = 8
        # the GPU arm's recipe on the host generator; the first nb sequences
        p, q, draft, u, v = (t[:nb].numpy().copy() for t in spec_inputs(torch.device("cpu")))
        _, rn = oracle.spec_verify(p, q, draft, u, v)
        nbytes = spec_bytes(rn, c["K"], c["V"])
        step = lambda: oracle.spec_verify(p, q, draft, u, v)
        metric, unit, sample = ("speculative rejection sampling GB/s on 1 GB300 (fraction of HBM peak)", "GB/s",
                                f"each step: the first {nb} of the {c['B']} sequences (same recipe, host generator)")
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = round(nbytes / dt / 1e9, 4)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": dist_env()[0],
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 / raw words", "data": "synthetic (seeded)",
            "config": {"workload": f"{args.workload}: {DESCR[k]}", **c},
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="cfg3", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kv", default="16bit", choices=["16bit", "fp8"], help="KV cache storage")
    ap.add_argument("--layers", type=int, default=None, help="layer pools (cfg3: default 80; prefill: default 8)")
    ap.add_argument("--batch", type=int, default=None, help="sequences (default: the workload's)")
    ap.add_argument("--dtype", default="fp16", choices=sorted(synth.DTYPES), help="prefill workload dtype")
    ap.add_argument("--no-secondary", action="store_true",
                    help="default workload: skip the long-context workload timed after it in the same run")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="decode workloads with a shared prefix (cfg4) through pa_decode_shared_prefix")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "cow":
        run_cow(args)
    elif args.workload == "spec":
        run_spec(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
