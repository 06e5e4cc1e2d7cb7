#!/usr/bin/env python3
"""Paged-attention decode benchmark on GB300 (one JSON line on rank 0).

A step is one pass of the hot path over one batch: for every layer pool, the cache write
of the newest tokens (pa_cache_write) and the paged decode (pa_decode: decode kernel plus
the partition merge). Default workload: Llama-3-70B-shaped decode, 64 sequences x 8192
tokens, Hq 64 / Hkv 8 / d 128, block size 16, fp16, 80 independent layer pools (172 GB of
KV, far larger than L2, so no flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload cfg3|cfg5|cfg2|cfg4|cfg1]
    python bench.py --impl reference      # the fp64 CPU oracle as the reference arm
    python bench.py --workload prefill    # chunked prefill (pa_prefill), tensor-core bound: TFLOP/s

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

WORKLOADS = {"cfg1": 1, "cfg2": 2, "cfg3": 3, "cfg4": 4, "cfg5": 5, "prefill": 0}
DESCR = {
    1: "tiny paged decode (B4, lens 17/64/100/200, Hq8 Hkv2 d64 bs16, fp16)",
    2: "Llama-3-8B-shaped decode layer (B64, lens U[512,4096], Hq32 Hkv8 d128 bs16, bf16)",
    3: "Llama-3-70B-shaped decode, 80 layer pools (B64, ctx 8192, Hq64 Hkv8 d128 bs16, fp16)",
    4: "shared 1024-token prefix + 5-token causal verify (B128, suffix U[64,512], Hq32 Hkv8 d128 bs16, bf16)",
    5: "long-context split decode (B4, ctx 131072, Hq32 Hkv8 d128 bs32, fp16, 512-token partitions)",
    0: "chunked prefill, Llama-3-70B-shaped: 8 sequences each attending with a 512-token chunk that ends at "
       "context 4608 (the 9th chunk of the prompt), Hq64 Hkv8 d128 bs16, 8 layer pools",
}
PREFILL = dict(batch=8, chunk=512, context=4608, layers=8)


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


def decode_source_sha() -> str:
    h = hashlib.sha256()
    for fn in ("decode.cu", "pa_device.cuh", "pa_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_223_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == decode_source_sha():
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


def run_gpu(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    k = WORKLOADS[args.workload]
    wl = synth.workload(k, layers=args.layers, batch=args.batch)
    kv_format = 1 if args.kv == "fp8" else 0
    G = GpuWorkload(wl, dev, kv_format, args.shared_prefix)
    total_bytes, decode_bytes = step_bytes(wl, kv_format)
    kv_tokens = int(wl.context_lens.sum()) * wl.layers

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        G.step()
    barrier()
    nl = len(G.layers)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nl)]
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
            G.step(evs[s])
        stop.record()
        barrier()
    elapsed_ms = start.elapsed_time(stop)
    dec_ms = [evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps) for i in range(nl)]
    elapsed_ms = reduce_max(elapsed_ms, dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_value(total_bytes, args.steps, elapsed_ms, ws)

    # end to end through the public API: pinned host inputs -> device, kernels, result -> host
    e2e = None if args.no_e2e else run_e2e(G, wl, dev, max(3, args.steps // 5), barrier, kv_format)

    if rank == 0:
        peak, peak_kind = peaks()
        dec_avg_ms = float(np.mean(dec_ms))
        achieved = decode_bytes / (dec_avg_ms * 1e-3) / 1e9
        line = {
            "metric": "paged-attn decode KV GB/s & KV tokens/s on 1 GB300 (fraction of HBM peak)",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("fp16" if wl.dtype == synth.FP16 else "bf16") + ("+fp8-kv" if kv_format else ""),
            "data": "synthetic (seeded, N(0,1)-shaped)",
            "config": {**synth.describe(wl), "workload": f"{args.workload}: {DESCR[k]}",
                       "decode_call": "pa_decode_shared_prefix" if G.shared_prefix else "pa_decode",
                       "kv_cache": "fp8 e4m3 + fp32 scale per (slot, head)" if kv_format else "16-bit",
                       "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas{ws}"},
            "kv_tokens_per_s": round(ws * kv_tokens * args.steps / (elapsed_ms * 1e-3), 1),
            "fraction_of_hbm_peak": round(value / peak, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": None if kv_format else measured_traffic(args.workload),
                         "kernel": ("pa_decode_shared_prefix call (prefix kernel + suffix decode + merge)"
                                    if G.shared_prefix else "pa_decode call (decode kernel + partition merge)"),
                         "algorithmic_bytes_per_launch": decode_bytes, "avg_launch_ms": round(dec_avg_ms, 5),
                         "peak_kind": peak_kind},
            "e2e": e2e,
            "gpu_launches": G.launches_per_step() * args.steps,
            "clocks": clk.summary(),
        }
        if ws == 1 and not args.no_cpu_baseline and not kv_format:
            line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_e2e(G: GpuWorkload, wl: synth.Workload, dev, steps: int, barrier, kv_format: int = 0):
    """Same step through the Python binding with per-step inputs copied from pinned host memory and the outputs
    read back, all inside the timed region."""
    import torch
    host = []
    for L in G.layers:
        host.append({k: L[k].cpu().pin_memory() for k in ("kn", "vn", "slots", "q", "tables", "lens")})
        host[-1]["out"] = torch.empty(L["out"].shape, dtype=L["out"].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for hl in host for k, t in hl.items() if k != "out")
    d2h = sum(hl["out"].numel() * hl["out"].element_size() for hl in host)

    def one():
        for L, hl in zip(G.layers, host):
            for k in ("kn", "vn", "slots", "q", "tables", "lens"):
                L[k].copy_(hl[k], non_blocking=True)
            G.pool.cache_write(L["kn"], L["vn"], L["slots"], L["kc"], L["vc"])
            G.decode(L)
            hl["out"].copy_(L["out"], non_blocking=True)
        torch.cuda.current_stream().synchronize()

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
                         "frac": round(achieved / peak, 4), "traffic": None,
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
    t0 = time.perf_counter()
    threads = oracle_step(wl, hk, hv, news, q, nseq)
    dt = time.perf_counter() - t0
    nbytes, toks = sample_bytes(wl, nseq)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"layer 0, sequences 0..{nseq - 1} of {wl.name}: cache write of the newest tokens + fp64 "
                      f"paged attention ({toks} KV tokens, {nbytes} algorithmic bytes) in {dt:.2f} s",
            "kv_tokens_per_s": round(toks / dt, 1)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    k = WORKLOADS[args.workload]
    if k == 0:
        run_prefill_reference(args)
        return
    wl = synth.workload(k, layers=1)
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
    wl_full = synth.workload(k, layers=1 if k != 3 else 80)
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
    ap.add_argument("--shared-prefix", action="store_true",
                    help="decode workloads with a shared prefix (cfg4) through pa_decode_shared_prefix")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill":
        run_prefill(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
