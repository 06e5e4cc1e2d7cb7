"""Shared machinery of the GPU parity tests and the benchmark's checks.

Device side: pool caches filled with a NaN word, then every token written through
pa_cache_write from device-generated rows (synth.device), then pa_decode.
Host side: the fp64 oracle's own chain (cache write -> gather -> attention) on the
same seeded recipe, drawn on the host (synth), for all or a sample of sequences.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np
import torch

import oracle
import synth
import synth.device as sdev
from paged_kv_cache_223_gb300 import pagedattn as pa

TORCH_DT = {synth.FP16: torch.float16, synth.BF16: torch.bfloat16}
ATOL, RTOL = 2e-3, 1e-2          # |gpu - oracle| <= ATOL + RTOL * |oracle|, element-wise
DEV = torch.device("cuda", 0)


def make_pool(wl: synth.Workload, partition_tokens: int = 0, k_cache=None, v_cache=None,
              max_context_len: Optional[int] = None, kv_format: int = pa.PA_KV_16BIT) -> pa.Pool:
    return pa.Pool(wl.num_blocks, wl.bs, wl.Hkv, wl.d, TORCH_DT[wl.dtype], 0,
                   partition_tokens=partition_tokens or wl.partition_tokens, max_seqs=wl.B, max_q_heads=wl.Hq,
                   max_q_len=min(wl.q_len, 8), max_context_len=max_context_len or wl.stride * wl.bs,
                   k_cache=k_cache, v_cache=v_cache, kv_format=kv_format)


FP8_NAN_CODE = 0x7F


def alloc_caches(wl: synth.Workload, kv_format: int = pa.PA_KV_16BIT) -> Tuple[torch.Tensor, torch.Tensor]:
    """Caches filled with NaN sentinels (16-bit: the NaN word; FP8: the NaN code and NaN scales)."""
    if kv_format == pa.PA_KV_FP8_E4M3:
        codes = wl.num_blocks * wl.Hkv * wl.bs * wl.d
        out = []
        for _ in range(2):
            buf = torch.empty(codes + 4 * wl.num_blocks * wl.Hkv * wl.bs, dtype=torch.uint8, device=DEV)
            buf[:codes].fill_(FP8_NAN_CODE)
            buf[codes:].view(torch.int32).fill_(0x7FC00000)
            out.append(buf)
        return out[0], out[1]
    shape = (wl.num_blocks, wl.Hkv, wl.bs, wl.d)
    kc = torch.empty(shape, dtype=TORCH_DT[wl.dtype], device=DEV)
    vc = torch.empty_like(kc)
    sdev.fill_word(kc, synth.NAN16[wl.dtype])
    sdev.fill_word(vc, synth.NAN16[wl.dtype])
    return kc, vc


def fill(pool: pa.Pool, wl: synth.Workload, layer: int, kc, vc, new_only: bool, chunk: int = 1 << 18) -> int:
    """Write the workload's tokens (all but the newest, or only the newest) through pa_cache_write.
    Returns the number of pa_cache_write calls."""
    wl = synth.with_layer(wl, layer)
    calls = 0
    for kind, rows, slots in wl.write_plan(new_only):
        for i in range(0, len(rows), chunk):
            r = torch.from_numpy(np.ascontiguousarray(rows[i:i + chunk])).to(DEV)
            k, v = sdev.kv_rows(wl, layer, kind, r, DEV)
            s = torch.from_numpy(np.ascontiguousarray(slots[i:i + chunk], dtype=np.int64)).to(DEV)
            pool.cache_write(k, v, s, kc, vc)
            calls += 1
    return calls


def device_inputs(wl: synth.Workload, layer: int):
    wl = synth.with_layer(wl, layer)
    q = sdev.q_tensor(wl, layer, DEV)
    tables = torch.from_numpy(np.ascontiguousarray(wl.block_tables)).to(DEV)
    lens = torch.from_numpy(np.ascontiguousarray(wl.context_lens, dtype=np.int32)).to(DEV)
    return q, tables, lens


def build_device(wl: synth.Workload, layer: int = 0, partition_tokens: int = 0, kv_format: int = pa.PA_KV_16BIT):
    """Pool + caches filled through pa_cache_write (fill, then the newest tokens) + q/tables/lens."""
    kc, vc = alloc_caches(wl, kv_format)
    pool = make_pool(wl, partition_tokens, kc, vc, kv_format=kv_format)
    fill(pool, wl, layer, kc, vc, new_only=False)
    fill(pool, wl, layer, kc, vc, new_only=True)
    q, tables, lens = device_inputs(wl, layer)
    return pool, kc, vc, q, tables, lens


def oracle_reference(wl: synth.Workload, layer: int, seqs: Optional[Sequence[int]] = None,
                     full_pool: bool = False, num_threads: int = 0):
    """The oracle chain for sequences `seqs` (default: all). Returns (out float64, host K pool, host V pool).

    full_pool=True starts from NaN words everywhere (so the whole pool can be compared bit for bit);
    otherwise the host pool starts as zeros and only the listed sequences' slots are written."""
    wl = synth.with_layer(wl, layer)
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    shape = (wl.num_blocks, wl.Hkv, wl.bs, wl.d)
    if full_pool:
        hk = np.full(shape, synth.NAN16[wl.dtype], dtype=np.uint16)
    else:
        hk = np.zeros(shape, dtype=np.uint16)
    hv = hk.copy() if full_pool else np.zeros(shape, dtype=np.uint16)
    for b in seqs:
        t = np.arange(int(wl.context_lens[b]), dtype=np.int64)
        oracle.cache_write(hk, hv, wl.kv_values(layer, b, t, "k"), wl.kv_values(layer, b, t, "v"), wl.slots(b, t))
    q = wl.q_values(layer, np.array(seqs))
    out, _ = oracle.paged_attention(q, hk, hv, wl.block_tables, wl.context_lens, wl.dtype, wl.scale,
                                    seqs=np.array(seqs), num_threads=num_threads)
    return out, hk, hv


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def compare(gpu: torch.Tensor, ref: np.ndarray):
    """(max abs err, max rel err, #violations of ATOL + RTOL*|ref|)."""
    g = to_f64(gpu)
    err = np.abs(g - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    rel = err / np.maximum(np.abs(ref), 1e-30)
    return float(err.max()), float(rel.max()), int(bad.sum())


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    mx, mr, nbad = compare(gpu, ref)
    assert nbad == 0, f"{what}: {nbad} elements outside {ATOL} + {RTOL}*|ref| (max abs {mx:.3g}, max rel {mr:.3g})"
    return mx, mr


def pool_words(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_pool_blocks(wl: synth.Workload, layer: int, kc, vc, hk, hv, seqs: Sequence[int]):
    """Valid slots of the listed sequences equal the oracle's words; slots past each context hold the NaN word."""
    wl = synth.with_layer(wl, layer)
    nanw = synth.NAN16[wl.dtype]
    for b in seqs:
        L = int(wl.context_lens[b])
        nb = -(-L // wl.bs)
        ids = torch.from_numpy(wl.block_tables[b, :nb].astype(np.int64)).to(DEV)
        for dev_pool, host_pool in ((kc, hk), (vc, hv)):
            got = pool_words(dev_pool.index_select(0, ids))            # [nb, Hkv, bs, d]
            exp = host_pool[wl.block_tables[b, :nb]]
            got_t = got.transpose(0, 2, 1, 3).reshape(nb * wl.bs, wl.Hkv, wl.d)
            exp_t = exp.transpose(0, 2, 1, 3).reshape(nb * wl.bs, wl.Hkv, wl.d)
            assert np.array_equal(got_t[:L], exp_t[:L]), f"seq {b}: cache words differ"
            assert (got_t[L:] == nanw).all(), f"seq {b}: slots past the context were written"


def oracle_reference_fp8(wl: synth.Workload, layer: int, seqs: Optional[Sequence[int]] = None):
    """The oracle's FP8 chain (quantising cache write -> gather -> dequantise -> attention) for `seqs`.
    Returns (out float64, host K buffer, host V buffer) in the pool's FP8 layout."""
    wl = synth.with_layer(wl, layer)
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    geo = (wl.num_blocks, wl.Hkv, wl.bs, wl.d)
    hk = oracle.fp8_pool(*geo)
    hv = oracle.fp8_pool(*geo)
    for b in seqs:
        t = np.arange(int(wl.context_lens[b]), dtype=np.int64)
        oracle.cache_write_fp8(hk, hv, geo, wl.kv_values(layer, b, t, "k"), wl.kv_values(layer, b, t, "v"),
                               wl.slots(b, t), wl.dtype)
    q = wl.q_values(layer, np.array(seqs))
    out = oracle.paged_attention_fp8(q, hk, hv, geo, wl.block_tables, wl.context_lens, wl.dtype, wl.scale,
                                     seqs=np.array(seqs))
    return out, hk, hv


def check_fp8_pool_rows(wl: synth.Workload, layer: int, kc, vc, hk, hv, seqs: Sequence[int]):
    """Codes and scales of the listed sequences' valid slots equal the oracle's, bit for bit."""
    wl = synth.with_layer(wl, layer)
    geo = (wl.num_blocks, wl.Hkv, wl.bs, wl.d)
    for dev_buf, host_buf in ((kc, hk), (vc, hv)):
        dc, ds = oracle.fp8_views(dev_buf.cpu().numpy(), *geo)
        hc, hs = oracle.fp8_views(host_buf, *geo)
        for b in seqs:
            t = np.arange(int(wl.context_lens[b]))
            pb, off = wl.block_tables[b, t // wl.bs], t % wl.bs
            assert np.array_equal(dc[pb, :, off], hc[pb, :, off]), f"seq {b}: codes differ"
            assert np.array_equal(ds[pb, :, off].view(np.uint32), hs[pb, :, off].view(np.uint32)), f"seq {b}: scales"
