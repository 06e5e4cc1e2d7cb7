"""Device-side generation of the synth recipe (libpasynth.so), for workloads of many GB.

Produces the same 16-bit words as synth.values16 for the same (seed, stream, counter).
Test and benchmark infrastructure only.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Optional

import torch

from . import FP16, NAN16, Workload, K_Q

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpasynth.so")
_lock = threading.Lock()
_lib = None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} missing (run `python -m paged_kv_cache_223_gb300._build`)")
            L = C.CDLL(LIB_PATH)
            L.synth_fill_rows.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_uint64, C.c_uint64,
                                          C.c_int, C.c_float, C.c_float, C.c_void_p]
            L.synth_fill_rows.restype = C.c_int
            L.synth_fill_word.argtypes = [C.c_void_p, C.c_int64, C.c_uint16, C.c_void_p]
            L.synth_fill_word.restype = C.c_int
            L.synth_stream_base.argtypes = [C.c_uint64, C.c_uint64]
            L.synth_stream_base.restype = C.c_uint64
            _lib = L
    return _lib


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def fill_rows(dst: torch.Tensor, rows: Optional[torch.Tensor], row_len: int, seed: int, stream: int, dtype: int,
              sigma: float = 1.0, mean: float = 0.0) -> None:
    """dst (16-bit, contiguous) viewed as [nrows, row_len]: row r gets counters rows[r]*row_len + c."""
    assert dst.is_cuda and dst.is_contiguous() and dst.element_size() == 2
    nrows = dst.numel() // row_len
    if rows is not None:
        assert rows.dtype == torch.int64 and rows.is_cuda and rows.numel() == nrows
    rc = lib().synth_fill_rows(dst.data_ptr(), None if rows is None else rows.data_ptr(), nrows, row_len,
                               seed & ((1 << 64) - 1), stream & ((1 << 64) - 1), dtype, sigma, mean, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_fill_rows failed with CUDA error {rc}")


def fill_word(dst: torch.Tensor, word: int) -> None:
    assert dst.is_cuda and dst.is_contiguous() and dst.element_size() == 2
    rc = lib().synth_fill_word(dst.data_ptr(), dst.numel(), word, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_fill_word failed with CUDA error {rc}")


def q_tensor(wl: Workload, layer: int, device) -> torch.Tensor:
    tdt = torch.float16 if wl.dtype == FP16 else torch.bfloat16
    q = torch.empty((wl.B, wl.q_len, wl.Hq, wl.d), dtype=tdt, device=device)
    fill_rows(q, None, q.numel(), wl.seed, wl.stream(layer, K_Q), wl.dtype, wl.q_sigma, 0.0)
    return q


def kv_rows(wl: Workload, layer: int, kind_k: int, rows: torch.Tensor, device):
    """k, v [len(rows), Hkv, d] for counter rows of the K stream `kind_k` (and its V partner)."""
    tdt = torch.float16 if wl.dtype == FP16 else torch.bfloat16
    n = rows.numel()
    k = torch.empty((n, wl.Hkv, wl.d), dtype=tdt, device=device)
    v = torch.empty_like(k)
    HD = wl.Hkv * wl.d
    fill_rows(k, rows, HD, wl.seed, wl.stream(layer, kind_k), wl.dtype, 1.0, 0.0)
    fill_rows(v, rows, HD, wl.seed, wl.stream(layer, kind_k + 1), wl.dtype, 1.0, wl.v_mean)
    return k, v


def nan_word(wl: Workload) -> int:
    return NAN16[wl.dtype]
