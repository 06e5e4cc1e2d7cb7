"""ctypes binding of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg. The product path (the CUDA library and its Python
binding) never imports this package.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_libs = {}

OK, ERR_ARG, ERR_BOUNDS, ERR_OOM = 0, 1, 2, 3
FP16, BF16 = 0, 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile oracle.c with gcc (plain C11, fp contraction off so both hosts agree)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


_active = threading.local()


def use(path: Optional[str]):
    """Route this thread's oracle calls to the library at `path` (None: the built-in one)."""
    _active.path = path


def lib():
    path = getattr(_active, "path", None) or _LIB
    with _lock:
        if path not in _libs:
            if path == _LIB:
                build()
            L = C.CDLL(path)
            P = C.c_void_p
            L.oracle_f16_to_double.argtypes = [C.c_uint16]
            L.oracle_f16_to_double.restype = C.c_double
            L.oracle_bf16_to_double.argtypes = [C.c_uint16]
            L.oracle_bf16_to_double.restype = C.c_double
            L.oracle_cache_write.argtypes = [P, P, P, P, P, C.c_int64, C.c_int64, C.c_int, C.c_int, C.c_int]
            L.oracle_gather.argtypes = [P, P, C.c_int64, C.c_int64, C.c_int, C.c_int, C.c_int, P]
            L.oracle_copy_blocks.argtypes = [P, P, P, C.c_int64, C.c_int64, C.c_int, C.c_int, C.c_int]
            L.oracle_attention.argtypes = [P, P, P, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                           C.c_float, P, P]
            L.oracle_paged_attention.argtypes = [P, P, P, P, C.c_int64, P, P, C.c_int, C.c_int64, C.c_int,
                                                 C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float, P,
                                                 C.c_int, P]
            L.oracle_attention_partitions.argtypes = [P, P, P, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_int,
                                                      C.c_int, C.c_float, C.c_int64, P, P, P]
            L.oracle_lse_merge.argtypes = [C.c_int64, P, P, P, C.c_int, P]
            L.oracle_spec_verify.argtypes = [P, P, P, P, P, C.c_int64, C.c_int, C.c_int64, P, P]
            L.oracle_e4m3_to_double.argtypes = [C.c_uint8]
            L.oracle_e4m3_to_double.restype = C.c_double
            L.oracle_f32_to_e4m3.argtypes = [C.c_float]
            L.oracle_f32_to_e4m3.restype = C.c_uint8
            L.oracle_cache_write_fp8.argtypes = [P, P, P, P, P, C.c_int64, C.c_int64, C.c_int, C.c_int, C.c_int, C.c_int]
            L.oracle_cache_write_fp8.restype = C.c_int
            L.oracle_paged_attention_fp8.argtypes = [P, P, P, P, C.c_int64, P, P, C.c_int, C.c_int64, C.c_int, C.c_int,
                                                     C.c_int, C.c_int, C.c_int, C.c_int, C.c_float, P]
            L.oracle_paged_attention_fp8.restype = C.c_int
            L.oracle_num_cpus.argtypes = []
            for f in ("oracle_cache_write", "oracle_gather", "oracle_copy_blocks", "oracle_attention", "oracle_paged_attention",
                      "oracle_attention_partitions", "oracle_lse_merge", "oracle_num_cpus", "oracle_spec_verify"):
                getattr(L, f).restype = C.c_int
            _libs[path] = L
    return _libs[path]


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def _check(rc: int, what: str):
    if rc != OK:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def f16_to_double(w: int) -> float:
    return lib().oracle_f16_to_double(w)


def bf16_to_double(w: int) -> float:
    return lib().oracle_bf16_to_double(w)


def decode16(words: np.ndarray, dtype: int) -> np.ndarray:
    """Element-wise exact decode of 16-bit words (slow; for small arrays)."""
    f = bf16_to_double if dtype == BF16 else f16_to_double
    flat = np.asarray(words, dtype=np.uint16).ravel()
    return np.array([f(int(w)) for w in flat], dtype=np.float64).reshape(np.shape(words))


def cache_write(k_pool: np.ndarray, v_pool: np.ndarray, k: np.ndarray, v: np.ndarray,
                slot_mapping: np.ndarray) -> None:
    """In-place scatter of k, v [N, Hkv, d] into pools [NB, Hkv, bs, d] (uint16 words)."""
    NB, Hkv, bs, d = k_pool.shape
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    k, v = _u16(k), _u16(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    _check(lib().oracle_cache_write(_p(k_pool), _p(v_pool), _p(k), _p(v), _p(sm), len(sm), NB, bs, Hkv, d),
           "cache_write")


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs) -> None:
    """In-place copy of block pairs (src, dst) in both pools."""
    NB, Hkv, bs, d = k_pool.shape
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    _check(lib().oracle_copy_blocks(_p(k_pool), _p(v_pool), _p(pr), len(pr), NB, bs, Hkv, d), "copy_blocks")


def gather(pool: np.ndarray, table_row: np.ndarray, L: int) -> np.ndarray:
    NB, Hkv, bs, d = pool.shape
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    out = np.empty((L, Hkv, d), dtype=np.uint16)
    _check(lib().oracle_gather(_p(np.ascontiguousarray(pool)), _p(row), L, NB, bs, Hkv, d, _p(out)), "gather")
    return out


def attention(q: np.ndarray, kc: np.ndarray, vc: np.ndarray, dtype: int, scale: float,
              want_weights: bool = False):
    """q [q_len, Hq, d], kc/vc [L, Hkv, d] (words) -> out [q_len, Hq, d] float64 (and weights)."""
    q, kc, vc = _u16(q), _u16(kc), _u16(vc)
    q_len, Hq, d = q.shape
    L, Hkv, _ = kc.shape
    out = np.empty((q_len, Hq, d), dtype=np.float64)
    w = np.empty((q_len, Hq, L), dtype=np.float64) if want_weights else None
    _check(lib().oracle_attention(_p(q), _p(kc), _p(vc), L, q_len, Hq, Hkv, d, dtype, scale, _p(out), _p(w)),
           "attention")
    return (out, w) if want_weights else out


def paged_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, block_tables: np.ndarray,
                    context_lens: np.ndarray, dtype: int, scale: float, seqs: Optional[np.ndarray] = None,
                    num_threads: int = 0) -> Tuple[np.ndarray, int]:
    """q: one [q_len, Hq, d] row per computed sequence (all, or those in `seqs`, in order).

    Returns (out float64 [n, q_len, Hq, d], threads used)."""
    q = _u16(q)
    n, q_len, Hq, d = q.shape
    NB, Hkv, bs, _ = k_pool.shape
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    sq = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
    assert n == (len(lens) if sq is None else len(sq))
    out = np.empty((n, q_len, Hq, d), dtype=np.float64)
    used = C.c_int(0)
    _check(lib().oracle_paged_attention(_p(q), _p(np.ascontiguousarray(k_pool)), _p(np.ascontiguousarray(v_pool)),
                                        _p(tables), tables.shape[1], _p(lens), _p(sq), n, NB, bs, q_len, Hq,
                                        Hkv, d, dtype, scale, _p(out), num_threads, C.byref(used)),
           "paged_attention")
    return out, used.value


def attention_partitions(q, kc, vc, dtype: int, scale: float, P: int):
    q, kc, vc = _u16(q), _u16(kc), _u16(vc)
    q_len, Hq, d = q.shape
    L, Hkv, _ = kc.shape
    np_ = -(-L // P)
    m = np.empty((q_len, Hq, np_)); l = np.empty((q_len, Hq, np_)); o = np.empty((q_len, Hq, np_, d))
    _check(lib().oracle_attention_partitions(_p(q), _p(kc), _p(vc), L, q_len, Hq, Hkv, d, dtype, scale, P,
                                             _p(m), _p(l), _p(o)), "attention_partitions")
    return m, l, o


def lse_merge(m: np.ndarray, l: np.ndarray, o: np.ndarray) -> np.ndarray:
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    np_, d = o.shape
    out = np.empty(d)
    _check(lib().oracle_lse_merge(np_, _p(m), _p(l), _p(o), d, _p(out)), "lse_merge")
    return out


def num_cpus() -> int:
    return lib().oracle_num_cpus()


def spec_verify(p: np.ndarray, q: np.ndarray, draft: np.ndarray, u: np.ndarray, v: np.ndarray):
    """Speculative rejection sampling. p [B, K+1, V], q [B, K, V] fp32; draft int32 [B, K]; u fp32 [B, K];
    v fp32 [B]. Returns (out int32 [B, K+1], n_out int32 [B])."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    B, K1, V = p.shape
    out = np.empty((B, K1), dtype=np.int32)
    n = np.empty(B, dtype=np.int32)
    _check(lib().oracle_spec_verify(_p(p), _p(q), _p(draft), _p(u), _p(v), B, K1 - 1, V, _p(out), _p(n)),
           "spec_verify")
    return out, n


# ------------------------------------------------------------------------------ FP8 KV

def e4m3_to_double(c: int) -> float:
    return lib().oracle_e4m3_to_double(c)


def f32_to_e4m3(x: float) -> int:
    return lib().oracle_f32_to_e4m3(x)


def fp8_pool(num_blocks: int, Hkv: int, bs: int, d: int, fill_code: int = 0) -> np.ndarray:
    """An FP8 pool buffer: codes [NB, Hkv, bs, d] then float32 scales [NB, Hkv, bs], as one byte array."""
    codes = num_blocks * Hkv * bs * d
    buf = np.zeros(codes + 4 * num_blocks * Hkv * bs, dtype=np.uint8)
    buf[:codes] = fill_code
    return buf


def fp8_views(buf: np.ndarray, num_blocks: int, Hkv: int, bs: int, d: int):
    codes = num_blocks * Hkv * bs * d
    return buf[:codes].reshape(num_blocks, Hkv, bs, d), buf[codes:].view(np.float32).reshape(num_blocks, Hkv, bs)


def cache_write_fp8(k_buf: np.ndarray, v_buf: np.ndarray, geometry, k: np.ndarray, v: np.ndarray,
                    slot_mapping: np.ndarray, dtype: int) -> None:
    NB, Hkv, bs, d = geometry
    k, v = _u16(k), _u16(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    _check(lib().oracle_cache_write_fp8(_p(k_buf), _p(v_buf), _p(k), _p(v), _p(sm), len(sm), NB, bs, Hkv, d, dtype),
           "cache_write_fp8")


def paged_attention_fp8(q: np.ndarray, k_buf: np.ndarray, v_buf: np.ndarray, geometry, block_tables: np.ndarray,
                        context_lens: np.ndarray, dtype: int, scale: float, seqs=None) -> np.ndarray:
    NB, Hkv, bs, d = geometry
    q = _u16(q)
    n, q_len, Hq, _ = q.shape
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    sq = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
    out = np.empty((n, q_len, Hq, d), dtype=np.float64)
    _check(lib().oracle_paged_attention_fp8(_p(q), _p(k_buf), _p(v_buf), _p(tables), tables.shape[1], _p(lens), _p(sq),
                                            n, NB, bs, q_len, Hq, Hkv, d, dtype, scale, _p(out)),
           "paged_attention_fp8")
    return out
