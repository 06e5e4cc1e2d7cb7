"""Python binding of the C ABI in include/pagedattn.h (ctypes; argument marshalling only).

Torch tensors provide device memory and streams; every step of the paged-attention path
runs in the CUDA library. There is no fallback: if the library is missing this module
raises on load.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpagedattn.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_OOM, PA_ERR_DEVICE_BOUNDS, PA_ERR_TIMEOUT = range(7)
PA_FP16, PA_BF16 = 0, 1
PA_KV_16BIT, PA_KV_FP8_E4M3 = 0, 1
_TORCH_DTYPE = {PA_FP16: torch.float16, PA_BF16: torch.bfloat16}
_PA_DTYPE = {torch.float16: PA_FP16, torch.bfloat16: PA_BF16}


class PaPoolConfig(C.Structure):
    _fields_ = [("num_blocks", C.c_int32), ("block_size", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("dtype", C.c_int32), ("device", C.c_int32),
                ("partition_tokens", C.c_int32), ("max_seqs", C.c_int32), ("max_q_heads", C.c_int32),
                ("max_q_len", C.c_int32), ("max_context_len", C.c_int32), ("k_cache", C.c_void_p),
                ("v_cache", C.c_void_p), ("kv_format", C.c_int32)]


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib() -> C.CDLL:
    """Load libpagedattn.so (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                                   "(run `python -m paged_kv_cache_223_gb300._build`)")
            L = C.CDLL(LIB_PATH)
            P, I32, I64 = C.c_void_p, C.c_int32, C.c_int64
            L.pa_pool_create.argtypes = [C.POINTER(PaPoolConfig), C.POINTER(C.c_void_p)]
            L.pa_destroy.argtypes = [P]
            L.pa_destroy.restype = None
            L.pa_pool_caches.argtypes = [P, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.POINTER(C.c_uint64)]
            L.pa_cache_write.argtypes = [P, P, P, P, I32, P, P, P]
            L.pa_decode.argtypes = [P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P]
            L.pa_prefill.argtypes = [P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, P, P]
            L.pa_decode_shared_prefix.argtypes = [P, P, P, P, P, I32, P, I32, I32, I32, C.c_float, I32, P, P]
            L.pa_pool_check.argtypes = [P, P]
            L.pa_pool_selftest_wait.argtypes = [P, C.c_uint64, P]
            L.pa_pool_selftest_wait.restype = C.c_int
            L.pa_decode_launches.argtypes = [P, I32, I32, I32, I32]
            L.pa_decode_launches.restype = I32
            L.pa_status_string.argtypes = [C.c_int]
            L.pa_status_string.restype = C.c_char_p
            for f in ("pa_pool_create", "pa_pool_caches", "pa_cache_write", "pa_decode", "pa_prefill", "pa_decode_shared_prefix",
                      "pa_pool_check"):
                getattr(L, f).restype = C.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    """The CUDA stream handle: the given stream's, else the current device's current stream (read as a raw
    handle where torch offers it: building a torch Stream object costs about 3 us per call)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev(t: torch.Tensor, name: str, dtype: Optional[torch.dtype] = None) -> torch.Tensor:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


class Pool:
    """One paged KV pool (pa_pool_create) with its caches.

    The caches are torch tensors, created here unless given; the pool only borrows them.
    16-bit pools: [num_blocks, num_kv_heads, block_size, head_dim] of the model dtype.
    FP8 pools (kv_format=PA_KV_FP8_E4M3): one uint8 buffer each of num_blocks*Hkv*bs*(head_dim + 4)
    bytes (codes, then float32 scales).
    """

    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 dtype: torch.dtype = torch.float16, device: int = 0, partition_tokens: int = 0,
                 max_seqs: int = 256, max_q_heads: int = 64, max_q_len: int = 8, max_context_len: int = 8192,
                 k_cache: Optional[torch.Tensor] = None, v_cache: Optional[torch.Tensor] = None,
                 kv_format: int = PA_KV_16BIT):
        self.geometry = (num_blocks, num_kv_heads, block_size, head_dim)
        self.dtype = dtype
        self.kv_format = kv_format
        self.device = torch.device("cuda", device)
        if kv_format == PA_KV_FP8_E4M3:
            shape, cdt = (num_blocks * num_kv_heads * block_size * (head_dim + 4),), torch.uint8
        else:
            shape, cdt = self.geometry, dtype
        if k_cache is None:
            k_cache = torch.empty(shape, dtype=cdt, device=self.device)
            v_cache = torch.empty(shape, dtype=cdt, device=self.device)
        for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
            _dev(t, name, cdt)
            if tuple(t.shape) != tuple(shape):
                raise ValueError(f"{name} must have shape {tuple(shape)}")
        self.k_cache, self.v_cache = k_cache, v_cache
        cfg = PaPoolConfig(num_blocks, block_size, num_kv_heads, head_dim, _PA_DTYPE[dtype], device,
                           partition_tokens, max_seqs, max_q_heads, max_q_len, max_context_len,
                           k_cache.data_ptr(), v_cache.data_ptr(), kv_format)
        h = C.c_void_p()
        _check(lib().pa_pool_create(C.byref(cfg), C.byref(h)), "pa_pool_create")
        self._h = h

    @property
    def handle(self) -> C.c_void_p:
        if self._h is None:
            raise RuntimeError("pool is closed")
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None:
            lib().pa_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check_caches(self, k_cache: Optional[torch.Tensor], v_cache: Optional[torch.Tensor]) -> None:
        """Caches passed per call replace the pool's own: both or neither, each of the pool's shape."""
        if (k_cache is None) != (v_cache is None):
            raise ValueError("pass both k_cache and v_cache, or neither")
        if k_cache is not None:
            for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
                _dev(t, name, self.k_cache.dtype)
                if tuple(t.shape) != tuple(self.k_cache.shape):
                    raise ValueError(f"{name} must have shape {tuple(self.k_cache.shape)}")

    def _attn_args(self, q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                   out: Optional[torch.Tensor]) -> torch.Tensor:
        """Checks the shapes the library trusts (it sees only pointers) and returns out."""
        _dev(q, "q", self.dtype)
        _dev(block_tables, "block_tables", torch.int32)
        _dev(context_lens, "context_lens", torch.int32)
        d = self.geometry[3]
        if q.dim() != 4 or q.shape[3] != d:
            raise ValueError(f"q must be [B, q_len, Hq, {d}], got {tuple(q.shape)}")
        B = q.shape[0]
        if block_tables.dim() != 2 or block_tables.shape[0] < B:
            raise ValueError(f"block_tables must be [>= {B}, stride], got {tuple(block_tables.shape)}")
        if context_lens.dim() != 1 or context_lens.shape[0] < B:
            raise ValueError(f"context_lens must hold {B} entries, got {tuple(context_lens.shape)}")
        if out is None:
            out = torch.empty_like(q)
        _dev(out, "out", self.dtype)
        if tuple(out.shape) != tuple(q.shape):
            raise ValueError(f"out must have q's shape {tuple(q.shape)}, got {tuple(out.shape)}")
        return out

    def cache_write(self, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                    k_cache: Optional[torch.Tensor] = None, v_cache: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> None:
        """Scatter k, v [N, Hkv, d] into the slots given by slot_mapping (int64 [N]; -1 = skip)."""
        _dev(k, "k", self.dtype), _dev(v, "v", self.dtype), _dev(slot_mapping, "slot_mapping", torch.int64)
        hd = (self.geometry[1], self.geometry[3])
        if k.dim() != 3 or tuple(k.shape[1:]) != hd or tuple(v.shape) != tuple(k.shape):
            raise ValueError(f"k and v must be [N, {hd[0]}, {hd[1]}], got {tuple(k.shape)} and {tuple(v.shape)}")
        if slot_mapping.dim() != 1 or slot_mapping.shape[0] != k.shape[0]:
            raise ValueError(f"slot_mapping must be [{k.shape[0]}], got {tuple(slot_mapping.shape)}")
        self._check_caches(k_cache, v_cache)
        _check(lib().pa_cache_write(self.handle, _ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.numel(),
                                    _ptr(k_cache), _ptr(v_cache), _stream(stream)), "pa_cache_write")

    def decode(self, q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
               out: Optional[torch.Tensor] = None, k_cache: Optional[torch.Tensor] = None,
               v_cache: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Paged attention for q [B, q_len, Hq, d] -> out [B, q_len, Hq, d] (causal over the q_len rows)."""
        out = self._attn_args(q, block_tables, context_lens, out)
        self._check_caches(k_cache, v_cache)
        B, q_len, Hq, d = q.shape
        _check(lib().pa_decode(self.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               block_tables.shape[1], _ptr(context_lens), B, Hq, q_len, float(scale), _ptr(out),
                               _stream(stream)), "pa_decode")
        return out

    def decode_shared_prefix(self, q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                             scale: float, prefix_tokens: int, out: Optional[torch.Tensor] = None,
                             k_cache: Optional[torch.Tensor] = None, v_cache: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """pa_decode_shared_prefix: decode for sequences whose tables share their first prefix_tokens tokens."""
        out = self._attn_args(q, block_tables, context_lens, out)
        self._check_caches(k_cache, v_cache)
        B, q_len, Hq, d = q.shape
        _check(lib().pa_decode_shared_prefix(self.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                             block_tables.shape[1], _ptr(context_lens), B, Hq, q_len, float(scale),
                                             int(prefix_tokens), _ptr(out), _stream(stream)),
               "pa_decode_shared_prefix")
        return out

    def prefill(self, q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                out: Optional[torch.Tensor] = None, k_cache: Optional[torch.Tensor] = None,
                v_cache: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Chunked prefill (pa_prefill): q [B, C, Hq, 128] is a chunk of C new tokens per sequence, causal."""
        out = self._attn_args(q, block_tables, context_lens, out)
        self._check_caches(k_cache, v_cache)
        B, q_len, Hq, d = q.shape
        _check(lib().pa_prefill(self.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                block_tables.shape[1], _ptr(context_lens), B, Hq, q_len, float(scale), _ptr(out),
                                _stream(stream)), "pa_prefill")
        return out

    def launches(self, block_table_stride: int, num_seqs: int, num_q_heads: int, q_len: int) -> int:
        return lib().pa_decode_launches(self.handle, block_table_stride, num_seqs, num_q_heads, q_len)

    def selftest_wait(self, limit_ns: int, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Run the bounded-wait self-test kernel (a wait that nothing completes; see pa_pool_selftest_wait)."""
        _check(lib().pa_pool_selftest_wait(self.handle, limit_ns, _stream(stream)), "pa_pool_selftest_wait")

    def check(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        """Synchronise and return (and clear) the device status: PA_OK, PA_ERR_DEVICE_BOUNDS or PA_ERR_TIMEOUT."""
        return lib().pa_pool_check(self.handle, _stream(stream))


def pool_create_status(**cfg) -> int:
    """pa_pool_create's status for a raw config (host-side validation; destroys the pool on success)."""
    c = PaPoolConfig(**cfg)
    h = C.c_void_p()
    st = lib().pa_pool_create(C.byref(c), C.byref(h))
    if st == PA_OK:
        lib().pa_destroy(h)
    return st


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # PA_NOALLOC_SCRATCH_BYTES
_noalloc_ready = False


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                   context_lens: torch.Tensor, scale: float, out: torch.Tensor, partition_tokens: int = 0,
                   stream: Optional[torch.cuda.Stream] = None) -> int:
    """pa_decode_noalloc: the paged decode for callers that cannot allocate device memory.

    The caches carry the pool geometry ([num_blocks, Hkv, block_size, d]); the split workspace is the
    library's static device array, so nothing is allocated. Returns the pa_status code."""
    global _noalloc_ready
    L = lib()
    if not _noalloc_ready:
        P, I32 = C.c_void_p, C.c_int32
        L.pa_decode_noalloc.argtypes = [P, P, P, I32, I32, I32, I32, I32, P, I32, P, I32, I32, I32, C.c_float, I32,
                                        P, P]
        L.pa_decode_noalloc.restype = C.c_int
        _noalloc_ready = True
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        _dev(t, name, q.dtype)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    if k_cache.dim() != 4 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must both be [num_blocks, Hkv, block_size, d]")
    NB, Hkv, bs, d = k_cache.shape
    if q.dim() != 4 or q.shape[3] != d or tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"q and out must be [B, q_len, Hq, {d}], got {tuple(q.shape)} and {tuple(out.shape)}")
    B, q_len, Hq, _ = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] < B or context_lens.dim() != 1 or context_lens.shape[0] < B:
        raise ValueError("block_tables must be [>= B, stride] and context_lens [>= B]")
    return L.pa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), NB, bs, Hkv, d, _PA_DTYPE[q.dtype],
                               _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, q_len,
                               float(scale), partition_tokens, _ptr(out), _stream(stream))


# ------------------------------------------------------------------------------ block manager

_alloc_ready = False


def _alloc_lib() -> C.CDLL:
    global _alloc_ready
    L = lib()
    if not _alloc_ready:
        P, I32 = C.c_void_p, C.c_int32
        L.pa_allocator_create.argtypes = [I32, I32, C.POINTER(C.c_void_p)]
        L.pa_allocator_destroy.argtypes = [P]
        L.pa_allocator_destroy.restype = None
        L.pa_allocator_num_free.argtypes = [P]
        L.pa_allocator_num_free.restype = I32
        L.pa_allocator_ref_count.argtypes = [P, I32]
        L.pa_allocator_ref_count.restype = I32
        L.pa_allocator_alloc.argtypes = [P, I32, P]
        L.pa_allocator_fork.argtypes = [P, P, I32]
        L.pa_allocator_free.argtypes = [P, P, I32]
        L.pa_allocator_cow.argtypes = [P, I32, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
        L.pa_allocator_append.argtypes = [P, P, I32, C.POINTER(C.c_int32), I32, P, P, C.POINTER(C.c_int32)]
        L.pa_copy_blocks.argtypes = [P, P, I32, P, P, P]
        for f in ("pa_allocator_create", "pa_allocator_alloc", "pa_allocator_fork", "pa_allocator_free",
                  "pa_allocator_cow", "pa_allocator_append", "pa_copy_blocks"):
            getattr(L, f).restype = C.c_int
        _alloc_ready = True
    return L


class BlockAllocator:
    """Host-side free pool with reference counts and copy-on-write (pa_allocator_*). No GPU needed."""

    def __init__(self, num_blocks: int, block_size: int):
        import numpy as np
        self._np = np
        self.block_size = block_size
        h = C.c_void_p()
        _check(_alloc_lib().pa_allocator_create(num_blocks, block_size, C.byref(h)), "pa_allocator_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None:
            _alloc_lib().pa_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ids(self, ids):
        return self._np.ascontiguousarray(ids, dtype=self._np.int32)

    @property
    def num_free(self) -> int:
        return _alloc_lib().pa_allocator_num_free(self._h)

    def ref_count(self, block_id: int) -> int:
        return _alloc_lib().pa_allocator_ref_count(self._h, block_id)

    def alloc(self, n: int):
        out = self._np.empty(n, dtype=self._np.int32)
        _check(_alloc_lib().pa_allocator_alloc(self._h, n, out.ctypes.data), "pa_allocator_alloc")
        return out

    def fork(self, ids) -> None:
        a = self._ids(ids)
        _check(_alloc_lib().pa_allocator_fork(self._h, a.ctypes.data, len(a)), "pa_allocator_fork")

    def free(self, ids) -> None:
        a = self._ids(ids)
        _check(_alloc_lib().pa_allocator_free(self._h, a.ctypes.data, len(a)), "pa_allocator_free")

    def cow(self, block_id: int):
        out, copy = C.c_int32(), C.c_int32()
        _check(_alloc_lib().pa_allocator_cow(self._h, block_id, C.byref(out), C.byref(copy)), "pa_allocator_cow")
        return out.value, bool(copy.value)

    def append(self, table_row, length: int, n_new: int):
        """Extend a sequence by n_new tokens. table_row: int32 numpy row, updated in place.
        Returns (slots int64[n_new], new length, copy pair or None)."""
        assert table_row.dtype == self._np.int32 and table_row.flags.c_contiguous
        slots = self._np.empty(n_new, dtype=self._np.int64)
        pair = self._np.empty(2, dtype=self._np.int32)
        ln, nc = C.c_int32(length), C.c_int32()
        _check(_alloc_lib().pa_allocator_append(self._h, table_row.ctypes.data, len(table_row), C.byref(ln), n_new,
                                                slots.ctypes.data, pair.ctypes.data, C.byref(nc)), "pa_allocator_append")
        return slots, ln.value, (tuple(int(x) for x in pair) if nc.value else None)


def copy_blocks(pool: "Pool", pairs: torch.Tensor, k_cache: Optional[torch.Tensor] = None,
                v_cache: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> None:
    """pa_copy_blocks: copy whole blocks pairs[i, 0] -> pairs[i, 1] (device int32 [n, 2])."""
    _dev(pairs, "pairs", torch.int32)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError(f"pairs must be [n, 2], got {tuple(pairs.shape)}")
    pool._check_caches(k_cache, v_cache)
    _check(_alloc_lib().pa_copy_blocks(pool.handle, _ptr(pairs), pairs.shape[0], _ptr(k_cache), _ptr(v_cache),
                                       _stream(stream)), "pa_copy_blocks")


_spec_ready = False


def spec_verify(p: torch.Tensor, q: torch.Tensor, draft: torch.Tensor, u: torch.Tensor, v: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None):
    """pa_spec_verify: speculative rejection sampling. Returns (out int32 [B, K+1], n_out int32 [B])."""
    global _spec_ready
    L = lib()
    if not _spec_ready:
        P, I32 = C.c_void_p, C.c_int32
        L.pa_spec_verify.argtypes = [P, P, P, P, P, I32, I32, C.c_int64, P, P, P]
        L.pa_spec_verify.restype = C.c_int
        _spec_ready = True
    for name, t, dt in (("p", p, torch.float32), ("q", q, torch.float32), ("draft", draft, torch.int32),
                        ("u", u, torch.float32), ("v", v, torch.float32)):
        _dev(t, name, dt)
    if p.dim() != 3:
        raise ValueError(f"p must be [B, K + 1, V], got {tuple(p.shape)}")
    B, K1, V = p.shape
    for name, t, shape in (("q", q, (B, K1 - 1, V)), ("draft", draft, (B, K1 - 1)), ("u", u, (B, K1 - 1)),
                           ("v", v, (B,))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    out = torch.empty((B, K1), dtype=torch.int32, device=p.device)
    n_out = torch.empty((B,), dtype=torch.int32, device=p.device)
    _check(L.pa_spec_verify(_ptr(p), _ptr(q), _ptr(draft), _ptr(u), _ptr(v), B, K1 - 1, V, _ptr(out), _ptr(n_out),
                            _stream(stream)), "pa_spec_verify")
    return out, n_out
