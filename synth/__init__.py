"""Seeded synthetic inputs for the paged-attention decode path.

This module is test and benchmark infrastructure. It is the one thing the CPU
oracle and the CUDA path share, and it holds none of the attention arithmetic:
only counter-based random draws, the recipe that turns a draw into an fp16/bf16
value, and the shapes of the workloads (context lengths, shuffled physical
block placement, block tables, the slot of every token).

Random draws (SplitMix64, Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014):
    mix(z)   = splitmix64 output function applied to z + 0x9E3779B97F4A7C15
    base     = mix(seed XOR (stream * 0xD1B54A32D192ED03))
    h(i)     = mix(base + i)                         (all arithmetic mod 2**64)

Value recipe (an Irwin-Hall sum of twelve 16-bit uniforms, centred: the classic
"twelve uniforms minus six" stand-in for N(0,1), unit variance, tails out to 6 sigma;
every step is an exactly rounded IEEE operation, so the host and the device produce
the same bits):
    s   = sum of the four 16-bit fields of each of h(3i), h(3i+1), h(3i+2)
                                                     (integer in [0, 786420])
    z   = float32(2*s - 786420) * 2**-17             (exact: |2s - 786420| < 2**20)
    x   = z * sigma + mean                           (two float32 operations, not fused)
    out = round-to-nearest-even of x to fp16 or bf16
Each 16-bit field has variance (2**32 - 1)/12, so 2s - 786420 has variance
4 (2**32 - 1) and z has variance 1 - 2**-32.

synth/csrc/synth.cu implements the same definitions on the device for
workloads too large to draw on the host; the two agree bit for bit.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import threading
from typing import Dict, List, Optional, Tuple

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
STREAM_MUL = 0xD1B54A32D192ED03
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
N_HASH = 3                                # hashes (four 16-bit fields each) per value
S_MAX = N_HASH * 4 * 0xFFFF               # largest field sum, 786420
SCALE_F32 = np.float32(2.0 ** -17)        # 1 / sqrt(Var(2s - S_MAX)) up to 2**-33 relative

FP16, BF16 = 0, 1
DTYPES = {"fp16": FP16, "bf16": BF16}
NAN16 = {FP16: 0x7E00, BF16: 0x7FC0}     # quiet-NaN words used as pool sentinels

# stream kinds
K_Q, K_K, K_V, K_KP, K_VP, K_LENS, K_PERM = 1, 2, 3, 4, 5, 6, 7


def _mix_py(z: int) -> int:
    z = (z + GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def stream_base(seed: int, stream: int) -> int:
    return _mix_py((seed ^ ((stream * STREAM_MUL) & MASK64)) & MASK64)


def make_stream(tag: int, layer: int, kind: int) -> int:
    """Stream id: workload tag, layer index and tensor kind packed in 64 bits."""
    return ((tag & 0xFFFFFF) << 40) | ((layer & 0xFFFFFF) << 16) | (kind & 0xFFFF)


def hash64(seed: int, stream: int, idx) -> np.ndarray:
    """h(i) for an array of uint64 counters."""
    base = np.uint64(stream_base(seed, stream))
    z = np.asarray(idx, dtype=np.uint64) + base
    with np.errstate(over="ignore"):
        z = z + np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def unit_f32(seed: int, stream: int, idx, sigma: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """The float32 value x of the recipe for each counter in idx."""
    idx = np.asarray(idx, dtype=np.uint64)
    m16 = np.uint64(0xFFFF)
    s = np.zeros(idx.shape, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for j in range(N_HASH):
            h = hash64(seed, stream, idx * np.uint64(N_HASH) + np.uint64(j))
            s += (h & m16) + ((h >> np.uint64(16)) & m16) + ((h >> np.uint64(32)) & m16) + (h >> np.uint64(48))
    num = (2 * s.astype(np.int64) - S_MAX).astype(np.float32)
    z = num * SCALE_F32
    z = z * np.float32(sigma)
    z = z + np.float32(mean)
    return z


def f32_to_bits16(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 to fp16 or bf16 (nearest, ties to even); return the 16-bit words."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == FP16:
        return x.astype(np.float16).view(np.uint16)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + rounding) >> np.uint64(16)).astype(np.uint16)


def values16(seed: int, stream: int, idx, dtype: int, sigma: float = 1.0, mean: float = 0.0) -> np.ndarray:
    return f32_to_bits16(unit_f32(seed, stream, idx, sigma, mean), dtype)


_HOST_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libsynthhost.so")
_host_lock = threading.Lock()
_host = None


def _host_lib():
    """The C statement of the same recipe (synth/csrc/synth_host.c), multithreaded; None if not built."""
    global _host
    with _host_lock:
        if _host is None:
            if not os.path.exists(_HOST_LIB):
                return None
            L = ctypes.CDLL(_HOST_LIB)
            L.synth_host_fill_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int, ctypes.c_float,
                                               ctypes.c_float, ctypes.c_int]
            L.synth_host_fill_rows.restype = ctypes.c_int
            _host = L
    return _host


def fill_rows16(rows: Optional[np.ndarray], nrows: int, row_len: int, seed: int, stream: int, dtype: int,
                sigma: float = 1.0, mean: float = 0.0, use_c: bool = True) -> np.ndarray:
    """[nrows, row_len] words; row r holds counters rows[r]*row_len + c (rows None: r)."""
    L = _host_lib() if use_c else None
    if L is None:
        r = np.arange(nrows, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
        idx = (r[:, None] * row_len + np.arange(row_len, dtype=np.int64)[None, :]).astype(np.uint64)
        return values16(seed, stream, idx, dtype, sigma, mean)
    out = np.empty((nrows, row_len), dtype=np.uint16)
    rr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    L.synth_host_fill_rows(out.ctypes.data, None if rr is None else rr.ctypes.data, nrows, row_len,
                           seed & MASK64, stream & MASK64, dtype, sigma, mean, os.cpu_count() or 1)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers in [lo, hi] (h(i) mod (hi - lo + 1) + lo)."""
    h = hash64(seed, stream, np.arange(n, dtype=np.uint64))
    return (h % np.uint64(hi - lo + 1)).astype(np.int64) + lo


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1: counters ordered by their hash (stable sort)."""
    h = hash64(seed, stream, np.arange(n, dtype=np.uint64))
    return np.argsort(h, kind="stable").astype(np.int64)


# --------------------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    """One paged-decode problem: shapes, the placement of its blocks and its value streams.

    Layouts (all row-major):
      q, out         [B, q_len, Hq, d]
      new k, v       [N, Hkv, d]           (rows of the tokens written by one cache-write call)
      K/V pool       [num_blocks, Hkv, block_size, d]
      block_tables   int32 [B, stride], -1 beyond each sequence's last block
      context_lens   int32 [B], counting the q_len newest tokens
    """
    name: str
    tag: int
    seed: int
    B: int
    Hq: int
    Hkv: int
    d: int
    bs: int
    q_len: int
    dtype: int
    context_lens: np.ndarray
    num_blocks: int
    block_tables: np.ndarray
    layers: int = 1
    prefix_tokens: int = 0              # tokens shared by every sequence (copy-on-write prefix)
    partition_tokens: int = 512
    q_sigma: float = 1.0
    v_mean: float = 0.0
    perms: Optional[List[np.ndarray]] = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def stride(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    def stream(self, layer: int, kind: int) -> int:
        return make_stream(self.tag, layer, kind)

    # ---- logical token rows -------------------------------------------------------
    def suffix_base(self) -> np.ndarray:
        """First logical row of each sequence's private tokens."""
        own = self.context_lens.astype(np.int64) - self.prefix_tokens
        return np.concatenate([[0], np.cumsum(own)[:-1]]).astype(np.int64)

    def token_rows(self, b: int, t: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """(is_prefix, row) of logical tokens t of sequence b: the counter row in the K/V streams."""
        t = np.asarray(t, dtype=np.int64)
        is_pre = t < self.prefix_tokens
        row = np.where(is_pre, t, self.suffix_base()[b] + t - self.prefix_tokens)
        return is_pre, row

    def slots(self, b: int, t: np.ndarray) -> np.ndarray:
        """Pool slot (physical block * block_size + offset) of logical tokens t of sequence b."""
        t = np.asarray(t, dtype=np.int64)
        return self.block_tables[b, t // self.bs].astype(np.int64) * self.bs + t % self.bs

    def kv_values(self, layer: int, b: int, t: np.ndarray, which: str) -> np.ndarray:
        """16-bit words of K or V for tokens t of sequence b: shape [len(t), Hkv, d]."""
        is_pre, row = self.token_rows(b, t)
        HD = self.Hkv * self.d
        kind, pkind = (K_K, K_KP) if which == "k" else (K_V, K_VP)
        mean = self.v_mean if which == "v" else 0.0
        out = np.empty((len(row), HD), dtype=np.uint16)
        for flag, kd in ((True, pkind), (False, kind)):
            sel = is_pre == flag
            if not sel.any():
                continue
            out[sel] = fill_rows16(row[sel], int(sel.sum()), HD, self.seed, self.stream(layer, kd), self.dtype,
                                   1.0, mean)
        return out.reshape(len(row), self.Hkv, self.d)

    def q_values(self, layer: int, seqs: Optional[np.ndarray] = None) -> np.ndarray:
        """16-bit words of q for sequences `seqs` (default all): [len(seqs), q_len, Hq, d]."""
        seqs = np.arange(self.B) if seqs is None else np.asarray(seqs)
        per = self.q_len * self.Hq * self.d
        w = fill_rows16(seqs.astype(np.int64), len(seqs), per, self.seed, self.stream(layer, K_Q), self.dtype,
                        self.q_sigma, 0.0)
        return w.reshape(len(seqs), self.q_len, self.Hq, self.d)

    # ---- cache-write plans ----------------------------------------------------------
    def write_plan(self, new_only: bool) -> List[Tuple[int, np.ndarray, np.ndarray]]:
        """Writes that fill the pool: a list of (kind, counter rows, slots).

        new_only=False: every token except the q_len newest of each sequence (the fill).
        new_only=True: the q_len newest tokens of each sequence (the step's cache write).
        The shared prefix is written once, from sequence 0's table.
        """
        plans = []
        P = self.prefix_tokens
        if not new_only and P > 0:
            t = np.arange(P, dtype=np.int64)
            plans.append((K_KP, t, self.slots(0, t)))
        rows, slots = [], []
        for b in range(self.B):
            L = int(self.context_lens[b])
            t = np.arange(L - self.q_len, L) if new_only else np.arange(P, L - self.q_len)
            _, r = self.token_rows(b, t)
            rows.append(r)
            slots.append(self.slots(b, t))
        plans.append((K_K, np.concatenate(rows), np.concatenate(slots)))
        return plans

    def used_blocks(self) -> np.ndarray:
        """Distinct physical blocks referenced by the tables (sorted)."""
        ids = []
        for b in range(self.B):
            nb = -(-int(self.context_lens[b]) // self.bs)
            ids.append(self.block_tables[b, :nb])
        return np.unique(np.concatenate(ids))

    def kv_bytes_unique(self) -> int:
        """K and V bytes of the valid tokens, counting shared prefix tokens once."""
        toks = int(self.context_lens.sum()) - (self.B - 1) * self.prefix_tokens
        return 2 * toks * self.Hkv * self.d * 2

    def algorithmic_bytes(self) -> int:
        """Bytes one decode call must move: Q + K/V (valid tokens, unique) + used table entries + lens + out."""
        qo = 2 * self.B * self.q_len * self.Hq * self.d * 2
        tbl = int(sum(-(-int(L) // self.bs) for L in self.context_lens)) * 4
        return qo + self.kv_bytes_unique() + tbl + 4 * self.B


def _tables_from_perm(perm: np.ndarray, lens: np.ndarray, bs: int, stride: int,
                      prefix_blocks: int = 0) -> np.ndarray:
    B = len(lens)
    tables = np.full((B, stride), -1, dtype=np.int32)
    pos = prefix_blocks
    for b in range(B):
        nb = -(-int(lens[b]) // bs)
        tables[b, :prefix_blocks] = perm[:prefix_blocks]
        own = nb - prefix_blocks
        tables[b, prefix_blocks:nb] = perm[pos:pos + own]
        pos += own
    return tables


def workload(k: int, layers: Optional[int] = None, batch: Optional[int] = None,
             stress: str = "") -> Workload:
    """The five paged-decode workloads (k = 1..5) with seed 0x5EED0000 + k.

    batch overrides the batch size (a smaller instance of the same recipe for fast parity
    tests); layers overrides the layer count of workload 3. stress = "vmean" draws V with
    mean 1, "qx8" draws q with standard deviation 8 (both keep every shape).
    """
    seed = 0x5EED0000 + k
    tag = k + (16 if stress == "vmean" else 32 if stress == "qx8" else 0)
    q_sigma = 8.0 if stress == "qx8" else 1.0
    v_mean = 1.0 if stress == "vmean" else 0.0
    if k == 1:
        lens = np.array([17, 64, 100, 200], dtype=np.int32)
        B, Hq, Hkv, d, bs, ql, dt, NB, nl, pre = 4, 8, 2, 64, 16, 1, FP16, 64, 1, 0
    elif k == 2:
        B = batch or 64
        lens = uniform_int(seed, make_stream(tag, 0, K_LENS), B, 512, 4096).astype(np.int32)
        Hq, Hkv, d, bs, ql, dt, nl, pre = 32, 8, 128, 16, 1, BF16, 1, 0
        NB = int(math.ceil(1.1 * sum(-(-int(L) // bs) for L in lens)))
    elif k == 3:
        B = batch or 64
        lens = np.full(B, 8192, dtype=np.int32)
        Hq, Hkv, d, bs, ql, dt, pre = 64, 8, 128, 16, 1, FP16, 0
        nl = 80 if layers is None else layers
        NB = B * 512
    elif k == 4:
        B = batch or 128
        suf = uniform_int(seed, make_stream(tag, 0, K_LENS), B, 64, 512)
        pre = 1024
        lens = (pre + suf).astype(np.int32)
        Hq, Hkv, d, bs, ql, dt, nl = 32, 8, 128, 16, 5, BF16, 1
        own = sum(-(-int(s) // bs) for s in suf)
        NB = int(math.ceil(1.1 * (pre // bs + own)))
    elif k == 5:
        B = batch or 4
        lens = np.full(B, 131072, dtype=np.int32)
        Hq, Hkv, d, bs, ql, dt, nl, pre = 32, 8, 128, 32, 1, FP16, 1, 0
        NB = B * (131072 // 32)
    else:
        raise ValueError(f"no workload {k}")
    stride = max(-(-int(L) // bs) for L in lens)
    perms = []
    tables = None
    for layer in range(nl):
        perm = permutation(seed, make_stream(tag, layer, K_PERM), NB)
        perms.append(perm)
        if layer == 0:
            tables = _tables_from_perm(perm, lens, bs, stride, pre // bs)
    wl = Workload(name=f"cfg{k}", tag=tag, seed=seed, B=B, Hq=Hq, Hkv=Hkv, d=d, bs=bs, q_len=ql,
                  dtype=dt, context_lens=lens, num_blocks=NB, block_tables=tables, layers=nl,
                  prefix_tokens=pre, q_sigma=q_sigma, v_mean=v_mean, perms=perms)
    return wl


def custom_workload(lens, Hq: int, Hkv: int, d: int, bs: int, q_len: int, dtype: int, prefix_tokens: int = 0,
                    free_frac: float = 0.1, tag: int = 99, partition_tokens: int = 512, q_sigma: float = 1.0,
                    v_mean: float = 0.0, stride: Optional[int] = None) -> Workload:
    """A workload with explicit context lengths (edge cases); blocks placed by a seeded shuffle."""
    lens = np.asarray(lens, dtype=np.int32)
    seed = 0x5EED0000 + tag
    own = sum(-(-int(L) // bs) - prefix_tokens // bs for L in lens)
    NB = int(math.ceil((1 + free_frac) * (prefix_tokens // bs + own))) + 1
    st = max(-(-int(L) // bs) for L in lens) if stride is None else stride
    perm = permutation(seed, make_stream(tag, 0, K_PERM), NB)
    tables = _tables_from_perm(perm, lens, bs, st, prefix_tokens // bs)
    return Workload(name=f"custom{tag}", tag=tag, seed=seed, B=len(lens), Hq=Hq, Hkv=Hkv, d=d, bs=bs, q_len=q_len,
                    dtype=dtype, context_lens=lens, num_blocks=NB, block_tables=tables, layers=1,
                    prefix_tokens=prefix_tokens, partition_tokens=partition_tokens, q_sigma=q_sigma, v_mean=v_mean,
                    perms=[perm])


def layer_tables(wl: Workload, layer: int) -> np.ndarray:
    """Block tables of one layer (each layer's pool has its own shuffled placement)."""
    if layer == 0:
        return wl.block_tables
    return _tables_from_perm(wl.perms[layer], wl.context_lens, wl.bs, wl.stride,
                             wl.prefix_tokens // wl.bs)


def with_layer(wl: Workload, layer: int) -> Workload:
    """A view of wl whose block_tables are those of `layer`."""
    return dataclasses.replace(wl, block_tables=layer_tables(wl, layer))


def describe(wl: Workload) -> Dict[str, object]:
    return {"workload": wl.name, "batch": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": wl.d,
            "block_size": wl.bs, "q_len": wl.q_len, "dtype": "fp16" if wl.dtype == FP16 else "bf16",
            "context_lens": "const %d" % wl.context_lens[0] if len(set(wl.context_lens.tolist())) == 1
            else "%d..%d (mean %.0f)" % (wl.context_lens.min(), wl.context_lens.max(), wl.context_lens.mean()),
            "num_blocks": wl.num_blocks, "layers": wl.layers, "prefix_tokens": wl.prefix_tokens,
            "partition_tokens": wl.partition_tokens}
