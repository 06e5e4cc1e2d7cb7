"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Cache writes are compared word for word; attention outputs element-wise within
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import synth.device as sdev
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402


def test_device_generator_matches_host():
    rows = torch.tensor([0, 7, 123456, 2 ** 33 + 5], dtype=torch.int64, device=H.DEV)
    for dt in (synth.FP16, synth.BF16):
        for sigma, mean in ((1.0, 0.0), (8.0, 0.0), (1.0, 1.0)):
            t = torch.empty((4, 1024), dtype=torch.int16, device=H.DEV)
            sdev.fill_rows(t, rows, 1024, 0x5EED0001, 99, dt, sigma, mean)
            host = synth.fill_rows16(rows.cpu().numpy(), 4, 1024, 0x5EED0001, 99, dt, sigma, mean, use_c=False)
            assert np.array_equal(t.cpu().numpy().view(np.uint16), host)


def test_tiny_config_full_chain():
    """Tiny paged decode (4 sequences, lens 17/64/100/200, Hq 8, Hkv 2, d 64, bs 16, fp16): whole pool bit-exact,
    outputs within tolerance."""
    wl = synth.workload(1)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, hk, hv = H.oracle_reference(wl, 0, full_pool=True)
    assert np.array_equal(H.pool_words(kc), hk)
    assert np.array_equal(H.pool_words(vc), hv)
    H.assert_close(out, ref, "cfg1")


@pytest.mark.parametrize("k,batch", [(2, 8), (3, 4), (4, 16), (5, 1)])
def test_reduced_configs(k, batch):
    """Each workload's recipe at a reduced batch: every output and every used block checked."""
    wl = synth.workload(k, batch=batch, layers=1)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, hk, hv = H.oracle_reference(wl, 0)
    H.check_pool_blocks(wl, 0, kc, vc, hk, hv, range(wl.B))
    H.assert_close(out, ref, f"cfg{k} batch {batch}")


@pytest.mark.parametrize("k", [2, 3, 4, 5])
def test_full_size_every_row(k):
    """The workloads at full size, launched as the benchmark launches them (same batch, heads and pool
    geometry, hence the same partitions per CTA): every output row of every sequence against the oracle,
    and every used block of every sequence word for word. Workload 3 is checked on its second layer pool
    (its own shuffled placement); the benchmark runs the same launch on each of its 80 pools."""
    wl = synth.workload(k, layers=2 if k == 3 else None)
    layer = 1 if k == 3 else 0
    pool, kc, vc, q, tables, lens = H.build_device(wl, layer)
    out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, hk, hv = H.oracle_reference(wl, layer)
    H.check_pool_blocks(wl, layer, kc, vc, hk, hv, range(wl.B))
    mx, mr = H.assert_close(out, ref, f"cfg{k} full")
    print(f"cfg{k} full size, all {wl.B} sequences x {wl.q_len} x {wl.Hq} rows: max abs err {mx:.3g}, "
          f"max rel err {mr:.3g}")


EDGE = [
    # (lens, Hq, Hkv, d, bs, q_len, dtype, prefix, partition)
    ([1], 8, 2, 64, 16, 1, synth.FP16, 0, 512),                 # single token
    ([5, 6, 21], 32, 8, 128, 16, 5, synth.BF16, 0, 512),        # context == q_len, just above
    ([16, 32, 512, 513, 1024], 16, 8, 128, 16, 1, synth.FP16, 0, 512),   # block / partition boundaries
    ([33, 64, 95], 8, 8, 64, 32, 1, synth.BF16, 0, 32),         # MHA (G = 1), bs 32, tiny partitions
    ([700, 1000], 32, 4, 128, 32, 4, synth.FP16, 0, 256),       # G = 8, q_len 4: 32 rows
    ([300, 517], 24, 8, 64, 16, 3, synth.BF16, 0, 64),          # G = 3, q_len 3: 9 rows
    ([1024 + 7, 1024 + 100], 32, 8, 128, 16, 5, synth.BF16, 1024, 512),  # shared prefix + verify
    ([2000, 31, 4097], 64, 8, 128, 16, 1, synth.FP16, 0, 512),  # ragged lengths, G = 8
    ([516, 1030], 16, 4, 128, 16, 5, synth.FP16, 0, 512),       # draft rows straddle a partition edge
    ([1500, 40], 32, 1, 128, 16, 1, synth.BF16, 0, 256),        # G = 32 (one KV head): 32 rows, wide merge
]


@pytest.mark.parametrize("case", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
def test_edge_cases(case):
    lens, Hq, Hkv, d, bs, ql, dt, pre, part = case
    wl = synth.custom_workload(lens, Hq, Hkv, d, bs, ql, dt, prefix_tokens=pre, partition_tokens=part,
                               tag=200 + EDGE.index(case))
    pool, kc, vc, q, tables, lens_d = H.build_device(wl)
    out = pool.decode(q, tables, lens_d, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, hk, hv = H.oracle_reference(wl, 0)
    H.check_pool_blocks(wl, 0, kc, vc, hk, hv, range(wl.B))
    H.assert_close(out, ref, f"edge {case}")


def test_coarsened_partitions_every_sequence():
    """Enough (sequence, KV head) units that the launch merges 512-token partitions in pairs (on a
    152-SM part: 320 units x 8 merged partitions >= 8 waves of 2 CTAs per SM), with contexts on and
    around the merged and unmerged partition edges and one at the table's maximum; every sequence
    is checked against the oracle."""
    edges = []
    for c in range(1, 8):
        edges += [1024 * c - 1, 1024 * c, 1024 * c + 1, 1024 * c + 512, 1024 * c - 511]
    rng = np.random.default_rng(77)
    lens = edges + [8192, 1, 16, 17] + [int(x) for x in rng.integers(1, 8193, size=160 - len(edges) - 4)]
    wl = synth.custom_workload(lens, 16, 2, 64, 16, 1, synth.FP16, tag=260)
    pool, kc, vc, q, tables, lens_d = H.build_device(wl)
    out = pool.decode(q, tables, lens_d, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(out, ref, "coarsened partitions")


@pytest.mark.parametrize("stress", ["vmean", "qx8"])
def test_stress_variants(stress):
    """Same shapes, harder numerics: V with mean 1 (relative tolerance governs) and q x 8 (peaked softmax)."""
    for k, batch in ((5, 1), (2, 4)):
        wl = synth.workload(k, batch=batch, stress=stress)
        pool, kc, vc, q, tables, lens = H.build_device(wl)
        out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
        ref, _, _ = H.oracle_reference(wl, 0)
        H.assert_close(out, ref, f"cfg{k} {stress}")


def _scaled_words(words: np.ndarray, factor: np.ndarray, dtype: int) -> np.ndarray:
    """16-bit words times a float32 factor, rounded to nearest even (test-side: builds inputs, not expected values)."""
    if dtype == synth.FP16:
        return (words.view(np.float16).astype(np.float32) * factor).astype(np.float16).view(np.uint16)
    f = (words.astype(np.uint32) << 16).view(np.float32) * factor
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


# (lens, Hq, Hkv, q_len, dtype): one 8-column tile of rows on the mma.sync decode, and 20 rows on the
# tensor-core decode; contexts over several partitions
RISING = [([1500, 3000, 700], 64, 8, 1, synth.FP16), ([900, 2100, 1300], 32, 8, 5, synth.BF16)]


@pytest.mark.parametrize("case", RISING, ids=["decode_g8", "verify_20rows"])
def test_rising_scores_move_the_softmax_reference(case):
    """Keys scaled by 1 + 15 t / L along each context, so that the scores' spread grows from N(0,1) to 16
    sigma: every row's running maximum passes its reference by more than 2^8 several times, in late tiles and
    partitions too, which makes the kernels rescale O and the merge combine partitions whose references differ
    widely."""
    lens, Hq, Hkv, q_len, dt = case
    wl = synth.custom_workload(lens, Hq, Hkv, 128, 16, q_len, dt, tag=360 + RISING.index(case))
    pool, kc, vc, q, tables, lens_d = H.build_device(wl)
    _, hk, hv = H.oracle_reference(wl, 0)
    kw = kc.view(torch.int16)
    for b, L in enumerate(wl.context_lens):
        t = np.arange(int(L))
        slots = wl.slots(b, t)
        blk, off = slots // wl.bs, slots % wl.bs
        factor = (1.0 + 15.0 * t / float(L)).astype(np.float32)[:, None, None]
        words = _scaled_words(hk[blk, :, off, :], factor, dt)
        hk[blk, :, off, :] = words
        kw[torch.from_numpy(blk).to(H.DEV), :, torch.from_numpy(off).to(H.DEV), :] = \
            torch.from_numpy(words.view(np.int16)).to(H.DEV)
    out = pool.decode(q, tables, lens_d, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _ = oracle.paged_attention(wl.q_values(0), hk, hv, wl.block_tables, wl.context_lens, wl.dtype, wl.scale)
    H.assert_close(out, ref, f"rising scores {case}")

