"""The tensor-core decode kernel (9..32 query rows per KV head) against the fp64 oracle.

pa_decode routes a KV head's query rows to this kernel when there are more than 8 of them (a wide
GQA group, or draft rows of a verify pass: q_len * G), for 16-bit pools with head_dim 128. These
cases cover its item walk (several items per CTA, partitions merged or written directly), the
keys past an item (context end and partition ends that are not multiples of its 128-key tile),
both 16-bit types (bf16 weights carried as high + low parts), a shared copy-on-write prefix, and
harder numerics.
"""
import numpy as np
import pytest
import torch

import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402

CASES = [
    # (lens, Hq, Hkv, bs, q_len, dtype, prefix, partition)
    ([5, 37, 300, 1000, 4097], 32, 4, 16, 4, synth.BF16, 0, 512),   # 32 rows, ragged, some shorter than a tile
    ([129, 640, 2500], 28, 4, 32, 4, synth.FP16, 0, 256),          # 28 rows, block size 32
    ([6000, 777], 25, 5, 16, 5, synth.BF16, 0, 512),               # 25 rows (G = 5, q_len 5)
    ([500, 1000, 61], 32, 4, 16, 4, synth.FP16, 0, 48),            # partitions of 48 tokens: items end mid-tile
    ([9, 100, 2049], 32, 8, 16, 8, synth.BF16, 0, 512),            # q_len 8, G = 4
    ([1024 + 40, 1024 + 300, 1024 + 511], 32, 4, 16, 4, synth.BF16, 1024, 512),   # shared copy-on-write prefix
    ([32768, 20000], 64, 2, 32, 1, synth.FP16, 0, 512),            # one 32-head group, long contexts
    ([80, 600, 4], 24, 8, 16, 4, synth.FP16, 0, 512),              # 12 rows (G = 3, q_len 4), context = q_len
    ([5000, 17], 16, 1, 32, 1, synth.BF16, 0, 256),                # 16 rows: one 16-head group
    ([1300, 1100, 1536], 32, 8, 16, 5, synth.BF16, 0, 512),        # 20 rows: the verify workload's shape
]


@pytest.mark.parametrize("case", CASES, ids=[f"tc{i}" for i in range(len(CASES))])
def test_tensor_core_decode_matches_oracle(case):
    lens, Hq, Hkv, bs, ql, dt, pre, part = case
    assert 8 < Hq // Hkv * ql <= 32
    wl = synth.custom_workload(lens, Hq, Hkv, 128, bs, ql, dt, prefix_tokens=pre, partition_tokens=part,
                               tag=400 + CASES.index(case))
    pool, kc, vc, q, tables, lens_d = H.build_device(wl)
    out = pool.decode(q, tables, lens_d, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, hk, hv = H.oracle_reference(wl, 0)
    H.check_pool_blocks(wl, 0, kc, vc, hk, hv, range(wl.B))
    mx, mr = H.assert_close(out, ref, f"tensor-core decode {case}")
    print(f"case {case}: max abs err {mx:.3g}, max rel err {mr:.3g}")
    if pre:
        out2 = pool.decode_shared_prefix(q, tables, lens_d, wl.scale, pre, k_cache=kc, v_cache=vc)
        assert pool.check() == pa.PA_OK
        H.assert_close(out2, ref, "shared-prefix decode, 32 rows")


@pytest.mark.parametrize("stress", ["vmean", "qx8"])
def test_tensor_core_decode_stress(stress):
    """32 rows per KV head with V of mean 1 (relative tolerance governs) and q x 8 (peaked softmax: the lazily
    raised reference max rescales O)."""
    for dt in (synth.BF16, synth.FP16):
        wl = synth.custom_workload([3000, 130, 1200], 32, 4, 128, 16, 4, dt, tag=420 + dt,
                                   q_sigma=8.0 if stress == "qx8" else 1.0, v_mean=1.0 if stress == "vmean" else 0.0)
        pool, kc, vc, q, tables, lens = H.build_device(wl)
        out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
        assert pool.check() == pa.PA_OK
        ref, _, _ = H.oracle_reference(wl, 0)
        H.assert_close(out, ref, f"tensor-core decode {stress} dtype {dt}")


def test_tensor_core_decode_deterministic_and_placement_invariant():
    """Two runs are bitwise equal, and so is the same problem with its blocks placed elsewhere in the pool."""
    wl = synth.custom_workload([2000, 513, 77], 32, 4, 128, 16, 4, synth.BF16, tag=430)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    a = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    b = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # the same tokens, each block moved to another physical id (a fixed permutation of the pool)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(wl.num_blocks).astype(np.int64)).to(H.DEV)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = torch.where(tables >= 0, perm[tables.clamp(min=0).long()].int(), tables)
    c = pool.decode(q, t2, lens, wl.scale, k_cache=kc2, v_cache=vc2)
    assert pool.check() == pa.PA_OK
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
