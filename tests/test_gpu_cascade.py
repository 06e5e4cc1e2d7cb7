"""GPU parity of the shared-prefix decode (pa_decode_shared_prefix) against the fp64 oracle.

The prefix's attention is computed once for all sequences' query rows on the tensor cores and
merged with each sequence's own decode partitions; the result must equal pa_decode's definition:
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise.
"""
import numpy as np
import pytest
import torch

import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402

CASES = [
    # (suffix lens, Hq, Hkv, bs, q_len, dtype, prefix, partition)
    ([64, 300, 517, 100], 32, 8, 16, 5, synth.BF16, 1024, 512),     # the verify workload's shape
    ([1, 700, 2000], 64, 8, 16, 1, synth.FP16, 512, 512),           # G = 8 decode, suffix of one token
    ([4, 64, 1000], 8, 8, 16, 4, synth.BF16, 1536, 512),            # MHA (G = 1), 3 prefix partitions
    ([2, 257, 31], 16, 4, 32, 2, synth.FP16, 768, 256),             # bs 32, 256-token partitions
    ([5, 5, 6, 7], 24, 8, 16, 5, synth.FP16, 512, 512),             # G = 3 (15 rows), suffix == q_len
    ([3, 90, 700], 24, 4, 16, 3, synth.BF16, 1536, 512),            # 18 rows, 3 prefix partitions
    ([10, 300, 4], 32, 8, 32, 4, synth.FP16, 1280, 256),            # 16 rows, bs 32, 5 prefix partitions
]


def build(case, tag):
    suf, Hq, Hkv, bs, ql, dt, pre, part = case
    lens = [pre + s for s in suf]
    wl = synth.custom_workload(lens, Hq, Hkv, 128, bs, ql, dt, prefix_tokens=pre, partition_tokens=part, tag=tag)
    return wl, H.build_device(wl, partition_tokens=part)


@pytest.mark.parametrize("case", CASES, ids=[f"prefix{i}" for i in range(len(CASES))])
def test_shared_prefix_parity(case):
    wl, (pool, kc, vc, q, tables, lens) = build(case, 340 + CASES.index(case))
    out = pool.decode_shared_prefix(q, tables, lens, wl.scale, wl.prefix_tokens, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(out, ref, f"shared prefix {case}")
    # the generic decode computes the same definition
    gen = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    H.assert_close(gen, ref, "pa_decode")


def test_many_sequences_many_row_tiles():
    """40 sequences x 20 rows per KV head = 800 rows: 7 row tiles, a ragged last one."""
    rng = np.random.default_rng(5)
    suf = [int(x) for x in rng.integers(5, 600, size=40)]
    wl, (pool, kc, vc, q, tables, lens) = build((suf, 32, 8, 16, 5, synth.BF16, 1024, 512), 350)
    out = pool.decode_shared_prefix(q, tables, lens, wl.scale, wl.prefix_tokens, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(out, ref, "40 sequences")


def test_verify_workload_full_size_sampled():
    """The verify workload at full size (128 sequences sharing a 1024-token prefix, q_len 5), launched as the
    benchmark launches it; the oracle checks the first, middle and last sequences."""
    wl = synth.workload(4)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    out = pool.decode_shared_prefix(q, tables, lens, wl.scale, wl.prefix_tokens, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    seqs = [0, wl.B // 2, wl.B - 1]
    ref, _, _ = H.oracle_reference(wl, 0, seqs)
    H.assert_close(out[seqs], ref, "verify workload")
    gen = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert torch.isfinite(out.float()).all()
    d = (out.float() - gen.float()).abs().max().item()
    assert d < 4e-3, d


def test_preconditions_flagged_and_rejected():
    wl, (pool, kc, vc, q, tables, lens) = build(([64, 100], 32, 8, 16, 5, synth.BF16, 1024, 512), 351)
    # a table whose prefix names another block
    t2 = tables.clone()
    t2[1, 3] = t2[1, 40]
    pool.decode_shared_prefix(q, t2, lens, wl.scale, 1024, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_ERR_DEVICE_BOUNDS
    # a query row inside the prefix (context shorter than prefix + q_len)
    l2 = lens.clone()
    l2[0] = 1026
    pool.decode_shared_prefix(q, tables, l2, wl.scale, 1024, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_ERR_DEVICE_BOUNDS
    # host-side rejections: not a multiple of the partition, non-positive, beyond the table
    for bad in (1000, 0, -512, 512 * 64):
        with pytest.raises(RuntimeError):
            pool.decode_shared_prefix(q, tables, lens, wl.scale, bad, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
