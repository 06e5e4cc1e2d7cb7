"""FP8 E4M3 KV pools on the GPU against the oracle's FP8 chain.

Codes and per-(slot, head) scales written by pa_cache_write must equal the oracle's quantisation bit for
bit (both divide in float32 and round to nearest even); decode outputs must be within the suite's tolerance
of the oracle's fp64 attention on the dequantised K/V."""
import numpy as np
import pytest
import torch

import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402

FP8 = pa.PA_KV_FP8_E4M3


def _run(wl, seqs=None, layer=0):
    pool, kc, vc, q, tables, lens = H.build_device(wl, layer, kv_format=FP8)
    out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, hk, hv = H.oracle_reference_fp8(wl, layer, seqs)
    sq = list(range(wl.B)) if seqs is None else list(seqs)
    H.check_fp8_pool_rows(wl, layer, kc, vc, hk, hv, sq)
    H.assert_close(out[sq], ref, f"fp8 {wl.name}")
    assert torch.isfinite(out.float()).all()
    return out


@pytest.mark.parametrize("k,batch", [(1, None), (2, 6), (3, 4), (4, 12), (5, 1)])
def test_fp8_reduced(k, batch):
    wl = synth.workload(k, batch=batch, layers=1)
    if wl.d != 128:
        wl = synth.custom_workload([17, 64, 100, 200], 8, 2, 128, 16, 1, synth.FP16, tag=301)
    _run(wl)


@pytest.mark.parametrize("k", [3, 5])
def test_fp8_full_size_sampled(k):
    wl = synth.workload(k, layers=1)
    _run(wl, seqs=sorted({0, wl.B // 2, wl.B - 1}))


@pytest.mark.parametrize("case", [([1, 2, 33], 8, 8, 16, 1, synth.BF16, 0, 512),
                                  ([5, 40, 517], 32, 8, 16, 5, synth.FP16, 0, 256),
                                  ([1024 + 9, 1024 + 300], 32, 8, 16, 5, synth.BF16, 1024, 512),
                                  ([700, 95], 32, 4, 32, 4, synth.BF16, 0, 256)])
def test_fp8_edges(case):
    lens, Hq, Hkv, bs, ql, dt, pre, part = case
    _run(synth.custom_workload(lens, Hq, Hkv, 128, bs, ql, dt, prefix_tokens=pre, partition_tokens=part, tag=310))


def test_fp8_stress_values():
    for stress in ("vmean", "qx8"):
        _run(synth.workload(2, batch=4, stress=stress))


def test_fp8_copy_blocks():
    wl = synth.custom_workload([300, 77], 16, 8, 128, 16, 1, synth.FP16, tag=320)
    pool, kc, vc, q, tables, lens = H.build_device(wl, kv_format=FP8)
    before_k, before_v = kc.cpu().numpy(), vc.cpu().numpy()
    free = sorted(set(range(wl.num_blocks)) - set(wl.used_blocks().tolist()))
    src = wl.block_tables[0, :3]
    pairs = np.stack([src, np.array(free[:3])], axis=1).astype(np.int32)
    pa.copy_blocks(pool, torch.from_numpy(pairs).to(H.DEV), kc, vc)
    assert pool.check() == pa.PA_OK
    geo = (wl.num_blocks, wl.Hkv, wl.bs, wl.d)
    import oracle
    for dev, before in ((kc, before_k), (vc, before_v)):
        exp_c, exp_s = [a.copy() for a in oracle.fp8_views(before, *geo)]
        for s_, d_ in pairs:
            exp_c[d_] = exp_c[s_]
            exp_s[d_] = exp_s[s_]
        got_c, got_s = oracle.fp8_views(dev.cpu().numpy(), *geo)
        assert np.array_equal(got_c, exp_c) and np.array_equal(got_s.view(np.uint32), exp_s.view(np.uint32))
