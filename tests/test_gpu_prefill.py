"""GPU parity of the chunked prefill (pa_prefill, tcgen05 tensor cores) against the fp64 oracle.

A chunk of C new tokens per sequence is written to the pool through pa_cache_write after the
earlier tokens; pa_prefill then computes the chunk's causal attention, which the oracle computes
as paged attention with q_len = C. Outputs element-wise within |gpu - oracle| <= 2e-3 + 1e-2 |oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402

CASES = [
    # (lens, Hq, Hkv, bs, C, dtype, prefix)
    ([512], 32, 8, 16, 512, synth.FP16, 0),                 # first chunk of a prompt: context == chunk
    ([1024, 1536], 32, 8, 16, 512, synth.BF16, 0),          # later chunks, G = 4
    ([77, 300, 1000], 16, 4, 16, 77, synth.FP16, 0),        # ragged contexts, 308 rows: ragged row tile
    ([200, 1000], 8, 8, 32, 200, synth.BF16, 0),            # MHA (G = 1), bs 32
    ([100, 450], 24, 8, 16, 100, synth.FP16, 0),            # G = 3: a chunk position spans two row tiles
    ([1, 300], 8, 2, 16, 1, synth.BF16, 0),                 # C = 1 (a decode step through the prefill path)
    ([63, 64, 65, 129], 16, 2, 16, 63, synth.FP16, 0),      # contexts at the 64-token tile edges
    ([1024 + 300, 1024 + 300], 32, 8, 16, 300, synth.BF16, 1024),   # shared copy-on-write prefix
    ([4096 + 512], 64, 8, 16, 512, synth.BF16, 0),          # 70B-style heads (G = 8), 4096 rows per KV head
    ([2048 + 7], 16, 1, 32, 7, synth.FP16, 0),              # one KV head (G = 16), short chunk, long context
]


def run_prefill(wl, stress_rows=None):
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    out = pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    return pool, kc, vc, out


@pytest.mark.parametrize("case", CASES, ids=[f"chunk{i}" for i in range(len(CASES))])
def test_prefill_parity(case):
    lens, Hq, Hkv, bs, C, dt, pre = case
    wl = synth.custom_workload(lens, Hq, Hkv, 128, bs, C, dt, prefix_tokens=pre, tag=300 + CASES.index(case))
    pool, kc, vc, out = run_prefill(wl)
    ref, hk, hv = H.oracle_reference(wl, 0)
    H.check_pool_blocks(wl, 0, kc, vc, hk, hv, range(wl.B))
    H.assert_close(out, ref, f"prefill {case}")


@pytest.mark.parametrize("stress", ["qx8", "vmean"])
def test_prefill_stress(stress):
    """Peaked softmax (q x 8: the running max moves often and far) and V with mean 1."""
    kw = dict(q_sigma=8.0) if stress == "qx8" else dict(v_mean=1.0)
    wl = synth.custom_workload([700, 1300], 32, 8, 128, 16, 256, synth.BF16, tag=320, **kw)
    _, _, _, out = run_prefill(wl)
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(out, ref, f"prefill {stress}")


def _bf16_words(f: np.ndarray) -> np.ndarray:
    """float32 -> bf16 words, rounded to nearest even (test-side: builds inputs, not expected values)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_prefill_bf16_values_beyond_fp16_range():
    """bf16 V values far outside fp16's range (where an fp16 shortcut for the weights would overflow): one
    sequence's key tile 1 holds values near 3e5, the other's tile 4 (partly, up to its context end) values near
    -1e5, the rest N(0,1)."""
    wl = synth.custom_workload([700, 1300], 32, 8, 128, 16, 256, synth.BF16, tag=321)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    _, hk, hv = H.oracle_reference(wl, 0)
    vw = vc.view(torch.int16)
    for b, t0, t1, shift in ((1, 128, 256, 3.0e5), (0, 512, 700, -1.0e5)):
        slots = wl.slots(b, np.arange(t0, t1))
        blk, off = slots // wl.bs, slots % wl.bs
        vals = (hv[blk, :, off, :].astype(np.uint32) << 16).view(np.float32) + np.float32(shift)
        words = _bf16_words(vals)
        hv[blk, :, off, :] = words
        vw[torch.from_numpy(blk).to(H.DEV), :, torch.from_numpy(off).to(H.DEV), :] = \
            torch.from_numpy(words.view(np.int16)).to(H.DEV)
    out = pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _ = oracle.paged_attention(wl.q_values(0), hk, hv, wl.block_tables, wl.context_lens, wl.dtype, wl.scale)
    assert np.abs(ref).max() > 1e4
    H.assert_close(out, ref, "prefill with V beyond fp16's range")


def test_prefill_matches_decode_for_short_chunks():
    """For q_len <= 8 both entry points compute the same definition: both within tolerance of the oracle,
    and close to each other."""
    wl = synth.custom_workload([40, 700, 2000], 32, 8, 128, 16, 4, synth.FP16, tag=321)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    a = pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    b = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(a, ref, "prefill")
    H.assert_close(b, ref, "decode")


def test_prefill_deterministic_and_rejects():
    wl = synth.custom_workload([300, 500], 16, 4, 128, 16, 128, synth.FP16, tag=322)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    a = pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    b = pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # a context shorter than the chunk is flagged on the device
    bad = lens.clone()
    bad[0] = 100
    pool.prefill(q, tables, bad, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_ERR_DEVICE_BOUNDS
    # the softmax scale must be positive
    with pytest.raises(RuntimeError):
        pool.prefill(q, tables, lens, -wl.scale, k_cache=kc, v_cache=vc)
    # head_dim 64 pools are not supported by the prefill path
    small = pa.Pool(16, 16, 2, 64, torch.float16, 0, max_seqs=1, max_q_heads=4, max_q_len=1, max_context_len=256)
    q64 = torch.zeros((1, 4, 4, 64), dtype=torch.float16, device=H.DEV)
    t = torch.zeros((1, 16), dtype=torch.int32, device=H.DEV)
    n = torch.full((1,), 4, dtype=torch.int32, device=H.DEV)
    with pytest.raises(RuntimeError):
        small.prefill(q64, t, n, 0.125)


@pytest.mark.parametrize("dt", [synth.FP16, synth.BF16], ids=["fp16", "bf16"])
def test_prefill_benchmark_workload_sampled(dt):
    """The benchmark's prefill pool at full size (8 sequences, 512-token chunk ending at context 4608, Hq 64,
    Hkv 8), launched as the benchmark launches it; the oracle checks the first and last sequences."""
    wl = synth.custom_workload([4608] * 8, 64, 8, 128, 16, 512, dt, tag=500)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    out = pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    seqs = [0, wl.B - 1]
    ref, hk, hv = H.oracle_reference(wl, 0, seqs)
    H.check_pool_blocks(wl, 0, kc, vc, hk, hv, seqs)
    H.assert_close(out[seqs], ref, "prefill benchmark workload")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("case", [([2048], 8, 2, 16, 2048, synth.FP16),      # a 2048-token first chunk
                                  ([1536, 3000], 16, 4, 32, 1024, synth.BF16)],  # 1024-token chunks, bs 32
                         ids=["chunk2048", "chunk1024_bs32"])
def test_prefill_long_chunks(case):
    lens, Hq, Hkv, bs, C, dt = case
    wl = synth.custom_workload(lens, Hq, Hkv, 128, bs, C, dt, tag=330 + C // 512)
    pool, kc, vc, q, tables, lens_d = H.build_device(wl)
    out = pool.prefill(q, tables, lens_d, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(out, ref, f"prefill {case}")


def test_prefill_rejects_fp8_pools():
    wl = synth.custom_workload([64], 8, 2, 128, 16, 16, synth.FP16, tag=331)
    pool, kc, vc, q, tables, lens = H.build_device(wl, kv_format=pa.PA_KV_FP8_E4M3)
    with pytest.raises(RuntimeError):
        pool.prefill(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
