"""GPU parity on seeded random shapes, against the fp64 oracle.

Each case draws head_dim (64, 128), block size (16, 32), KV heads, the GQA group and q_len (up to 32
query rows per KV head), the 16-bit type, the batch, ragged context lengths (some no longer than q_len)
and the partition size, and for some head_dim-128 cases an FP8 E4M3 pool. Together the cases run every
decode variant: the mma.sync decode with one to four 8-column row tiles, the tensor-core decode, both
merges, both head dims and block sizes, FP8 codes. Outputs within 2e-3 + 1e-2 |oracle| element-wise.
"""
import numpy as np
import pytest
import torch

import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402

N_CASES = 24


def draw(seed: int):
    rng = np.random.default_rng(7000 + seed)
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    while True:
        G = int(rng.choice([1, 2, 3, 4, 6, 8]))
        q_len = int(rng.integers(1, 9))
        if G * q_len <= 32:
            break
    dt = int(rng.choice([synth.FP16, synth.BF16]))
    B = int(rng.integers(1, 7))
    part = int(rng.choice([8 * bs, 256, 512, 1024]))
    lens = [int(x) for x in rng.integers(q_len, 2600, size=B)]
    if rng.random() < 0.3:
        lens[0] = q_len                     # a context that holds only the new tokens
    fp8 = d == 128 and rng.random() < 0.3
    return lens, G * Hkv, Hkv, d, bs, q_len, dt, part, fp8


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape(seed):
    lens, Hq, Hkv, d, bs, q_len, dt, part, fp8 = draw(seed)
    wl = synth.custom_workload(lens, Hq, Hkv, d, bs, q_len, dt, partition_tokens=part, tag=700 + seed)
    fmt = pa.PA_KV_FP8_E4M3 if fp8 else pa.PA_KV_16BIT
    pool, kc, vc, q, tables, lens_d = H.build_device(wl, partition_tokens=part, kv_format=fmt)
    out = pool.decode(q, tables, lens_d, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref = H.oracle_reference_fp8(wl, 0)[0] if fp8 else H.oracle_reference(wl, 0)[0]
    H.assert_close(out, ref, f"random shape {seed}: {draw(seed)}")
    assert torch.isfinite(out.float()).all()
