"""pa_decode_noalloc, the allocation-free decode, against pa_decode.

Callers that cannot allocate device memory (a host runtime that owns every device
allocation, or a loop that must not make cudaMalloc's synchronising call) use
pa_decode_noalloc, whose split workspace is a static device array inside the library.
Its outputs must match pa_decode's within the suite's tolerance, call after call,
even though every call reuses the same scratch array.
"""
import pytest
import torch

import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402


def _case(wl):
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    ref = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    return dict(wl=wl, kc=kc, vc=vc, q=q, tables=tables, lens=lens, ref=ref)


def _noalloc(c):
    out = torch.empty_like(c["q"])
    st = pa.decode_noalloc(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], c["wl"].scale, out,
                           partition_tokens=c["wl"].partition_tokens)
    assert st == pa.PA_OK, pa.status_string(st)
    return out


def test_noalloc_matches_pa_decode_on_consecutive_calls():
    # long fp16 context: 64 partitions of 512 tokens share the static scratch
    a = _case(synth.custom_workload([32768, 1000], 32, 8, 128, 32, 1, synth.FP16, tag=91))
    # bf16 shared prefix + 5-token verify, 256-token partitions
    b = _case(synth.custom_workload([1024 + 300, 1024 + 45, 1024 + 512], 32, 8, 128, 16, 5, synth.BF16,
                                    prefix_tokens=1024, partition_tokens=256, tag=92))
    for c in (a, b, a, a, b):
        out = _noalloc(c)
        torch.cuda.synchronize()
        ref = H.to_f64(c["ref"])
        H.assert_close(out, ref, "pa_decode_noalloc vs pa_decode")


def test_noalloc_rejects_requests_beyond_the_static_scratch():
    wl = synth.custom_workload([64], 8, 2, 64, 16, 1, synth.FP16, tag=93)
    kc, vc = H.alloc_caches(wl)
    B, Hq, d = 64, 64, 128
    stride = 4096                                   # 65536 tokens at bs 16 -> 128 partitions of 512
    q = torch.zeros((B, 1, Hq, d), dtype=torch.float16, device=H.DEV)
    out = torch.empty_like(q)
    tables = torch.zeros((B, stride), dtype=torch.int32, device=H.DEV)
    lens = torch.full((B,), 64, dtype=torch.int32, device=H.DEV)
    kc2 = torch.empty((wl.num_blocks, 8, 16, d), dtype=torch.float16, device=H.DEV)
    need = B * Hq * 128 * (d * 4 + 8)
    assert need > pa.NOALLOC_SCRATCH_BYTES
    st = pa.decode_noalloc(q, kc2, kc2, tables, lens, 0.1, out)
    assert st == pa.PA_ERR_INVALID_ARG
