"""pa_decode_noalloc, the allocation-free decode, against the oracle and against pa_decode.

Callers that cannot allocate device memory (a host runtime that owns every device
allocation, or a loop that must not make cudaMalloc's synchronising call) use
pa_decode_noalloc, whose scratch is a static device array inside the library. Its
outputs must match the fp64 oracle and pa_decode within the suite's tolerance, call
after call, even though every call reuses the same scratch array; a call must not
change the device's free memory; a request just under the array's size must run and
one just over it must be refused; and a call whose kernels flag bad input must not
hand back stale numbers.
"""
import numpy as np
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
    oracle_out, _, _ = H.oracle_reference(wl, 0)
    return dict(wl=wl, kc=kc, vc=vc, q=q, tables=tables, lens=lens, ref=ref, oracle=oracle_out, pool=pool)


def _noalloc(c, out=None):
    out = torch.empty_like(c["q"]) if out is None else out
    st = pa.decode_noalloc(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], c["wl"].scale, out,
                           partition_tokens=c["wl"].partition_tokens)
    assert st == pa.PA_OK, pa.status_string(st)
    return out


def _check(out, c, what):
    H.assert_close(out, c["oracle"], what + " vs the oracle")
    H.assert_close(out, H.to_f64(c["ref"]), what + " vs pa_decode")


def test_noalloc_matches_oracle_and_pa_decode_on_consecutive_calls():
    # long fp16 context: 64 partitions of 512 tokens share the static scratch
    a = _case(synth.custom_workload([32768, 1000], 32, 8, 128, 32, 1, synth.FP16, tag=91))
    # bf16 shared prefix + 5-token verify, 256-token partitions
    b = _case(synth.custom_workload([1024 + 300, 1024 + 45, 1024 + 512], 32, 8, 128, 16, 5, synth.BF16,
                                    prefix_tokens=1024, partition_tokens=256, tag=92))
    for i, c in enumerate((a, b, a, a, b)):
        out = _noalloc(c)
        torch.cuda.synchronize()
        _check(out, c, f"pa_decode_noalloc call {i}")


def test_noalloc_changes_no_device_memory():
    """Warm-up call, then 20 calls into preallocated outputs: the device's free memory is unchanged."""
    c = _case(synth.custom_workload([5000, 700, 64], 32, 8, 128, 16, 1, synth.BF16, tag=94))
    out = torch.empty_like(c["q"])
    _noalloc(c, out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        _noalloc(c, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    _check(out, c, "pa_decode_noalloc after 21 calls")


def _boundary_workload():
    # 63 sequences x 32 query heads x 32 partitions (a table of 1024 blocks of 16 tokens, 512-token
    # partitions): 64512 partial slots = 33,030,144 + 516,096 bytes, plus the 256-byte status word:
    # 7,936 bytes under the 32 MiB array. Contexts are short: the table width alone sets the scratch.
    rng = np.random.default_rng(95)
    lens = [int(x) for x in rng.integers(1, 700, size=63)]
    return synth.custom_workload(lens, 32, 8, 128, 16, 1, synth.FP16, tag=95, stride=1024)


def _need(B, Hq, P, d, q_len=1):
    slots = B * q_len * Hq * P
    return 256 + -(-slots * d * 4 // 256) * 256 + slots * 8


def test_noalloc_at_the_scratch_limit_and_one_sequence_past_it():
    wl = _boundary_workload()
    assert wl.stride * wl.bs // 512 == 32
    assert _need(63, 32, 32, 128) <= pa.NOALLOC_SCRATCH_BYTES < _need(64, 32, 32, 128)
    c = _case(wl)
    out = _noalloc(c)
    torch.cuda.synchronize()
    _check(out, c, "63 sequences, just under the scratch limit")
    # the same request with one more sequence (batch size is the only change): refused before any launch
    q64 = torch.cat([c["q"], c["q"][:1]])
    t64 = torch.cat([c["tables"], c["tables"][:1]])
    l64 = torch.cat([c["lens"], c["lens"][:1]])
    out64 = torch.full_like(q64, 7.0)
    st = pa.decode_noalloc(q64, c["kc"], c["vc"], t64, l64, wl.scale, out64, partition_tokens=512)
    assert st == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out64 == 7.0).all()), "a refused call wrote its output"


def test_noalloc_flags_bad_input_with_nan_and_recovers():
    """An out-of-range block id is clamped on the device (no fault); with no status word to return, the call
    marks its whole output NaN. The next valid call clears the flag and returns correct numbers again."""
    c = _case(synth.custom_workload([900, 2000], 16, 4, 128, 16, 1, synth.FP16, tag=96))
    bad = c["tables"].clone()
    bad[1, 3] = c["wl"].num_blocks + 5
    out = torch.empty_like(c["q"])
    st = pa.decode_noalloc(c["q"], c["kc"], c["vc"], bad, c["lens"], c["wl"].scale, out)
    assert st == pa.PA_OK
    torch.cuda.synchronize()
    assert bool(torch.isnan(out.float()).all()), "a flagged call must not return numbers"
    out2 = _noalloc(c)
    torch.cuda.synchronize()
    _check(out2, c, "valid call after a flagged one")
