"""The C-ABI library without a GPU: it builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching the device."""
import ctypes as C
import os
import re
import subprocess

import pytest

from paged_kv_cache_223_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build_cuda()
    from paged_kv_cache_223_gb300 import pagedattn as pa
    return pa


def declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert {"pa_pool_create", "pa_cache_write", "pa_decode", "pa_destroy"} <= names
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pa_\w+)", out))
    assert names <= exported, names - exported
    handle = C.CDLL(lib.LIB_PATH)
    for n in names:
        getattr(handle, n)


def test_status_strings(lib):
    for s in range(7):
        assert lib.status_string(s) and lib.status_string(s) != "unknown status"


def test_host_validation_without_gpu(lib):
    good = dict(num_blocks=64, block_size=16, num_kv_heads=2, head_dim=64, dtype=0, device=0, partition_tokens=0,
                max_seqs=4, max_q_heads=8, max_q_len=1, max_context_len=256, k_cache=None, v_cache=None,
                kv_format=0)
    bad = [dict(block_size=8), dict(head_dim=96), dict(num_blocks=0), dict(dtype=5), dict(partition_tokens=24),
           dict(max_q_len=9), dict(k_cache=16), dict(max_seqs=0), dict(device=-1), dict(kv_format=3),
           dict(kv_format=1, head_dim=64)]
    for b in bad:
        st = lib.pool_create_status(**{**good, **b})
        assert st in (lib.PA_ERR_INVALID_ARG, lib.PA_ERR_UNSUPPORTED), b
    L = lib.lib()
    assert L.pa_decode(None, None, None, None, None, 1, None, 1, 8, 1, 0.1, None, None) == lib.PA_ERR_INVALID_ARG
    assert L.pa_prefill(None, None, None, None, None, 1, None, 1, 8, 16, 0.1, None, None) == lib.PA_ERR_INVALID_ARG
    assert L.pa_decode_shared_prefix(None, None, None, None, None, 1, None, 1, 8, 1, 0.1, 512, None,
                                     None) == lib.PA_ERR_INVALID_ARG
    assert L.pa_cache_write(None, None, None, None, 1, None, None, None) == lib.PA_ERR_INVALID_ARG
    assert L.pa_pool_check(None, None) == lib.PA_ERR_INVALID_ARG
    L.pa_destroy(None)
