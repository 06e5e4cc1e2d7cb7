"""GPU invariants that need no oracle value: placement invariance, shared == duplicated blocks,
run-to-run determinism, NaN tails, and the device-side bounds flags."""
import numpy as np
import pytest
import torch

import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402


def _decode(wl, partition_tokens=0):
    pool, kc, vc, q, tables, lens = H.build_device(wl, partition_tokens=partition_tokens)
    out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    return out, (pool, kc, vc, q, tables, lens)


def test_placement_invariance_bitwise():
    """The same logical K/V under two different physical shuffles give bit-identical outputs."""
    a = synth.custom_workload([900, 37, 2048], 32, 8, 128, 16, 1, synth.FP16, tag=31)
    b = synth.custom_workload([900, 37, 2048], 32, 8, 128, 16, 1, synth.FP16, tag=31)
    perm = synth.permutation(1234, 5, b.num_blocks)
    b.block_tables = synth._tables_from_perm(perm, b.context_lens, b.bs, b.stride)
    assert not np.array_equal(a.block_tables, b.block_tables)
    oa, _ = _decode(a)
    ob, _ = _decode(b)
    assert torch.equal(oa, ob)


def test_shared_prefix_equals_duplicated_bitwise():
    """Tables naming one physical copy of a prefix == tables naming private copies of it."""
    shared = synth.custom_workload([1024 + 40, 1024 + 300, 1024 + 77], 32, 8, 128, 16, 5, synth.BF16,
                                   prefix_tokens=1024, tag=41)
    priv = synth.custom_workload([1024 + 40, 1024 + 300, 1024 + 77], 32, 8, 128, 16, 5, synth.BF16,
                                 prefix_tokens=1024, tag=41)
    # private copies: every sequence gets its own 64 prefix blocks (same values: the prefix stream)
    NB = priv.num_blocks + 64 * priv.B
    perm = synth.permutation(77, 3, NB)
    tables = np.full_like(priv.block_tables, -1)
    pos = 0
    for b in range(priv.B):
        nb = -(-int(priv.context_lens[b]) // 16)
        tables[b, :nb] = perm[pos:pos + nb]
        pos += nb
    priv.block_tables, priv.num_blocks = tables, NB
    # write the prefix into each private copy: fill() writes the prefix from sequence 0's table only,
    # so add the other sequences' prefix writes explicitly.
    out_s, _ = _decode(shared)
    kc, vc = H.alloc_caches(priv)
    pool = H.make_pool(priv, 0, kc, vc)
    H.fill(pool, priv, 0, kc, vc, new_only=False)
    for b in range(1, priv.B):
        t = np.arange(1024)
        rows = torch.from_numpy(t.astype(np.int64)).to(H.DEV)
        import synth.device as sdev
        k, v = sdev.kv_rows(priv, 0, synth.K_KP, rows, H.DEV)
        pool.cache_write(k, v, torch.from_numpy(priv.slots(b, t)).to(H.DEV), kc, vc)
    H.fill(pool, priv, 0, kc, vc, new_only=True)
    q, tables_d, lens = H.device_inputs(priv, 0)
    out_p = pool.decode(q, tables_d, lens, priv.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    assert torch.equal(out_s, out_p)


def test_inputs_written_just_before_the_call_are_seen():
    """A kernel that writes the decode's query right before the call on the same stream, with no synchronisation in
    between, is seen: the decode kernels may be launched while it runs (programmatic stream serialization), but they
    wait for it before reading. A long kernel ahead of the write keeps it pending when the decode is launched."""
    for wl in (synth.custom_workload([3000, 700, 4100], 64, 8, 128, 16, 1, synth.FP16, tag=51),   # 8 rows: decode + merge
               synth.custom_workload([2000, 900], 32, 8, 128, 16, 5, synth.BF16, tag=52)):      # 20 rows: tensor-core kernel
        pool, kc, vc, q, tables, lens = H.build_device(wl)
        q2 = torch.flip(q, dims=[-1]).contiguous()
        ref = pool.decode(q2, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
        torch.cuda.synchronize()
        qq = q.clone()
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        qq.copy_(q2)
        out = pool.decode(qq, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
        torch.cuda.synchronize()
        assert pool.check() == pa.PA_OK
        assert not torch.equal(ref, pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc))
        assert torch.equal(out, ref)


def test_deterministic_run_to_run():
    wl = synth.workload(5, batch=2)
    out, (pool, kc, vc, q, tables, lens) = _decode(wl)
    for _ in range(3):
        again = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
        assert torch.equal(out, again)


def test_nan_tails_do_not_leak():
    """Every slot past each context holds NaN (the fill word); outputs stay finite."""
    wl = synth.custom_workload([17, 33, 250, 511], 16, 4, 128, 32, 1, synth.FP16, tag=51)
    out, _ = _decode(wl)
    assert torch.isfinite(out.float()).all()


def test_bad_block_id_is_flagged_not_faulted():
    wl = synth.custom_workload([100, 60], 8, 2, 64, 16, 1, synth.FP16, tag=61)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    bad = tables.clone()
    bad[1, 2] = wl.num_blocks + 5          # outside the pool
    pool.decode(q, bad, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_ERR_DEVICE_BOUNDS
    assert pool.check() == pa.PA_OK        # read-and-clear
    bad_lens = lens.clone()
    bad_lens[0] = wl.stride * wl.bs + 1    # longer than the table holds
    pool.decode(q, tables, bad_lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_ERR_DEVICE_BOUNDS


def test_bad_slot_is_flagged_and_skipped():
    wl = synth.custom_workload([40], 8, 2, 64, 16, 1, synth.FP16, tag=62)
    kc, vc = H.alloc_caches(wl)
    pool = H.make_pool(wl, 0, kc, vc)
    before = H.pool_words(kc).copy()
    k = torch.ones((2, 2, 64), dtype=torch.float16, device=H.DEV)
    slots = torch.tensor([wl.num_blocks * wl.bs + 3, -1], dtype=torch.int64, device=H.DEV)
    pool.cache_write(k, k, slots, kc, vc)
    assert pool.check() == pa.PA_ERR_DEVICE_BOUNDS
    assert np.array_equal(H.pool_words(kc), before)


def test_host_side_argument_errors():
    wl = synth.custom_workload([40], 8, 2, 64, 16, 1, synth.FP16, tag=63)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    L = pa.lib()
    out = torch.empty_like(q)
    # Hq not a multiple of Hkv
    st = L.pa_decode(pool.handle, q.data_ptr(), None, None, tables.data_ptr(), tables.shape[1], lens.data_ptr(), 1, 7,
                     1, 0.125, out.data_ptr(), None)
    assert st == pa.PA_ERR_INVALID_ARG
    # misaligned q
    st = L.pa_decode(pool.handle, q.data_ptr() + 2, None, None, tables.data_ptr(), tables.shape[1], lens.data_ptr(),
                     1, 8, 1, 0.125, out.data_ptr(), None)
    assert st == pa.PA_ERR_INVALID_ARG
    # more rows per KV head than supported: G = 8, q_len = 5 -> 40 rows
    st = L.pa_decode(pool.handle, q.data_ptr(), None, None, tables.data_ptr(), tables.shape[1], lens.data_ptr(), 1,
                     16, 5, 0.125, out.data_ptr(), None)
    assert st in (pa.PA_ERR_INVALID_ARG, pa.PA_ERR_UNSUPPORTED)


def test_bounded_wait_times_out_and_context_survives():
    """A wait that nothing completes gives up after its limit, reports PA_ERR_TIMEOUT, and the next decode
    on the same context still runs and is correct."""
    wl = synth.custom_workload([300, 77], 16, 4, 128, 16, 1, synth.FP16, tag=64)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    pool.selftest_wait(2_000_000)           # 2 ms
    assert pool.check() == pa.PA_ERR_TIMEOUT
    assert pool.check() == pa.PA_OK
    out = pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc)
    assert pool.check() == pa.PA_OK
    ref, _, _ = H.oracle_reference(wl, 0)
    H.assert_close(out, ref, "decode after a timed-out wait")


def test_binding_rejects_inconsistent_shapes():
    """The library sees only pointers; the binding refuses shapes that would make it read or write past a buffer."""
    wl = synth.custom_workload([40, 50], 8, 2, 64, 16, 1, synth.FP16, tag=64)
    pool, kc, vc, q, tables, lens = H.build_device(wl)
    bad = [
        dict(out=torch.empty((1,) + tuple(q.shape[1:]), dtype=q.dtype, device=q.device)),   # out smaller than q
    ]
    for kw in bad:
        with pytest.raises(ValueError):
            pool.decode(q, tables, lens, wl.scale, k_cache=kc, v_cache=vc, **kw)
    with pytest.raises(ValueError):                                   # one context length for two sequences
        pool.decode(q, tables, lens[:1], wl.scale, k_cache=kc, v_cache=vc)
    with pytest.raises(ValueError):                                   # one table row for two sequences
        pool.decode(q, tables[:1], lens, wl.scale, k_cache=kc, v_cache=vc)
    with pytest.raises(ValueError):                                   # head dim other than the pool's
        pool.decode(torch.zeros(q.shape[:3] + (128,), dtype=q.dtype, device=q.device), tables, lens, wl.scale)
    with pytest.raises(ValueError):                                   # only one of the two caches
        pool.decode(q, tables, lens, wl.scale, k_cache=kc)
    k = torch.zeros((3, 2, 64), dtype=torch.float16, device=H.DEV)
    with pytest.raises(ValueError):                                   # fewer slots than rows
        pool.cache_write(k, k, torch.zeros(2, dtype=torch.int64, device=H.DEV))
    p = torch.full((2, 3, 10), 0.1, device=H.DEV)
    qd = torch.full((2, 1, 10), 0.1, device=H.DEV)                     # K = 1 draft where p implies 2
    d = torch.zeros((2, 2), dtype=torch.int32, device=H.DEV)
    u = torch.zeros((2, 2), device=H.DEV)
    with pytest.raises(ValueError):
        pa.spec_verify(p, qd, d, u, torch.zeros(2, device=H.DEV))
    with pytest.raises(ValueError):                                   # pairs must be [n, 2]
        pa.copy_blocks(pool, torch.zeros((4, 3), dtype=torch.int32, device=H.DEV))
    assert pool.check() == pa.PA_OK
