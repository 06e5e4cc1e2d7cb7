"""Copy-on-write on the GPU: pa_copy_blocks against the oracle's copy, and a full fork / diverge /
decode scenario driven by the host allocator, against the oracle chain and against private copies."""
import numpy as np
import pytest
import torch

import oracle
import synth
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

import gpu_harness as H  # noqa: E402
from oracle_pins import words  # noqa: E402


def _pool(NB, Hkv, bs, d, dtype):
    kc = torch.empty((NB, Hkv, bs, d), dtype=dtype, device=H.DEV)
    vc = torch.empty_like(kc)
    return kc, vc


def test_copy_blocks_bit_exact():
    rng = np.random.default_rng(1)
    NB, Hkv, bs, d = 50, 8, 16, 128
    hk = words(rng, (NB, Hkv, bs, d), synth.BF16)
    hv = words(rng, (NB, Hkv, bs, d), synth.BF16)
    kc = torch.from_numpy(hk.view(np.int16)).to(H.DEV).view(torch.bfloat16)
    vc = torch.from_numpy(hv.view(np.int16)).to(H.DEV).view(torch.bfloat16)
    pool = pa.Pool(NB, bs, Hkv, d, torch.bfloat16, max_context_len=512, k_cache=kc, v_cache=vc)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int32)     # distinct sources and targets
    pa.copy_blocks(pool, torch.from_numpy(pairs).to(H.DEV), kc, vc)
    assert pool.check() == pa.PA_OK
    oracle.copy_blocks(hk, hv, pairs)
    assert np.array_equal(H.pool_words(kc), hk) and np.array_equal(H.pool_words(vc), hv)


@pytest.mark.parametrize("dt", [synth.FP16, synth.BF16])
def test_fork_diverge_decode(dt):
    """A 40-token prompt, forked into 4 samples that each append their own tokens (the shared, partly
    filled block is copied before the first write): decode == oracle chain, and bit-identical to the
    same samples written into private blocks from scratch."""
    rng = np.random.default_rng(2)
    tdt = H.TORCH_DT[dt]
    NB, Hkv, bs, d, Hq = 64, 8, 16, 128, 32
    A = pa.BlockAllocator(NB, bs)
    kc, vc = _pool(NB, Hkv, bs, d, tdt)
    from synth import device as sdev
    sdev.fill_word(kc, synth.NAN16[dt])
    sdev.fill_word(vc, synth.NAN16[dt])
    hk = np.full((NB, Hkv, bs, d), synth.NAN16[dt], np.uint16)
    hv = hk.copy()
    pool = pa.Pool(NB, bs, Hkv, d, tdt, max_seqs=4, max_q_heads=Hq, max_context_len=512, k_cache=kc, v_cache=vc)
    stride = 12                                              # room for 40 + 90 tokens

    def dev_words(w):
        return torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).to(H.DEV).view(tdt)

    def write(k, v, slots):
        pool.cache_write(dev_words(k), dev_words(v), torch.from_numpy(slots).to(H.DEV), kc, vc)
        oracle.cache_write(hk, hv, k, v, slots)

    prompt_k, prompt_v = words(rng, (40, Hkv, d), dt), words(rng, (40, Hkv, d), dt)
    base = np.full(stride, -1, np.int32)
    slots, L, _ = A.append(base, 0, 40)
    write(prompt_k, prompt_v, slots)
    for _ in range(3):
        A.fork(base[:3])
    rows, lens, logical = [], [], []
    for i, n_new in enumerate([1, 7, 30, 90]):
        row = base.copy()
        slots, Ln, pair = A.append(row, 40, n_new)
        if pair is not None:
            pa.copy_blocks(pool, torch.tensor([pair], dtype=torch.int32, device=H.DEV), kc, vc)
            oracle.copy_blocks(hk, hv, [pair])
        nk, nv = words(rng, (n_new, Hkv, d), dt), words(rng, (n_new, Hkv, d), dt)
        write(nk, nv, slots)
        rows.append(row)
        lens.append(Ln)
        logical.append((np.concatenate([prompt_k, nk]), np.concatenate([prompt_v, nv])))
    assert pool.check() == pa.PA_OK
    # the device pool equals the oracle's pool word for word
    assert np.array_equal(H.pool_words(kc), hk) and np.array_equal(H.pool_words(vc), hv)
    tables = np.stack(rows)
    lens = np.array(lens, np.int32)
    q = words(rng, (4, 1, Hq, d), dt)
    scale = float(np.float32(1 / np.sqrt(d)))
    out = pool.decode(dev_words(q), torch.from_numpy(tables).to(H.DEV), torch.from_numpy(lens).to(H.DEV), scale,
                      k_cache=kc, v_cache=vc)
    ref, _ = oracle.paged_attention(q, hk, hv, tables, lens, dt, scale)
    H.assert_close(out, ref, "fork/diverge")
    # same samples in private blocks written from scratch
    kc2, vc2 = _pool(NB, Hkv, bs, d, tdt)
    pool2 = pa.Pool(NB, bs, Hkv, d, tdt, max_seqs=4, max_q_heads=Hq, max_context_len=512, k_cache=kc2, v_cache=vc2)
    priv = np.full((4, stride), -1, np.int32)
    nxt = 0
    for i in range(4):
        nb = -(-int(lens[i]) // bs)
        priv[i, :nb] = np.arange(nxt, nxt + nb)
        nxt += nb
        t = np.arange(lens[i])
        k, v = logical[i]
        pool2.cache_write(dev_words(k), dev_words(v),
                          torch.from_numpy(priv[i, t // bs].astype(np.int64) * bs + t % bs).to(H.DEV), kc2, vc2)
    out2 = pool2.decode(dev_words(q), torch.from_numpy(priv).to(H.DEV), torch.from_numpy(lens).to(H.DEV), scale,
                        k_cache=kc2, v_cache=vc2)
    assert torch.equal(out, out2)
