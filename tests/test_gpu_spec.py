"""Speculative rejection sampling on the GPU (pa_spec_verify) against the oracle.

The accept decisions are fp32 comparisons taken the same way on both sides, so the number of kept
drafts and the kept tokens must match exactly. The drawn token is an inverse CDF summed in fp64 in a
different order on each side; it must match, or sit on a CDF boundary (checked with the oracle's sums)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_223_gb300 import pagedattn as pa

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _dist(rng, shape, sharp=3.0):
    x = rng.random(shape) ** sharp
    return (x / x.sum(-1, keepdims=True)).astype(np.float32)


def _case(seed, B, K, V, agree=0.0):
    rng = np.random.default_rng(seed)
    p = _dist(rng, (B, K + 1, V))
    q = _dist(rng, (B, K, V))
    if agree:
        q = ((1 - agree) * q + agree * p[:, :K]).astype(np.float32)
    draft = np.empty((B, K), np.int32)
    for b in range(B):
        for i in range(K):
            w = q[b, i].astype(np.float64)
            draft[b, i] = rng.choice(V, p=w / w.sum())
    u = rng.random((B, K)).astype(np.float32)
    v = rng.random(B).astype(np.float32)
    return p, q, draft, u, v


def _check(p, q, draft, u, v):
    t = lambda a: torch.from_numpy(a).to(DEV)
    out, n = pa.spec_verify(t(p), t(q), t(draft), t(u), t(v))
    out, n = out.cpu().numpy(), n.cpu().numpy()
    ref, rn = oracle.spec_verify(p, q, draft, u, v)
    assert np.array_equal(n, rn)
    B, K1, V = p.shape
    boundary = 0
    for b in range(B):
        k = n[b] - 1
        assert np.array_equal(out[b, :k], ref[b, :k]) and (out[b, k + 1:] == -1).all()
        if out[b, k] != ref[b, k]:
            # must be a boundary case of the fp64 inverse CDF
            row = k if k < K1 - 1 else K1 - 1
            w = np.maximum(p[b, row].astype(np.float64) - (q[b, row].astype(np.float64) if k < K1 - 1 else 0), 0)
            c = np.cumsum(w)
            target = float(v[b]) * c[-1]
            j = out[b, k]
            assert abs(c[j] - target) < 1e-9 * c[-1] or abs((c[j - 1] if j else 0) - target) < 1e-9 * c[-1]
            boundary += 1
    assert boundary <= max(1, B // 1000)
    return out, n


@pytest.mark.parametrize("B,K,V,agree", [(64, 5, 1000, 0.0), (64, 5, 1000, 0.9), (7, 1, 3, 0.5), (16, 0, 50, 0.0),
                                         (32, 4, 128256, 0.8)])
def test_matches_oracle(B, K, V, agree):
    _check(*_case(B * 1000 + K + V, B, K, V, agree))


def test_lossless_in_distribution():
    """With a fixed target p and draft q, the first emitted token over many draws follows p."""
    rng = np.random.default_rng(5)
    V, B = 8, 200_000
    p1 = _dist(rng, (V,))
    q1 = _dist(rng, (V,))
    p = np.broadcast_to(np.stack([p1, _dist(rng, (V,))]), (B, 2, V)).copy()
    q = np.broadcast_to(q1, (B, 1, V)).copy()
    w = q1.astype(np.float64)
    draft = rng.choice(V, size=(B, 1), p=w / w.sum()).astype(np.int32)
    u = rng.random((B, 1)).astype(np.float32)
    v = rng.random(B).astype(np.float32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    out, n = pa.spec_verify(t(p), t(q), t(draft), t(u), t(v))
    freq = np.bincount(out[:, 0].cpu().numpy(), minlength=V) / B
    sigma = np.sqrt(p1 * (1 - p1) / B)
    assert (np.abs(freq - p1) < 5 * sigma + 1e-4).all(), (freq, p1)
