"""Speculative rejection sampling on the GPU (pa_spec_verify) against the oracle.

The accept decisions are fp32 comparisons taken the same way on both sides, so the number of kept
drafts and the kept tokens must match exactly. The drawn token is an inverse CDF, summed in fp64 by the
oracle and in float pairs (about 44 significant bits, another order) by the kernel; it must match, or sit
on a CDF boundary (checked with the oracle's fp64 sums)."""
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
                                         (32, 4, 128256, 0.8),
                                         (16, 40, 1000, 0.98),   # accept tests past the first 32 drafts
                                         (8, 2, 1, 0.0)])        # one-token vocabulary
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


def test_residual_without_mass_draws_from_target():
    """p == q with zeros; every draft sits on a zero-probability token, so it is rejected at position 0 and
    max(0, p - q) has no mass: the token is drawn from p itself."""
    rng = np.random.default_rng(11)
    B, K, V = 48, 3, 4099
    p = _dist(rng, (B, K + 1, V))
    p[:, :, ::3] = 0
    p /= p.sum(-1, keepdims=True)
    q = p[:, :K].copy()
    draft = np.zeros((B, K), np.int32)                      # token 0 has zero probability
    u = rng.random((B, K)).astype(np.float32)
    v = rng.random(B).astype(np.float32)
    out, n = _check(p, q, draft, u, v)
    assert (n == 1).all()
    assert (p[np.arange(B), 0, out[:, 0]] > 0).all()


@pytest.mark.parametrize("vv", [0.0, np.nextafter(np.float32(1), np.float32(0))])
def test_extreme_uniforms(vv):
    """v = 0 draws the first token of positive weight; v just below 1 puts the target next to the total,
    where the kernel's sums may round past it: the token must still match (or sit on a boundary) and
    carry positive weight."""
    B, K, V = 32, 2, 128256
    p, q, draft, u, _ = _case(99, B, K, V, agree=0.5)
    v = np.full(B, vv, np.float32)
    out, n = _check(p, q, draft, u, v)
    for b in range(B):
        k = n[b] - 1
        row = k if k < K else K
        w = np.maximum(p[b, row].astype(np.float64) - (q[b, row].astype(np.float64) if k < K else 0), 0)
        if not w.any():
            w = np.maximum(p[b, row].astype(np.float64), 0)
        assert w[out[b, k]] > 0
        if vv == 0.0:
            assert out[b, k] == np.flatnonzero(w > 0)[0]


@pytest.mark.parametrize("V", [50257, 129, 1 << 17])
def test_sparse_rows(V):
    """Mass on a few scattered tokens (most segments of the row are empty), odd and power-of-two sizes."""
    rng = np.random.default_rng(V)
    B, K = 24, 4
    p = np.zeros((B, K + 1, V), np.float32)
    q = np.zeros((B, K, V), np.float32)
    for b in range(B):
        for i in range(K + 1):
            idx = rng.choice(V, size=min(V, 7), replace=False)
            p[b, i, idx] = rng.random(len(idx)) + 0.01
        for i in range(K):
            idx = rng.choice(V, size=min(V, 7), replace=False)
            q[b, i, idx] = rng.random(len(idx)) + 0.01
    p /= p.sum(-1, keepdims=True)
    q /= q.sum(-1, keepdims=True)
    draft = np.stack([[rng.choice(V, p=q[b, i].astype(np.float64) / q[b, i].astype(np.float64).sum()) for i in range(K)]
                      for b in range(B)]).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    v = rng.random(B).astype(np.float32)
    _check(p, q, draft, u, v)
