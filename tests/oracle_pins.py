"""Pins of the fp64 oracle to things other than itself.

Each pin_* function raises AssertionError when the oracle (whichever build
`oracle.use()` routes to) disagrees with what the pages or the mathematics fix:
the pages' worked numbers (tests/golden), closed forms, special cases that reduce
to a library routine (torch's fp64 scaled_dot_product_attention, numpy's fp16
decoding), and invariants. The same functions run against the real oracle and
against deliberately mutated builds (tests/test_oracle_pins.py), so each
plausible mistake is shown to fail at least one pin.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FP16, BF16 = oracle.FP16, oracle.BF16


def _rng(seed):
    return np.random.default_rng(seed)


def words(rng, shape, dtype, sigma=1.0, mean=0.0):
    """Random 16-bit words of N(mean, sigma) values (test data, numpy RNG)."""
    x = (rng.standard_normal(shape) * sigma + mean).astype(np.float32)
    return synth.f32_to_bits16(x, dtype)


def lib_decode(w, dtype):
    """Library decode of 16-bit words to float64 (numpy's float16 / a float32 bit view)."""
    w = np.asarray(w, dtype=np.uint16)
    if dtype == FP16:
        return w.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return (w.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def read_mapping(name):
    rows, bs = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("block_size"):
                bs = int(line.split()[1])
                continue
            a, b, p = (int(x) for x in line.split())
            rows.append((a, b, p))
    return bs, rows


def sdpa_reference(q, kc, vc, dtype, scale):
    """torch fp64 SDPA on decoded inputs: causal self-attention over all L positions with the
    q_len given query rows placed at the last q_len positions (other positions get zero queries);
    returns those last q_len rows [q_len, Hq, d]."""
    q_len, Hq, d = q.shape
    L, Hkv, _ = kc.shape
    qf = np.zeros((L, Hq, d))
    qf[L - q_len:] = lib_decode(q, dtype)
    Q = torch.from_numpy(qf).permute(1, 0, 2)[None]
    K = torch.from_numpy(lib_decode(kc, dtype)).permute(1, 0, 2)[None]
    V = torch.from_numpy(lib_decode(vc, dtype)).permute(1, 0, 2)[None]
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=float(scale),
                                                         enable_gqa=(Hq != Hkv))
    return O[0].permute(1, 0, 2).numpy()[L - q_len:]


# ----------------------------------------------------------------------------- pins

def pin_decode_fp16():
    """All 65536 fp16 words decode as numpy's float16 does (NaNs where numpy has NaN)."""
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    sample = np.concatenate([w[::97], np.array([0, 1, 0x3FF, 0x400, 0x3C00, 0x7BFF, 0x7C00, 0x8001, 0xFC00,
                                                0x7E00, 0x0200], dtype=np.uint16)])
    got = oracle.decode16(sample, FP16)
    ref = lib_decode(sample, FP16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_decode_bf16():
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    sample = np.concatenate([w[::89], np.array([0, 1, 0x3F80, 0x7F7F, 0x7F80, 0xFF80, 0x7FC0, 0x0080],
                                               dtype=np.uint16)])
    got = oracle.decode16(sample, BF16)
    ref = lib_decode(sample, BF16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _tagged_pool(NB, Hkv, bs, d):
    """Pool whose every element encodes (block, head, offset, dim) - readable after a gather."""
    blk, h, off, k = np.meshgrid(np.arange(NB), np.arange(Hkv), np.arange(bs), np.arange(d), indexing="ij")
    return ((blk * 1000003 + h * 7919 + off * 131 + k) % 65521).astype(np.uint16), blk, off


def _pin_mapping(fixture):
    bs, rows = read_mapping(fixture)
    Hkv, d = 2, 8
    NB = max(p for _, _, p in rows) + 1
    table = np.full(8, -1, dtype=np.int32)
    for a, b, p in rows:
        table[a // bs] = p
    L = rows[-1][1] + 1
    pool, _, _ = _tagged_pool(NB, Hkv, bs, d)
    got = oracle.gather(pool, table, L)
    for a, b, p in rows:
        for t in range(a, b + 1):
            assert np.array_equal(got[t], pool[p, :, t - a, :]), (fixture, t)
    # the cache write with the slot the figure implies puts token t where the gather finds it
    kp = np.zeros((NB, Hkv, bs, d), dtype=np.uint16)
    vp = np.zeros_like(kp)
    toks = np.arange(L)
    slot = np.array([next(p for a, b, p in rows if a <= t <= b) * bs + (t % bs) for t in toks], dtype=np.int64)
    kn = np.arange(L * Hkv * d, dtype=np.uint16).reshape(L, Hkv, d) + 1
    vn = kn + 7
    oracle.cache_write(kp, vp, kn, vn, slot)
    assert np.array_equal(oracle.gather(kp, table, L), kn)
    assert np.array_equal(oracle.gather(vp, table, L), vn)


def pin_mapping_yangyu():
    _pin_mapping("block_table_figure_yangyu.txt")
    # token 20 -> logical block 1 -> page 2, offset 4 -> slot 36
    bs, rows = read_mapping("block_table_figure_yangyu.txt")
    kp = np.zeros((20, 1, bs, 4), dtype=np.uint16)
    vp = np.zeros_like(kp)
    oracle.cache_write(kp, vp, np.full((1, 1, 4), 9, np.uint16), np.full((1, 1, 4), 5, np.uint16),
                       np.array([36]))
    assert (kp[2, 0, 4] == 9).all() and (vp[2, 0, 4] == 5).all()
    assert int(kp.astype(np.int64).sum()) == 36


def pin_mapping_tanhdev():
    _pin_mapping("block_table_diagram_tanhdev.txt")


def pin_kv_size_closed_form():
    """Writing one token into every layer's pool changes exactly 4*L*Hkv*d bytes (327,680 for 70B)."""
    with open(os.path.join(GOLDEN, "kv_size_closed_form.txt")) as f:
        vals = [l.split() for l in f if l.strip() and not l.startswith("#")][0]
    layers, Hkv, d, eb, per_token = (int(x) for x in vals)
    bs, NB = 16, 2
    changed = 0
    for layer in range(layers):
        kp = np.zeros((NB, Hkv, bs, d), dtype=np.uint16)
        vp = np.zeros_like(kp)
        kn = np.full((1, Hkv, d), 0x3C00, np.uint16)
        oracle.cache_write(kp, vp, kn, kn, np.array([bs + 3]))
        changed += int((kp != 0).sum() + (vp != 0).sum()) * eb
    assert changed == per_token, changed


def pin_sdpa_contiguous():
    """Identity placement: oracle == torch fp64 SDPA (causal, GQA, several shapes and dtypes)."""
    rng = _rng(1)
    cases = [(1, 1, 1, 16, FP16, 1), (37, 4, 2, 16, FP16, 1), (64, 8, 2, 64, FP16, 1), (100, 8, 8, 32, BF16, 1),
             (23, 6, 3, 8, BF16, 5), (70, 32, 8, 16, FP16, 5), (5, 4, 1, 8, FP16, 5), (129, 12, 4, 64, BF16, 3)]
    for L, Hq, Hkv, d, dt, ql in cases:
        q = words(rng, (ql, Hq, d), dt)
        kc = words(rng, (L, Hkv, d), dt)
        vc = words(rng, (L, Hkv, d), dt)
        scale = float(np.float32(1 / np.sqrt(d)))
        got = oracle.attention(q, kc, vc, dt, scale)
        ref = sdpa_reference(q, kc, vc, dt, scale)
        assert np.allclose(got, ref, rtol=1e-10, atol=1e-12), (L, Hq, Hkv, d, dt, ql, np.abs(got - ref).max())


def pin_paged_equals_contiguous_under_permutation():
    """Any shuffle of physical placement gives bit-identical oracle outputs."""
    rng = _rng(2)
    B, Hq, Hkv, d, bs, dt = 3, 8, 2, 16, 16, FP16
    lens = np.array([5, 40, 77], dtype=np.int32)
    outs = []
    q = words(rng, (B, 1, Hq, d), dt)
    kn = [words(rng, (int(L), Hkv, d), dt) for L in lens]
    vn = [words(rng, (int(L), Hkv, d), dt) for L in lens]
    for perm_seed in (10, 11, 12):
        NB = 12
        perm = _rng(perm_seed).permutation(NB)
        tables = np.full((B, 5), -1, dtype=np.int32)
        pos = 0
        kp = np.full((NB, Hkv, bs, d), 0x7E00, np.uint16)
        vp = kp.copy()
        for b, L in enumerate(lens):
            nb = -(-int(L) // bs)
            tables[b, :nb] = perm[pos:pos + nb]
            pos += nb
            t = np.arange(L)
            oracle.cache_write(kp, vp, kn[b], vn[b], tables[b, t // bs].astype(np.int64) * bs + t % bs)
        out, _ = oracle.paged_attention(q, kp, vp, tables, lens, dt, 0.25)
        outs.append(out)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    for b, L in enumerate(lens):
        ref = oracle.attention(q[b], kn[b], vn[b], dt, 0.25)
        assert np.array_equal(outs[0][b], ref)


def pin_closed_forms():
    rng = _rng(3)
    dt, d, Hq, Hkv = FP16, 16, 4, 2
    # L = 1: the single value vector, exactly
    q = words(rng, (1, Hq, d), dt)
    kc = words(rng, (1, Hkv, d), dt)
    vc = words(rng, (1, Hkv, d), dt)
    out = oracle.attention(q, kc, vc, dt, 0.25)
    for h in range(Hq):
        assert np.array_equal(out[0, h], lib_decode(vc[0, h // 2], dt))
    # q = 0: the arithmetic mean of the attended values
    L = 57
    q0 = np.zeros((1, Hq, d), np.uint16)
    kc = words(rng, (L, Hkv, d), dt)
    vc = words(rng, (L, Hkv, d), dt)
    out = oracle.attention(q0, kc, vc, dt, 0.25)
    mean = lib_decode(vc, dt).mean(axis=0)
    for h in range(Hq):
        assert np.allclose(out[0, h], mean[h // 2], rtol=0, atol=1e-12)
    # constant V = c: c
    vconst = np.full((L, Hkv, d), 0x3E00, np.uint16)        # 1.5
    out = oracle.attention(words(rng, (1, Hq, d), dt), kc, vconst, dt, 0.25)
    assert np.allclose(out, 1.5, rtol=0, atol=1e-12)
    # one key with a huge score: exactly its value vector
    q = np.zeros((1, Hq, d), np.uint16)
    q[0, :, 0] = 0x5C00                                      # 256
    kc = np.zeros((L, Hkv, d), np.uint16)
    kc[31, :, 0] = 0x5C00
    out = oracle.attention(q, kc, vc, dt, 0.125)
    for h in range(Hq):
        assert np.array_equal(out[0, h], lib_decode(vc[31, h // 2], dt))


def pin_weights():
    """Softmax weights: non-negative, sum to 1, zero beyond each row's causal limit."""
    rng = _rng(4)
    L, Hq, Hkv, d, ql = 33, 4, 2, 8, 5
    q = words(rng, (ql, Hq, d), BF16)
    kc = words(rng, (L, Hkv, d), BF16)
    vc = words(rng, (L, Hkv, d), BF16)
    _, w = oracle.attention(q, kc, vc, BF16, 0.3, want_weights=True)
    assert (w >= 0).all()
    assert np.allclose(w.sum(-1), 1.0, rtol=0, atol=1e-12)
    for qi in range(ql):
        assert (w[qi, :, L - ql + qi + 1:] == 0).all()
        assert (w[qi, :, : L - ql + qi + 1] > 0).all()


def pin_gqa_is_mha_with_duplicated_heads():
    rng = _rng(5)
    L, Hq, Hkv, d, dt = 29, 12, 3, 16, BF16
    G = Hq // Hkv
    q = words(rng, (2, Hq, d), dt)
    kc = words(rng, (L, Hkv, d), dt)
    vc = words(rng, (L, Hkv, d), dt)
    a = oracle.attention(q, kc, vc, dt, 0.25)
    b = oracle.attention(q, np.repeat(kc, G, axis=1), np.repeat(vc, G, axis=1), dt, 0.25)
    assert np.array_equal(a, b)


def pin_verify_rows_are_decodes():
    """Row qi of a q_len = 5 verify equals a single-query decode over the first L - 5 + qi + 1 tokens."""
    rng = _rng(6)
    L, Hq, Hkv, d, dt, ql = 45, 8, 2, 16, FP16, 5
    q = words(rng, (ql, Hq, d), dt)
    kc = words(rng, (L, Hkv, d), dt)
    vc = words(rng, (L, Hkv, d), dt)
    full = oracle.attention(q, kc, vc, dt, 0.25)
    for qi in range(ql):
        n = L - ql + qi + 1
        one = oracle.attention(q[qi:qi + 1], kc[:n], vc[:n], dt, 0.25)
        assert np.array_equal(full[qi], one[0])


def pin_shared_prefix_equals_duplicated():
    """Tables sharing physical prefix blocks == tables with private copies of those blocks."""
    rng = _rng(7)
    B, Hq, Hkv, d, bs, dt, P = 3, 4, 2, 8, 16, BF16, 32
    suf = [7, 20, 33]
    lens = np.array([P + s for s in suf], dtype=np.int32)
    pre_k = words(rng, (P, Hkv, d), dt)
    pre_v = words(rng, (P, Hkv, d), dt)
    suf_k = [words(rng, (s, Hkv, d), dt) for s in suf]
    suf_v = [words(rng, (s, Hkv, d), dt) for s in suf]
    q = words(rng, (B, 5, Hq, d), dt)
    outs = []
    for shared in (True, False):
        NB = 32
        kp = np.full((NB, Hkv, bs, d), 0x7FC0, np.uint16)
        vp = kp.copy()
        tables = np.full((B, 6), -1, np.int32)
        nxt = 0
        if shared:
            tables[:, :2] = [0, 1]
            oracle.cache_write(kp, vp, pre_k, pre_v, np.arange(P))
            nxt = 2
        for b in range(B):
            if not shared:
                tables[b, :2] = [nxt, nxt + 1]
                oracle.cache_write(kp, vp, pre_k, pre_v, nxt * bs + np.arange(P))
                nxt += 2
            nb = -(-suf[b] // bs)
            tables[b, 2:2 + nb] = np.arange(nxt, nxt + nb)
            nxt += nb
            t = P + np.arange(suf[b])
            oracle.cache_write(kp, vp, suf_k[b], suf_v[b], tables[b, t // bs].astype(np.int64) * bs + t % bs)
        out, _ = oracle.paged_attention(q, kp, vp, tables, lens, dt, 0.35)
        outs.append(out)
    assert np.array_equal(outs[0], outs[1])


def pin_split_merge_equals_unsplit():
    """Partitions + log-sum-exp merge == the unsplit softmax (fp64, 1e-12), including causal rows
    whose last partition is empty."""
    rng = _rng(8)
    for L, ql, P, dt in [(100, 1, 16, FP16), (512, 1, 512, FP16), (1031, 1, 256, BF16), (37, 5, 16, BF16),
                         (516, 5, 512, FP16)]:
        Hq, Hkv, d = 4, 2, 16
        q = words(rng, (ql, Hq, d), dt, sigma=3.0)
        kc = words(rng, (L, Hkv, d), dt)
        vc = words(rng, (L, Hkv, d), dt, mean=0.5)
        ref = oracle.attention(q, kc, vc, dt, 0.25)
        m, l, o = oracle.attention_partitions(q, kc, vc, dt, 0.25, P)
        for qi in range(ql):
            for h in range(Hq):
                got = oracle.lse_merge(m[qi, h], l[qi, h], o[qi, h])
                assert np.allclose(got, ref[qi, h], rtol=1e-12, atol=1e-13), (L, ql, P, qi, h)


def pin_cache_write_skip_and_untouched():
    rng = _rng(9)
    NB, Hkv, bs, d = 6, 2, 16, 8
    kp = np.full((NB, Hkv, bs, d), 0xA5A5, np.uint16)
    vp = kp.copy()
    kn = words(rng, (4, Hkv, d), FP16)
    vn = words(rng, (4, Hkv, d), FP16)
    slots = np.array([5, -1, 17, 95])
    oracle.cache_write(kp, vp, kn, vn, slots)
    expect_k = np.full_like(kp, 0xA5A5)
    expect_v = expect_k.copy()
    for i, s in enumerate(slots):
        if s >= 0:
            expect_k[s // bs, :, s % bs] = kn[i]
            expect_v[s // bs, :, s % bs] = vn[i]
    assert np.array_equal(kp, expect_k) and np.array_equal(vp, expect_v)


def pin_copy_on_write_equals_private_write():
    """A sample that shares a prompt's blocks, copies the partly filled last block and writes its own token
    into the copy, gathers exactly its logical tokens; the prompt's owner still gathers its own; the copy
    touches nothing else (yangyu.win blog #54 section 5 question 2: copy-on-write on divergence)."""
    rng = _rng(10)
    NB, Hkv, bs, d = 8, 2, 16, 8
    kp = np.zeros((NB, Hkv, bs, d), np.uint16)
    vp = np.zeros_like(kp)
    prompt_k = words(rng, (40, Hkv, d), FP16)
    prompt_v = words(rng, (40, Hkv, d), FP16)
    table_a = np.array([5, 1, 6], np.int32)                 # 40 tokens: blocks 5, 1 and 6 (8 tokens used)
    t = np.arange(40)
    oracle.cache_write(kp, vp, prompt_k, prompt_v, table_a[t // bs].astype(np.int64) * bs + t % bs)
    before = (kp.copy(), vp.copy())
    # sample B shares blocks 5, 1, 6; its token 40 goes into block 6 -> copy 6 to the free block 3 first
    table_b = np.array([5, 1, 3], np.int32)
    oracle.copy_blocks(kp, vp, [(6, 3)])
    new_k = words(rng, (1, Hkv, d), FP16)
    new_v = words(rng, (1, Hkv, d), FP16)
    oracle.cache_write(kp, vp, new_k, new_v, np.array([3 * bs + 40 % bs]))
    assert np.array_equal(oracle.gather(kp, table_b, 41), np.concatenate([prompt_k, new_k]))
    assert np.array_equal(oracle.gather(vp, table_b, 41), np.concatenate([prompt_v, new_v]))
    assert np.array_equal(oracle.gather(kp, table_a, 40), prompt_k)
    changed = np.argwhere((kp != before[0]).any(axis=(1, 2, 3))).ravel().tolist()
    assert changed == [3]


def _normalised(rng, shape):
    x = rng.random(shape).astype(np.float64) ** 3
    return (x / x.sum(-1, keepdims=True)).astype(np.float32)


def pin_spec_verify_is_lossless():
    """The first emitted token is distributed as the target p, whatever the draft q (yangyu.win blog #54,
    section 5 question 3: P(x) = min(q(x), p(x)) + max(0, p(x) - q(x)) = p(x)). Checked by quadrature over the
    draft token x ~ q and midpoint grids of the two uniforms."""
    rng = _rng(11)
    V, N = 6, 120
    for trial in range(3):
        p = _normalised(rng, (V,))
        q = _normalised(rng, (V,))
        grid = (np.arange(N) + 0.5) / N
        xs, us, vs = np.meshgrid(np.arange(V), grid, grid, indexing="ij")
        B = xs.size
        P = np.broadcast_to(np.stack([p, _normalised(rng, (V,))]), (B, 2, V))
        Q = np.broadcast_to(q, (B, 1, V))
        out, n = oracle.spec_verify(P, Q, xs.reshape(B, 1), us.reshape(B, 1).astype(np.float32),
                                    vs.reshape(B).astype(np.float32))
        w = q[xs.reshape(B)] / (N * N)
        freq = np.bincount(out[:, 0], weights=w, minlength=V)
        assert np.allclose(freq, p, atol=0.02), (trial, freq, p)
        assert ((n == 1) | (n == 2)).all()


def pin_spec_verify_special_cases():
    rng = _rng(12)
    V, K, B = 50, 4, 64
    p = _normalised(rng, (B, K + 1, V))
    draft = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    v = rng.random(B).astype(np.float32)
    # draft == target: every draft kept, then one token from p_K at v (inverse CDF == numpy searchsorted)
    out, n = oracle.spec_verify(p, p[:, :K], draft, u, v)
    assert (n == K + 1).all() and np.array_equal(out[:, :K], draft)
    for b in range(B):
        c = np.cumsum(p[b, K].astype(np.float64))
        assert out[b, K] == np.searchsorted(c, float(v[b]) * c[-1], side="right")
    # the target gives the drafted token no mass: rejected at once, never resampled to it
    p0 = p.copy()
    p0[np.arange(B), 0, draft[:, 0]] = 0.0
    q = _normalised(rng, (B, K, V))
    out, n = oracle.spec_verify(p0, q, draft, u, v)
    assert (n == 1).all() and (out[:, 0] != draft[:, 0]).all() and (out[:, 1:] == -1).all()
    # the resampled token comes from max(0, p - q): its residual mass is positive
    r = np.maximum(0.0, p0[np.arange(B), 0].astype(np.float64) - q[:, 0].astype(np.float64))
    assert (r[np.arange(B), out[:, 0]] > 0).all()


def _torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_decode_matches_torch():
    ref = _torch_e4m3_values()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9


def pin_e4m3_encode_matches_torch():
    rng = _rng(13)
    x = np.concatenate([rng.uniform(-464, 464, 4000), rng.standard_normal(4000) * 3, rng.standard_normal(2000) * 0.01,
                        (_torch_e4m3_values()[:126] * np.array([1.0])), [0.0, -0.0, 2 ** -10, 3 * 2 ** -11, 1.0625,
                                                                       1.1875, 448.0, 464.0, -464.0]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in x], dtype=np.uint8)
    zero = (x == 0)
    assert np.array_equal(got[~zero], ref[~zero])
    assert all(oracle.f32_to_e4m3(v) == 0x7E for v in (465.0, 1e6)) and oracle.f32_to_e4m3(-1e30) == 0xFE


def pin_fp8_quantised_write_bounds():
    """Each (token, head) row maps its largest magnitude to 448; every value is within half a quantum."""
    rng = _rng(14)
    NB, Hkv, bs, d, dt = 4, 2, 16, 64, BF16
    kbuf, vbuf = oracle.fp8_pool(NB, Hkv, bs, d), oracle.fp8_pool(NB, Hkv, bs, d)
    k = words(rng, (10, Hkv, d), dt, sigma=2.0)
    v = words(rng, (10, Hkv, d), dt, sigma=0.01)
    slots = np.array([3, 17, 18, 40, 63, 0, 5, 6, 33, 34])
    oracle.cache_write_fp8(kbuf, vbuf, (NB, Hkv, bs, d), k, v, slots, dt)
    vals = _torch_e4m3_values()
    for buf, src in ((kbuf, k), (vbuf, v)):
        codes, scales = oracle.fp8_views(buf, NB, Hkv, bs, d)
        x = lib_decode(src, dt)
        for i, sl in enumerate(slots):
            for h in range(Hkv):
                sc = scales[sl // bs, h, sl % bs]
                assert sc == np.float32(np.float32(np.abs(x[i, h]).max()) / np.float32(448.0))
                deq = vals[codes[sl // bs, h, sl % bs]] * np.float64(sc)
                assert np.abs(vals[codes[sl // bs, h, sl % bs]]).max() == 448.0
                assert (np.abs(deq - x[i, h]) <= np.maximum(np.abs(x[i, h]) * 2.0 ** -4, float(sc) * 2.0 ** -10) * 1.0000001).all()


def pin_fp8_attention_matches_sdpa():
    """The FP8 paged chain (quantising write, gather, dequantise, attention) == torch fp64 SDPA on the
    dequantised K/V."""
    rng = _rng(15)
    NB, Hkv, bs, d, Hq, dt = 12, 2, 16, 32, 8, FP16
    lens = np.array([5, 37, 90], np.int32)
    tables = np.full((3, 6), -1, np.int32)
    perm = rng.permutation(NB)
    kbuf, vbuf = oracle.fp8_pool(NB, Hkv, bs, d), oracle.fp8_pool(NB, Hkv, bs, d)
    pos, ks, vs = 0, [], []
    for b, L in enumerate(lens):
        nb = -(-int(L) // bs)
        tables[b, :nb] = perm[pos:pos + nb]
        pos += nb
        k, v = words(rng, (int(L), Hkv, d), dt), words(rng, (int(L), Hkv, d), dt)
        t = np.arange(L)
        oracle.cache_write_fp8(kbuf, vbuf, (NB, Hkv, bs, d), k, v, tables[b, t // bs].astype(np.int64) * bs + t % bs, dt)
        ks.append(k)
        vs.append(v)
    for ql in (1, 5):
        q = words(rng, (3, ql, Hq, d), dt)
        scale = float(np.float32(0.2))
        out = oracle.paged_attention_fp8(q, kbuf, vbuf, (NB, Hkv, bs, d), tables, lens, dt, scale)
        vals = _torch_e4m3_values()
        kc, ksc = oracle.fp8_views(kbuf, NB, Hkv, bs, d)
        vc, vsc = oracle.fp8_views(vbuf, NB, Hkv, bs, d)
        for b, L in enumerate(lens):
            if L < ql:
                continue
            t = np.arange(L)
            pb, off = tables[b, t // bs], t % bs
            kd = vals[kc[pb, :, off]] * ksc[pb, :, off][..., None].astype(np.float64)
            vd = vals[vc[pb, :, off]] * vsc[pb, :, off][..., None].astype(np.float64)
            qf = np.zeros((L, Hq, d))
            qf[L - ql:] = lib_decode(q[b], dt)
            Q = torch.from_numpy(qf).permute(1, 0, 2)[None]
            K = torch.from_numpy(kd).permute(1, 0, 2)[None]
            V = torch.from_numpy(vd).permute(1, 0, 2)[None]
            ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=scale,
                                                                   enable_gqa=True)[0].permute(1, 0, 2).numpy()[L - ql:]
            assert np.allclose(out[b], ref, rtol=1e-10, atol=1e-12)


ALL_PINS = [pin_decode_fp16, pin_decode_bf16, pin_mapping_yangyu, pin_mapping_tanhdev, pin_kv_size_closed_form,
            pin_sdpa_contiguous, pin_paged_equals_contiguous_under_permutation, pin_closed_forms, pin_weights,
            pin_gqa_is_mha_with_duplicated_heads, pin_verify_rows_are_decodes, pin_shared_prefix_equals_duplicated,
            pin_split_merge_equals_unsplit, pin_cache_write_skip_and_untouched, pin_copy_on_write_equals_private_write,
            pin_spec_verify_is_lossless, pin_spec_verify_special_cases, pin_e4m3_decode_matches_torch,
            pin_e4m3_encode_matches_torch, pin_fp8_quantised_write_bounds, pin_fp8_attention_matches_sdpa]
