"""The seeded input generator: its published definitions and the workload recipes."""
import numpy as np

import synth


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator (state += gamma; mix).
    outs, state = [], 0
    for _ in range(3):
        outs.append(synth._mix_py(state))
        state = (state + synth.GAMMA) & synth.MASK64
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # the vectorised hash is the same function
    base = synth.stream_base(7, 9)
    h = synth.hash64(7, 9, np.arange(4, dtype=np.uint64))
    assert [int(x) for x in h] == [synth._mix_py((base + i) & synth.MASK64) for i in range(4)]


def test_scale_makes_unit_variance_exactly():
    # Var of one 16-bit uniform field is (2**32 - 1)/12; twelve of them, doubled and scaled by 2**-17
    # give 4 * 12 * (2**32 - 1) / 12 * 2**-34 = 1 - 2**-32.
    var_field = ((1 << 32) - 1) / 12.0
    assert synth.N_HASH * 4 == 12 and synth.S_MAX == 12 * 0xFFFF
    assert abs(4 * 12 * var_field * float(synth.SCALE_F32) ** 2 - 1.0) < 1e-9
    # |2s - S_MAX| < 2**20 and the scale is a power of two: z is exact in float32
    assert synth.S_MAX < (1 << 20) and float(synth.SCALE_F32) == 2.0 ** -17


def test_value_is_the_twelve_field_sum():
    # brute force for a few counters, straight from the recipe's definition
    base = synth.stream_base(3, 4)
    for i in (0, 1, 77, (1 << 40) + 5):
        s = 0
        for j in range(3):
            h = synth._mix_py((base + 3 * i + j) & synth.MASK64)
            s += sum((h >> (16 * f)) & 0xFFFF for f in range(4))
        want = np.float32((2 * s - 786420) / 131072.0)
        assert synth.unit_f32(3, 4, np.array([i], dtype=np.uint64))[0] == want


def test_values_moments_and_determinism():
    x = synth.unit_f32(5, 11, np.arange(1 << 20, dtype=np.uint64)).astype(np.float64)
    assert abs(float(x.mean())) < 5e-3 and abs(float(x.std()) - 1.0) < 5e-3
    assert np.abs(x).max() <= 6.0
    # Irwin-Hall(12) tails, from its CDF: P(|z| > 3) = 2.014e-3 (N(0,1): 2.70e-3), P(|z| > 4) = 1.71e-5,
    # so a 2**20 sample expects 2112 and 17.9 such values (Poisson bounds at about 4 standard deviations)
    assert 1930 < int((np.abs(x) > 3).sum()) < 2300
    assert 4 <= int((np.abs(x) > 4).sum()) <= 40
    # excess kurtosis of the sum of 12 uniforms is -1.2 / 12 = -0.1
    k = float(((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3.0)
    assert abs(k + 0.1) < 0.03
    a = synth.values16(5, 11, np.arange(1000, dtype=np.uint64), synth.BF16)
    b = synth.values16(5, 11, np.arange(1000, dtype=np.uint64), synth.BF16)
    assert np.array_equal(a, b)


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    w = synth.f32_to_bits16(x, synth.BF16)
    assert [hex(int(v)) for v in w] == ["0x3f80", "0x3f82", "0xbf80", "0x3f81"]


def test_permutation_is_permutation():
    p = synth.permutation(1, 2, 1000)
    assert np.array_equal(np.sort(p), np.arange(1000))


def test_workload_tables_valid():
    for k in (1, 2, 4, 5):
        wl = synth.workload(k, batch=8 if k in (2, 4) else None)
        used = []
        for b in range(wl.B):
            nb = -(-int(wl.context_lens[b]) // wl.bs)
            row = wl.block_tables[b]
            assert (row[:nb] >= 0).all() and (row[:nb] < wl.num_blocks).all() and (row[nb:] == -1).all()
            used.append(row[wl.prefix_tokens // wl.bs:nb])
        own = np.concatenate(used)
        assert len(np.unique(own)) == len(own)          # private blocks are never shared
        if wl.prefix_tokens:
            assert (wl.block_tables[:, :wl.prefix_tokens // wl.bs] == wl.block_tables[0, :wl.prefix_tokens // wl.bs]).all()


def test_workload_shapes():
    w1 = synth.workload(1)
    assert list(w1.context_lens) == [17, 64, 100, 200] and w1.num_blocks == 64 and w1.scale == 0.125
    w2 = synth.workload(2)
    assert w2.context_lens.min() >= 512 and w2.context_lens.max() <= 4096
    assert w2.num_blocks == int(np.ceil(1.1 * sum(-(-int(L) // 16) for L in w2.context_lens)))
    w4 = synth.workload(4)
    suf = w4.context_lens - 1024
    assert suf.min() >= 64 and suf.max() <= 512 and w4.q_len == 5
    w5 = synth.workload(5)
    assert w5.bs == 32 and w5.num_blocks == 16384


def test_host_c_generator_matches_numpy_definition():
    from paged_kv_cache_223_gb300 import _build
    _build.build_synth_host()
    rows = np.array([0, 5, 123456789, 2 ** 40 + 3], dtype=np.int64)
    for dt in (synth.FP16, synth.BF16):
        for sigma, mean in ((1.0, 0.0), (8.0, 0.0), (1.0, 1.0)):
            a = synth.fill_rows16(rows, len(rows), 1024, 0x5EED0002, 77, dt, sigma, mean, use_c=True)
            b = synth.fill_rows16(rows, len(rows), 1024, 0x5EED0002, 77, dt, sigma, mean, use_c=False)
            assert np.array_equal(a, b)
