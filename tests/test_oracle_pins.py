"""The oracle against its pins, and the pins against planted mistakes.

Every pin runs against the real oracle and must pass. Then each entry of
MUTANTS plants one plausible mistake in a copy of oracle.c (a dropped term, a
wrong index or sign, a transposed operand), builds it on the CPU, and the pin
suite must fail on it.
"""
import os
import shutil
import tempfile

import pytest

import oracle
import oracle_pins as pins

MUTANTS = {
    "drop_scale": ("s[t] = (double)scale * dot;", "s[t] = dot;"),
    "gqa_modulo": ("            int g = h / G;\n            const double *qr = qd",
                   "            int g = h % Hkv;\n            const double *qr = qd"),
    "no_causal_limit": ("        int64_t last = L - q_len + qi;                     /* inclusive causal limit */",
                        "        int64_t last = L - 1;"),
    "causal_off_by_one": ("        int64_t last = L - q_len + qi;                     /* inclusive causal limit */",
                          "        int64_t last = L - q_len + qi - (qi > 0);"),
    "gather_wrong_block": ("int64_t phys = table_row[t / bs];", "int64_t phys = table_row[t % bs];"),
    "gather_wrong_offset": ("int64_t off = t % bs;\n", "int64_t off = t / bs % bs;\n"),
    "head_gather_wrong_head": ("pool + ((phys * Hkv + g) * bs + off)", "pool + ((phys * Hkv + 0) * bs + off)"),
    "group_query_wrong_head": ("qb + ((int64_t)qi * J->Hq + g * G + hh) * J->d", "qb + ((int64_t)qi * J->Hq + hh) * J->d"),
    "group_out_wrong_row": ("ob + ((int64_t)qi * J->Hq + g * G + hh) * J->d", "ob + ((int64_t)qi * J->Hq + hh * J->Hkv + g) * J->d"),
    "no_normalise": ("double p = s[t] / l;", "double p = s[t];"),
    "dot_reads_v": ("const double *kr = kd + (t * Hkv + g) * (int64_t)d;",
                    "const double *kr = vd + (t * Hkv + g) * (int64_t)d;"),
    "no_max_shift_bug": ("{ s[t] = exp(s[t] - mx); l += s[t]; }", "{ s[t] = exp(s[t] - mx); l += 1.0; }"),
    "cache_write_offset": ("int64_t blk = s / bs, off = s % bs;", "int64_t blk = s / bs, off = 0;"),
    "cache_write_head_swap": ("int64_t dst = ((blk * Hkv + h) * bs + off) * (int64_t)d;",
                              "int64_t dst = ((blk * Hkv + (Hkv - 1 - h)) * bs + off) * (int64_t)d;"),
    "cache_write_no_skip": ("if (s < 0) continue;", "if (s < 0) s = 0;"),
    "fp16_bias": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "fp16_subnormal": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "bf16_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "merge_unweighted_den": ("den += w * l[p];", "den += l[p];"),
    "merge_weight_sign": ("double w = exp(m[p] - M);", "double w = exp(M - m[p]);"),
    "partition_no_shift": ("double e = exp(s[t - t0] - mx);", "double e = exp(s[t - t0]);"),
    "partition_tail": ("if (t1 > last + 1) t1 = last + 1;", "if (t1 > last + 2) t1 = last + 2;"),
    "copy_wrong_direction": ("memcpy(k_pool + dst * words, k_pool + src * words", "memcpy(k_pool + src * words, k_pool + dst * words"),
    "copy_one_head": ("const int64_t words = (int64_t)Hkv * bs * d;", "const int64_t words = (int64_t)bs * d;"),
    "spec_resample_from_p": ("const double r = (double)pr[t] - (double)qr[t];", "const double r = (double)pr[t];"),
    "spec_resample_q_minus_p": ("const double r = (double)pr[t] - (double)qr[t];", "const double r = (double)qr[t] - (double)pr[t];"),
    "spec_accept_inverted": ("if (uq < pi) {", "if (uq > pi) {"),
    "spec_bonus_wrong_row": ("const float *pr = p + (b * (K + 1) + K) * V;", "const float *pr = p + (b * (K + 1) + K - 1) * V;"),
    "spec_cdf_off_by_one": ("if (c > target) return t;", "if (c > target) return t > 0 ? t - 1 : 0;"),
    "e4m3_bias": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 9);"),
    "e4m3_round_down": ("double n = nearbyint(a / quantum);", "double n = floor(a / quantum);"),
    "fp8_scale_max": ("float scale = amax > 0.0f ? amax / 448.0f : 1.0f;", "float scale = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    "fp8_dequant_no_scale": ("kd[t * d + c] = oracle_e4m3_to_double(k_pool[sr * d + c]) * (double)ks[sr];",
                             "kd[t * d + c] = oracle_e4m3_to_double(k_pool[sr * d + c]);"),
    "weights_unmasked": ("w[t] = t <= last ? s[t] / l : 0.0;", "w[t] = t <= last ? s[t] / l : 1e-300;"),
}


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    oracle.use(None)
    pin()


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = os.path.join(mutant_dir, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.build(force=True, src=path, out=os.path.join(mutant_dir, name + ".so"))
    oracle.use(so)
    failed = []
    try:
        for pin in pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, RuntimeError):
                failed.append(pin.__name__)
    finally:
        oracle.use(None)
    assert failed, f"no pin caught mutant {name}"
