"""The oracle's pins have teeth: plant one plausible mistake at a time in a
copy of the oracle's C source (a wrong constant, a dropped term, a wrong
index or rounding), build it, route the oracle through it, and check that
the pins of tests/test_oracle_pins.py reject it.  CPU only; the real oracle
is never modified."""
import os
import shutil

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kvq_oracle.c")

# (name, exact text in the oracle, its replacement, the pins that must catch it)
MUTATIONS = [
    ("int8 scale constant 127 -> 128", "float s = a / 127.0f;", "float s = a / 128.0f;",
     [lambda: [pins.test_int8_closed_form(i) for i in range(len(pins._golden_int8()))]]),
    ("int8 rounding: half-even -> truncation",
     "float q = nearbyintf(x[i] / s);\n        if (q > 127.0f) q = 127.0f;\n        if (q < -127.0f) q = -127.0f;\n        codes[i] = (int8_t)q;\n    }\n}\n\n/* One dynamic-scale INT4",
     "float q = truncf(x[i] / s);\n        if (q > 127.0f) q = 127.0f;\n        if (q < -127.0f) q = -127.0f;\n        codes[i] = (int8_t)q;\n    }\n}\n\n/* One dynamic-scale INT4",
     [lambda: [pins.test_int8_closed_form(i) for i in range(len(pins._golden_int8()))],
      pins.test_int8_error_bound_and_range]),
    ("int4 scale constant 7 -> 8", "float s = a / 7.0f;", "float s = a / 8.0f;",
     [lambda: [pins.test_int4_closed_form(i) for i in range(len(pins._golden_int4()))],
      pins.test_int4_error_bound_and_range]),
    ("e4m3 ties to odd",
     "oracle_e4m3_decode((uint8_t)c) - a);\n            if (d < best_d || (d == best_d && (c & 1) == 0))",
     "oracle_e4m3_decode((uint8_t)c) - a);\n            if (d < best_d || (d == best_d && (c & 1) == 1))",
     [pins.test_e4m3_exhaustive_roundtrip_and_even_ties, pins.test_e4m3_matches_torch_cast]),
    ("e5m2 exponent bias 15 -> 16", "else v = ldexp(1.0 + (double)m / 4.0, e - 15);",
     "else v = ldexp(1.0 + (double)m / 4.0, e - 16);",
     [lambda: [pins.test_e5m2_golden(x, c) for x, c in pins._golden_e5m2()],
      pins.test_e5m2_exhaustive_roundtrip_and_even_ties]),
    ("decode drops the softmax scale", "z[t] = sm_scale * acc;", "z[t] = acc;",
     [lambda: pins.test_decode_matches_dense_bruteforce(oracle.INT8_PER_GROUP, 16)]),
    ("decode maps Q heads to KV heads modulo (interleaved groups)", "int h = hq / G;",
     "int h = hq % Hkv;",
     [pins.test_decode_gqa_equals_mha_with_replicated_heads,
      lambda: pins.test_decode_matches_dense_bruteforce(oracle.INT8_PER_GROUP, 16)]),
    ("decode drops the last token of every sequence", "for (int t = 0; t < L; ++t) {\n            int64_t slot = (int64_t)table[(int64_t)s * max_blocks + t / bs] * bs + t % bs;\n            double w",
     "for (int t = 0; t + 1 < L; ++t) {\n            int64_t slot = (int64_t)table[(int64_t)s * max_blocks + t / bs] * bs + t % bs;\n            double w",
     [pins.test_decode_single_token_returns_value,
      lambda: pins.test_decode_matches_dense_bruteforce(oracle.INT8_PER_GROUP, 16)]),
    ("decode reads V through the K half of the store", "chan_scales, slot, 1, h, d);",
     "chan_scales, slot, 0, h, d);",
     [lambda: pins.test_decode_matches_dense_bruteforce(oracle.FP16, 0)]),
    ("append stores K codes in the V half and V in the K half",
     "int64_t base = (slot * 2 + kv) * (int64_t)per;", "int64_t base = (slot * 2 + (1 - kv)) * (int64_t)per;",
     [lambda: pins.test_append_places_slots_and_keeps_sentinels(oracle.INT8_PER_TOKEN, 0)]),
    ("KV size formula drops the factor 2 (K and V)", "return 2ull * batch * seq_len", "return 1ull * batch * seq_len",
     [pins.test_kv_size_formula_examples]),
]


def _fails(fn) -> bool:
    try:
        fn()
    except (AssertionError, ValueError):
        return True
    return False


@pytest.mark.parametrize("name,old,new,checks", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(name, old, new, checks, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor must be unique: " + name
    mutated = tmp_path / "kvq_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_source(str(mutated), str(tmp_path / "liboracle_mutant.so"))
    with oracle.use_library(so):
        caught = [_fails(c) for c in checks]
    assert any(caught), "no pin caught: " + name


def test_unmutated_copy_passes_the_same_pins(tmp_path):
    """Control: a verbatim copy built the same way passes every check used above."""
    dst = tmp_path / "kvq_oracle_copy.c"
    shutil.copy(SRC, dst)
    so = oracle.compile_source(str(dst), str(tmp_path / "liboracle_copy.so"))
    with oracle.use_library(so):
        for _, _, _, checks in MUTATIONS:
            for c in checks:
                assert not _fails(c)
