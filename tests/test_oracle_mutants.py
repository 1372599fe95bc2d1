"""Plant plausible mistakes in copies of the oracle source and check that the
pins catch every one of them (the planted copies are built and run on the CPU
only)."""
import os

import pytest

import _pins
import oracle

# (name, original text, planted text) -- each replacement must occur in the source
MUTANTS = [
    ("drop_rope_term", "s[t] = (lat + rope) * J->scale;", "s[t] = (lat) * J->scale;"),
    ("no_scale", "s[t] = (lat + rope) * J->scale;", "s[t] = (lat + rope);"),
    ("exp_sign", "l += exp(s[t] - m);", "l += exp(m - s[t]);"),
    ("ctx_off_by_one", "long long ctx = (long long)J->d_pos[b] + 1;", "long long ctx = (long long)J->d_pos[b];"),
    ("value_shifted", "o[f] += w * kv_at(J, rows[t], f);", "o[f] += w * kv_at(J, rows[t], J->d_rope + f);"),
    ("e4m3_exponent_bias", "else v = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_subnormal_scale", "if (e == 0) v = ldexp((double)m / 8.0, -6);", "if (e == 0) v = ldexp((double)m / 8.0, -7);"),
    ("e4m3_scale_dropped", "[r * J->row_stride + i]) * J->kv_scale;", "[r * J->row_stride + i]);"),
    ("q_batch_head_transposed", "J->q + ((long long)b * J->heads + h) * D;",
     "J->q + ((long long)h * J->batch + b) * D;"),
    ("mask_inclusive_end", "if (i < 0 || i >= J->cache_len[b]) continue;\n            long long r = base + i;",
     "if (i < 0 || i > J->cache_len[b]) continue;\n            long long r = base + i;"),
    ("row_offset_ignored", "long long base = J->row_offset ? J->row_offset[b] : 0;\n    long long n = 0;",
     "long long base = 0;\n    long long n = 0;"),
    ("log2_for_ln", "double lse = m + log(l);", "double lse = m + log2(l);"),
    ("merge_weight_wrong", "double w = exp(lse_s[sp] - tot);", "double w = exp(lse_s[sp] - M);"),
    ("rope_from_latent_q", "rope += widen_bf16(qh[J->d_latent + i])", "rope += widen_bf16(qh[i])"),
]


def _run_pins(lib):
    failed = []
    for pin in _pins.ALL_PINS:
        try:
            pin(lib=lib)
        except AssertionError as e:
            failed.append(f"{pin.__name__}: {e}")
    return failed


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, planted):
    src = open(oracle.SOURCE_PATH).read()
    assert src.count(orig) == 1, f"mutation anchor for {name} must occur exactly once"
    mutated = tmp_path / f"mut_{name}.c"
    mutated.write_text(src.replace(orig, planted))
    lib = oracle.bind(oracle.compile_source(str(mutated), str(tmp_path / f"libmut_{name}.so")))
    failed = _run_pins(lib)
    assert failed, f"no pin caught the planted mistake {name}"
