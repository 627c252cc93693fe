"""Each planted mistake in a copy of the oracle must make at least one pin fail.

The mutants are plausible slips (a dropped term, a wrong sign or index, a reversed
tie-break, a transposed operand, ...). They are compiled from a textual edit of
oracle/ds4x_oracle.c into a temporary library; the oracle source itself is untouched.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ds4x_oracle.c")

MUTANTS = {
    "relu_after_weight": ("double relu = dot > 0.0 ? dot : 0.0;\n      acc += wd[h] * relu;",
                          "acc += (wd[h] * dot > 0.0 ? wd[h] * dot : 0.0);"),
    "no_relu": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "visibility_off_by_one": ("int64_t n = (p + 1) / ratio;", "int64_t n = p / ratio;"),
    "tie_to_higher_row": ("return (x->idx > y->idx) - (x->idx < y->idx);",
                          "return (x->idx < y->idx) - (x->idx > y->idx);"),
    "ascending_order_dropped": ("qsort(out, (size_t)c, sizeof(int32_t), ref_cmp_int);", ";"),
    "dropped_last_dim": ("for (int32_t d = 0; d < D; ++d) dot += qh[d] * ks[d];",
                         "for (int32_t d = 0; d + 1 < D; ++d) dot += qh[d] * ks[d];"),
    "transposed_q_index": ("const double* qh = qd + (int64_t)h * D;", "const double* qh = qd + h;"),
    "mask_not_applied": ("if (s >= n) { row[s] = -INFINITY; continue; }", ";"),
    "attn_scale_dropped": ("logit[j] = scale * dot;", "logit[j] = dot;"),
    "attn_not_normalised": ("oh[d] = ref_from_double(acc[d] / sum, dtype);",
                            "oh[d] = ref_from_double(acc[d], dtype);"),
    "attn_max_sign": ("double p = exp(logit[j] - m);", "double p = exp(m - logit[j]);"),
    "lse_without_max": ("lse[h] = (float)(m + log(sum));", "lse[h] = (float)(log(sum));"),
    "encode_truncates": ("double r = nearbyint(ldexp(a, mant - E));",
                         "double r = floor(ldexp(a, mant - E));"),
    "f16_exponent_bias": ("else v = ldexp((double)(f + 1024), e - 25);",
                          "else v = ldexp((double)(f + 1024), e - 24);"),
    "shortcut_wrong_count": ("for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;",
                             "for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(i + 1);"),
    "decode_append_one_early": ("(int64_t)S < (p + 1) / ratio) {", "(int64_t)S <= (p + 1) / ratio) {"),
    "decode_position_shifted": ("const int64_t p = (int64_t)pos0 + i;", "const int64_t p = (int64_t)pos0 + i + 1;"),
    "decode_first_staged_row_only": ("kv_new + (int64_t)a * Dkv,", "kv_new,"),
    "window_shifted_one_back": ("for (int64_t a = p - window + 1; a <= p; ++a) {",
                                "for (int64_t a = p - window; a < p; ++a) {"),
    "window_excludes_own_position": ("for (int64_t a = p - window + 1; a <= p; ++a) {",
                                     "for (int64_t a = p - window + 1; a < p; ++a) {"),
    "window_buffer_offset_sign": ("int64_t r = a - local_pos0;", "int64_t r = a - local_pos0 - 1;"),
    "window_rows_dropped": ("for (int32_t j = 0; j < nw; ++j)", "for (int32_t j = 0; j < 0; ++j)"),
    "window_rows_from_pooled_kv": ("ref_decode_n(kv_local + (int64_t)wrows[j] * Dkv",
                                   "ref_decode_n(kv + (int64_t)wrows[j] * Dkv"),
    "window_of_first_token": ("ref_window_rows(positions[t], window", "ref_window_rows(positions[0], window"),
    "compress_bias_reversed": ("(double)bias[(int64_t)i * D + d];", "(double)bias[(int64_t)(ratio - 1 - i) * D + d];"),
    "compress_bias_dropped": ("(double)bias[(int64_t)i * D + d];", "0.0;"),
    "compress_frontier_ignored": ("return v < n_frontier ? held + v * D : fresh + (v - n_frontier) * D;",
                                  "return fresh + (v < n_frontier ? 0 : v - n_frontier) * D;"),
    "compress_not_normalised": ("rows[j * D + d] = ref_from_double(acc / sum, dtype);",
                                "rows[j * D + d] = ref_from_double(acc, dtype);"),
    "compress_gate_of_next_position": ("const int64_t v = j * ratio + i;\n        z[i]",
                                       "const int64_t v = j * ratio + (i + 1) % ratio;\n        z[i]"),
    "compress_frontier_shifted": ("memcpy(fx_out + i * D, ref_seq_row(fx_in, x, n_frontier, v, D),",
                                  "memcpy(fx_out + i * D, ref_seq_row(fx_in, x, n_frontier, v + 1 < n ? v + 1 : v, D),"),
    "decode_raw_rows_one_late": ("memcpy(kv_raw + (int64_t)pos0 * Dkv, kv_raw_new",
                                 "memcpy(kv_raw + (int64_t)(pos0 + 1) * Dkv, kv_raw_new"),
    "decode_window_misses_new_rows": ("Dkv, 0, pos0 + n_steps, window, scale,", "Dkv, 0, pos0, window, scale,"),
    "w_index_transposed": ("ref_decode_n(w + (int64_t)t * H, H, REF_F16, wd);\n      int64_t n",
                           "ref_decode_n(w + (int64_t)t, H, REF_F16, wd);\n      int64_t n"),
}


# Each mutant's pins run in a child process: a planted slip may also read out of bounds, and a
# child that dies by a signal has caught it just as a failing pin would, without taking pytest down.
_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
o = oracle.Oracle({lib!r})
for check in oracle_pins.ALL_CHECKS:
    try:
        check(o)
    except (AssertionError, ValueError, IndexError):
        print("FAILED", check.__name__, flush=True)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so"))
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests), tests=tests, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    died = r.returncode < 0
    failed = [l.split()[1] for l in r.stdout.splitlines() if l.startswith("FAILED")]
    assert r.returncode == 0 or died, r.stderr[-2000:]
    assert failed or died, f"no pin catches the planted mistake {name}"
