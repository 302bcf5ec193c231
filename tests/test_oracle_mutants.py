"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU, in a
temporary directory), builds it, and runs the pin suite against the broken build in a
child process: the suite must fail.  The real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("if (causal && j > q_pos) return 0;", "if (causal && j >= q_pos) return 0;"),
    "window_off_by_one": ("j < q_pos - window + 1", "j < q_pos - window"),
    "gqa_modulo_map": ("return h / (hq / hkv);", "return h % hkv;"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "max_dropped_from_lse": ("return m + log(l);", "return log(l);"),
    "no_normalisation": ("p[j] = p[j] / l;", "p[j] = p[j];"),
    "top_left_alignment": ("return i + (skv - sq);", "return i;"),
    "pv_reads_k": ("oracle_pv(p, v, skv, d, o);", "oracle_pv(p, k, skv, d, o);"),
    "page_slot_swapped": ("(size_t)(j % page)) * d", "(size_t)(j / page % page)) * d"),
    "tril_strict": ("(uint8_t)(u <= t)", "(uint8_t)(u < t)"),
    "decode_qpos_drops_t": ("qp[t] = len - s_active + t;", "qp[t] = len - s_active;"),
    "exp_sign_flipped": ("exp(s[j] - m)", "exp(m - s[j])"),
    "sink_left_out_of_the_sum": ("double l = exp(sink - m);", "double l = 0.0;"),
    "sink_left_out_of_the_max": ("double m = sink;", "double m = -INFINITY;"),
    "sink_sign_flipped": ("double l = exp(sink - m);", "double l = exp(-sink - m);"),
    "e4m3_bias_off_by_one": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                             "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal_as_normal": ("if (e == 0) v = ldexp((double)m / 8.0, -6);",
                                 "if (e == 0) v = ldexp(1.0 + (double)m / 8.0, -7);"),
    "e4m3_v_scale_dropped": ("oracle_e4m3_to_f64(v_cache[row * D + x]) * v_scale;",
                             "oracle_e4m3_to_f64(v_cache[row * D + x]);"),
    "rope_sign_flipped": ("x[i] = a * c - b * sn;", "x[i] = a * c + b * sn;"),
    "rope_interleaved_pairs": ("const double a = x[i], b = x[i + h];",
                               "const double a = x[i], b = x[i ^ 1];"),
    "circular_row_not_wrapped": ("(size_t)(circular ? j % max_cache_len : j);",
                                 "(size_t)(circular ? j : j);"),
    "new_token_position_off_by_one": ("const long t = j - (len - s_active); /* >= 0: a new token */",
                                      "const long t = j - (len - s_active) - 1;"),
    "rope_q_at_cache_len": ("oracle_rope_row(qd, D, (double)qp, inv_freq);",
                            "oracle_rope_row(qd, D, (double)len, inv_freq);"),
    "varlen_alignment_dropped": ("for (long i = 0; i < nq; ++i) qp[i] = oracle_q_pos(i, nq, nk);",
                                 "for (long i = 0; i < nq; ++i) qp[i] = i;"),
    "varlen_keys_at_query_offset": ("const long q0 = cu_q[s], nq = cu_q[s + 1] - q0, k0 = cu_k[s], nk = cu_k[s + 1] - k0;",
                                    "const long q0 = cu_q[s], nq = cu_q[s + 1] - q0, k0 = cu_q[s], nk = cu_k[s + 1] - cu_k[s];"),
    "rotated_rows_not_rounded": ("for (int x = 0; x < D; ++x) qd[x] = round_bf16(qd[x]);",
                                 "for (int x = 0; x < D; ++x) qd[x] = qd[x];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(lib), str(mutant), "-lm"],
                   check=True)
    env = dict(os.environ, ATTN_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
