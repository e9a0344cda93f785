"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/orthros_ref.c, applies one plausible mistake (a
dropped term, a wrong index or bound, a swapped operand), builds it on the
CPU, and checks that at least one pin of tests/pins.py fails on it. This is
the evidence that the pins constrain every part of the oracle.
"""
import os
import subprocess

import pytest

from tests import pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "orthros_ref.c")

MUTANTS = {
    "window_off_by_one": ("t - window + 1 > 0 ? t - window + 1 : 0", "t - window > 0 ? t - window : 0"),
    "decode_window_off_by_one": ("L - window + 1 > 0 ? L - window + 1 : 0", "L - window + 2 > 0 ? L - window + 2 : 0"),
    "cross_row_excludes_self": ("attend_row(qa, krow + tab, vrow + tab, 0, t, d",
                                "attend_row(qa, krow + tab, vrow + tab, 0, t > 0 ? t - 1 : 0, d"),
    "decode_out_row_skips_new_key": ("attend_row(qa, krow + tab, vrow + tab, 0, L, d",
                                     "attend_row(qa, krow + tab, vrow + tab, 0, L > 0 ? L - 1 : 0, d"),
    "scale_dropped": ("double s = scale * dot;", "double s = dot;"),
    "beta_dropped": ("(double)alpha[c] * (double)qraw[c] + (double)beta[c]", "(double)alpha[c] * (double)qraw[c]"),
    "alpha_dropped": ("(double)alpha[c] * (double)qraw[c] + (double)beta[c]", "(double)qraw[c] + (double)beta[c]"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "gqa_interleaved": ("const int kv = h / g;", "const int kv = h % Hkv;"),
    "out_stream_uses_base_affine": ("affine(qraw, alpha_out + (size_t)h * d,", "affine(qraw, alpha_base + (size_t)h * d,"),
    "decode_out_ignores_q_out": ("(q_out ? q_out : q) + qoff", "q + qoff"),
    "values_are_keys": ("o[c] += p * (double)vj[c];", "o[c] += p * (double)krow[j][c];"),
    "no_normalisation": ("o[c] /= l;", "o[c] /= 1.0;"),
    "prefill_q_out_ignored": ("q_out ? q_out + ((size_t)r * Hq + h) * (size_t)d", "0 ? q_out + ((size_t)r * Hq + h) * (size_t)d"),
    "bw_delta_dropped": ("const double ds = p * (dp - D);", "const double ds = p * dp;"),
    "bw_dk_scale_dropped": ("dkrow[j][c] += scale * ds * qa[c];", "dkrow[j][c] += ds * qa[c];"),
    "bw_dv_uses_ds": ("dvrow[j][c] += p * (double)dO[c];", "dvrow[j][c] += ds * (double)dO[c];"),
    "bw_dp_uses_keys": ("dp += (double)dO[c] * (double)vrow[j][c];", "dp += (double)dO[c] * (double)krow[j][c];"),
    "bw_dq_alpha_dropped": ("dq[qoff + c] += (double)alpha_base[(size_t)h * d + c] * dqa[c];", "dq[qoff + c] += dqa[c];"),
    "bw_dalpha_uses_affined_q": ("d_alpha_base[(size_t)h * d + c] += dqa[c] * (double)q[qoff + c];",
                                 "d_alpha_base[(size_t)h * d + c] += dqa[c] * qa[c];"),
    "bw_out_rows_miss_dq": ("                            else\n                                dq[qoff + c] += gq;",
                            "                            else\n                                (void)gq;"),
    "bw_dbeta_out_to_base": ("d_beta_out[(size_t)h * d + c] += dqa[c];", "d_beta_base[(size_t)h * d + c] += dqa[c];"),
    "bw_out_row_band": ("attend_row_backward(qa, do_out + roff, krow, vrow, dkrow, dvrow, 0, t,",
                        "attend_row_backward(qa, do_out + roff, krow, vrow, dkrow, dvrow, t > 0 ? 1 : 0, t,"),
    "extend_position_shift": ("const int t = cache_lens[b] + (i - new_indptr[b]);",
                              "const int t = cache_lens[b] + (i - new_indptr[b]) - (i > new_indptr[b] ? 1 : 0);"),
    "extend_out_query_first_token": ("q + ((size_t)(new_indptr[b] + t - cache_lens[b]) * Hq + h)",
                                     "q + ((size_t)(new_indptr[b] + 0 * (t - cache_lens[b])) * Hq + h)"),
    "extend_base_sees_next_token": ("attend_row(qa, krow + tab, vrow + tab, lo, t, d, scale, o_base + qoff, &lse, w);\n                lse_base[(size_t)i * Hq + h] = lse;",
                                    "attend_row(qa, krow + tab, vrow + tab, lo, t + (i + 1 < new_indptr[b + 1] ? 1 : 0), d, scale, o_base + qoff, &lse, w);\n                lse_base[(size_t)i * Hq + h] = lse;"),
    "proj_out_rows_base_affine": ("q_out[(size_t)(r - n_base) * Nq + j] = (double)alpha_out[j] * y + (double)beta_out[j];",
                                  "q_out[(size_t)(r - n_base) * Nq + j] = (double)alpha_base[j] * y + (double)beta_out[j];"),
    "proj_k_v_swapped": ("k[(size_t)r * Nkv + (j - Nq)] = y;", "v[(size_t)r * Nkv + (j - Nq)] = y;"),
    "proj_beta_dropped": ("q_base[(size_t)r * Nq + j] = (double)alpha_base[j] * y + (double)beta_base[j];",
                          "q_base[(size_t)r * Nq + j] = (double)alpha_base[j] * y;"),
    "proj_cache_slot_off": ("const size_t off = ((size_t)pg * page_size + t % page_size) * (size_t)Nkv;",
                            "const size_t off = ((size_t)pg * page_size + (t + 1) % page_size) * (size_t)Nkv;"),
    "decode_append_wrong_slot": ("((size_t)pg * page_size + L % page_size) * tok;", "((size_t)pg * page_size + (L + 1) % page_size) * tok;"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found in the oracle source"
    mutated = src.replace(old, new)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"lib{name}.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so_path), str(c_path), "-lm"])
    return str(so_path)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name, oracle_mod):
    orc = oracle_mod.Oracle(_build_mutant(tmp_path, name))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError) as e:
            caught.append(f"{pin.__name__}: {str(e)[:80]}")
    assert caught, f"planted mistake {name!r} passed every pin"
