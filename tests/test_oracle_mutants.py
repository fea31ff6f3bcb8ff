"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a temporary copy of the oracle's C source (a
dropped rescale term, a flipped sign, a wrong operand or index, a missing
scale or log), builds it, and runs the pin suites (tests/test_oracle_pins.py,
tests/test_oracle_backward_pins.py and tests/test_oracle_fp8_pins.py) against
that copy in a subprocess.  The pin suite must fail for every mutant.  The
committed oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fa_oracle.c")

MUTANTS = {
    "merge_drops_alpha": ("*l_out = alpha * l_a + beta * l_b;", "*l_out = l_a + beta * l_b;"),
    "merge_u_wrong_factor": ("u_out[c] = alpha * u_a[c] + beta * u_b[c];",
                             "u_out[c] = beta * u_a[c] + beta * u_b[c];"),
    "softmax_sign_flipped": ("double p = exp(x[j] - m) / l;", "double p = exp(m - x[j]) / l;"),
    "lse_missing_log": ("*lse_out = m + log(l);", "*lse_out = m + l;"),
    "score_uses_values": ("acc += q[c] * widen_bf16(kbase[(size_t)j * d + c]);",
                          "acc += q[c] * widen_bf16(vbase[(size_t)j * d + c]);"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "causal_off_by_one": ("if (causal && i + 1 < nvalid) nvalid = i + 1;",
                          "if (causal && i < nvalid) nvalid = i;"),
    "key_len_ignored": ("if (key_len) nvalid = key_len[b] < nvalid ? key_len[b] : nvalid;", ""),
    "online_correction_inverted": ("double corr = (j == 0) ? 0.0 : exp(m - m_new);",
                                   "double corr = (j == 0) ? 0.0 : exp(m_new - m);"),
    "reduce_weight_no_rescale": ("double w = l_k[k] * exp(m_k[k] - m_f) / l_f;",
                                 "double w = l_k[k] / l_f;"),
    "bf16_widen_wrong_half": ("uint32_t word = ((uint32_t)bits) << 16;",
                              "uint32_t word = ((uint32_t)bits) << 15;"),
    "paged_row_in_block": ("const size_t row = (((size_t)phys * H + h) * bs + (size_t)(t % bs)) * d;",
                           "const size_t row = (((size_t)phys * H + h) * bs + (size_t)(t / bs)) * d;"),
    "paged_head_ignored": ("const size_t row = (((size_t)phys * H + h) * bs + (size_t)(t % bs)) * d;",
                           "const size_t row = (((size_t)phys * H + 0) * bs + (size_t)(t % bs)) * d;"),
    # backward
    "bwd_drops_D": ("const double ds = pr[j] * (dp[j] - D);", "const double ds = pr[j] * dp[j];"),
    "bwd_dS_sign": ("const double ds = pr[j] * (dp[j] - D);", "const double ds = pr[j] * (D - dp[j]);"),
    "bwd_P_unnormalised": ("pr[j] = exp(s[j] - L);", "pr[j] = exp(s[j] - m);"),
    "bwd_dP_uses_keys": ("acc += g[c] * vb[(size_t)j * d + c];", "acc += g[c] * kb[(size_t)j * d + c];"),
    "bwd_dV_uses_dS": ("dVb[(size_t)j * d + c] += pr[j] * g[c];", "dVb[(size_t)j * d + c] += ds * g[c];"),
    "bwd_dK_no_scale": ("dKb[(size_t)j * d + c] += scale * ds * q[c];", "dKb[(size_t)j * d + c] += ds * q[c];"),
    "bwd_dQ_uses_values": ("dq[c] += scale * ds * kb[(size_t)j * d + c];",
                           "dq[c] += scale * ds * vb[(size_t)j * d + c];"),
    # backward term magnitudes (the GPU gradient tolerance)
    "bwd_MdV_inflated": ("MdV[(size_t)j * d + c] += pr[j] * fabs(g[c]);",
                         "MdV[(size_t)j * d + c] += 64.0 * pr[j] * fabs(g[c]);"),
    "bwd_MdK_inflated": ("MdK[(size_t)j * d + c] += scale * w * fabs(q[c]);",
                         "MdK[(size_t)j * d + c] += 64.0 * scale * w * fabs(q[c]);"),
    "bwd_MdQ_inflated": ("MdQ[(size_t)i * d + c] += scale * w * fabs(kb[(size_t)j * d + c]);",
                         "MdQ[(size_t)i * d + c] += 64.0 * scale * w * fabs(kb[(size_t)j * d + c]);"),
    "bwd_mag_drops_A": ("const double w = pr[j] * (fabs(dp[j]) + A);", "const double w = pr[j] * fabs(dp[j]);"),
    "bwd_mag_A_drops_D": ("double A = fabs(D);", "double A = 0.0;"),
    # E4M3 decoding
    "e4m3_bias_off_by_one": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "e4m3_no_nan": ("if (e == 15 && m == 7)", "if (e == 16)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    # a mistake is planted everywhere its line appears (the forward's score and
    # mask lines recur in the float64-input forward and in the backward)
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutant_c = tmp_path / f"{name}.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", str(mutant_c),
                    "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, FA_ORACLE_LIB_OVERRIDE=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_backward_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_fp8_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pin suite passed with mutant {name}:\n{r.stdout[-2000:]}"
