"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is a one-line edit of a copy of oracle/oracle.c (a dropped term,
a wrong sign, index or operand, a wrong constant), compiled to a temporary
library and run through the pins of ``oracle_pins``.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "max_not_subtracted": ("const double p = exp(s[j] - m);", "const double p = exp(s[j]);"),
    "causal_diagonal_excluded": ("int64_t lim = i + (Nk - Nq) + 1;", "int64_t lim = i + (Nk - Nq);"),
    "value_is_key": ("const double* vb = v + (b * Hkv", "const double* vb = k + (b * Hkv"),
    "gqa_head_map": ("const double* kb = k + (b * Hkv + h / group)", "const double* kb = k + (b * Hkv + h % Hkv)"),
    "lse_log2": ("lse[bh * R + r] = m + log(l);", "lse[bh * R + r] = m + log2(l);"),
    "dot_index": ("dot += qi[c] * kj[c];", "dot += qi[c] * kj[0];"),
    "no_normalisation": ("oi[c] = acc[c] / l;", "oi[c] = acc[c];"),
    "e4m3_ties_away": ("double qn = nearbyint(ldexp(a, 3 - E));", "double qn = round(ldexp(a, 3 - E));"),
    "e4m3_bias": ("const int field = E + 7;", "const int field = E + 8;"),
    "quant_xmax_127": ("amax / 448.0f", "amax / 127.0f"),
    "quant_reciprocal_product": ("oracle_e4m3_encode_f64((double)yb[i] / (double)s)",
                                 "oracle_e4m3_encode(yb[i] * (1.0f / s))"),
    "quant_fp32_quotient_first": ("oracle_e4m3_encode_f64((double)yb[i] / (double)s)",
                                  "oracle_e4m3_encode(yb[i] / s)"),
    "fwht_sign": ("y[c + h] = a - b;", "y[c + h] = b - a;"),
    "signs_ignored": ("(signs && signs[c] < 0) ? -x[c] : x[c]", "x[c]"),
    "rotation_norm_missing": ("(float)(1.0 / sqrt((double)d))", "1.0f"),
    "rope_sign": ("y[ia] = ac - bs;", "y[ia] = ac + bs;"),
    "rope_pairing": ("const int64_t ib = (layout == 1) ? 2 * i + 1 : i + half;",
                     "const int64_t ib = (layout == 1) ? 2 * i + 1 : half - 1 - i;"),
    "rope_position": ("const int64_t n = r % N;", "const int64_t n = r / N;"),
    "bwd_D_dropped": ("const double ds = p[j] * (dp[j] - Di);", "const double ds = p[j] * dp[j];"),
    "bwd_dk_operand": ("dkj[c] += scale * ds * qi[c];", "dkj[c] += scale * ds * kj[c];"),
    "bwd_dq_scale": ("dqi[c] += scale * ds * kj[c];", "dqi[c] += ds * kj[c];"),
    "bwd_dv_operand": ("dvj[c] += p[j] * doi[c];", "dvj[c] += p[j] * qi[c];"),
    "bwd_unnormalised": ("for (int64_t j = 0; j < jend; ++j) p[j] /= l;",
                         "for (int64_t j = 0; j < jend; ++j) p[j] /= 1.0;"),
    "bwd_causal_diagonal_excluded": ("const int64_t visible = i + (Nk - Nq) + 1;",
                                     "const int64_t visible = i + (Nk - Nq);"),
    "bwd_dp_operand": ("for (int64_t c = 0; c < d; ++c) dot += doi[c] * vj[c];",
                       "for (int64_t c = 0; c < d; ++c) dot += qi[c] * vj[c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
                    "-o", str(lib), str(src), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_LIB", None)
    monkeypatch.setattr(oracle._build, "build", lambda force=False: str(lib))
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(oracle)
        except AssertionError:
            failed.append(pin.__name__)
    monkeypatch.setattr(oracle, "_LIB", None)
    assert failed, f"mutant {name} passed every pin"
