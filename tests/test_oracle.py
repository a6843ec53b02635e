"""The oracle against its pins (CPU only), and broken copies of the oracle
against the same pins: every planted mistake must fail at least one pin."""
import os
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


# Each mutant replaces one exact piece of oracle.c with a plausible mistake.
MUTANTS = {
    "rescale_sign": ("double a = (m == -INFINITY) ? 0.0 : exp(m - M);",
                     "double a = (m == -INFINITY) ? 0.0 : exp(M - m);"),
    "dropped_u_rescale": ("u[j] = a * u[j] + b * (double)V[t * d + j];",
                          "u[j] = u[j] + b * (double)V[t * d + j];"),
    "dropped_w_rescale": ("w = a * w + b;\n        m = M;\n        if (O)\n"
                          "            for (int64_t j = 0; j < d; ++j) O[t * d + j] = u[j] / w;",
                          "w = w + b;\n        m = M;\n        if (O)\n"
                          "            for (int64_t j = 0; j < d; ++j) O[t * d + j] = u[j] / w;"),
    "reversed_query": ("acc += (double)q[j] * (double)K[t * d + j];",
                       "acc += (double)q[d - 1 - j] * (double)K[t * d + j];"),
    "score_off_by_one": ("double b = exp(s[t] - M);",
                         "double b = exp(s[t > 0 ? t - 1 : 0] - M);"),
    "value_index": ("u[j] = a * u[j] + b * (double)V[t * d + j];",
                    "u[j] = a * u[j] + b * (double)V[t * d + (j + 1) % d];"),
    "combine_transposed": ("double eb = (m_b == -INFINITY) ? 0.0 : exp(m_b - M);",
                           "double eb = (m_b == -INFINITY) ? 0.0 : exp(m_a - M);"),
    "combine_w_dropped": ("*w_o = ea * w_a + eb * w_b;", "*w_o = ea * w_a + w_b;"),
    "hs_offset": ("const double *a = x + (t - k) * stride;",
                  "const double *a = x + (t - k + (t > k ? 1 : 0)) * stride;"),
    "brute_exclusive": ("for (int64_t i = 0; i <= t; ++i) den += exp(s[i] - mx);",
                        "for (int64_t i = 0; i < t; ++i) den += exp(s[i] - mx);"),
    "final_m": ("if (m_out) *m_out = m;\n    if (w_out) *w_out = w;\n    if (u_out)\n"
                "        for (int64_t j = 0; j < d; ++j) u_out[j] = u[j];\n    free(u);\n}\n\n"
                "/* Scores",
                "if (m_out) *m_out = m + 0.5;\n    if (w_out) *w_out = w;\n    if (u_out)\n"
                "        for (int64_t j = 0; j < d; ++j) u_out[j] = u[j];\n    free(u);\n}\n\n"
                "/* Scores"),
    "longdouble_sign": ("long double b = expl(s - M);", "long double b = expl(M - s);"),
    # differentiation
    "bwd_decay_sign": ("double decay = exp(lse[i] - lse[i + 1]);",
                       "double decay = exp(lse[i + 1] - lse[i]);"),
    "bwd_dropped_D": ("double dsi = pii * (vr - D);", "double dsi = pii * vr;"),
    "bwd_brute_dropped_go": ("dsl[i] += p[i] * (gv - go);", "dsl[i] += p[i] * gv;"),
    "bwd_brute_grad_index": ("dV[i * d + j] += p[i] * (double)G[t * d + j];",
                             "dV[i * d + j] += p[i] * (double)G[i * d + j];"),
    "bwd_dk_transposed": ("dK[i * d + j] = dsi * (double)q[j];",
                          "dK[i * d + j] = dsi * (double)K[i * d + j];"),
    "lse_direct_exclusive": ("for (int64_t i = 0; i <= t; ++i) acc += exp(s[i] - top);",
                             "for (int64_t i = 0; i < t; ++i) acc += exp(s[i] - top);"),
}


# The same for linattn.c (the causal cos-re-weighted linear attention).
LA_MUTANTS = {
    "la_no_relu_k": ("kp[a] = relu_d(K[t * d + a]);", "kp[a] = (double)K[t * d + a];"),
    "la_brute_no_relu_q": ("dot += relu_d(Q[i * d + c]) * relu_d(K[j * d + c]);",
                           "dot += (double)Q[i * d + c] * relu_d(K[j * d + c]);"),
    "la_brute_weight_sum": ("double s = dot * cos(hp * (double)(i - j) / M);",
                            "double s = dot * cos(hp * (double)(i + j) / M);"),
    "la_brute_exclusive": ("for (int64_t j = 0; j <= i; ++j) {", "for (int64_t j = 0; j < i; ++j) {"),
    "la_sin_sign": ("num += qp[a] * ct * Sc[a * d + b] + qp[a] * st * Ss[a * d + b];",
                    "num += qp[a] * ct * Sc[a * d + b] - qp[a] * st * Ss[a * d + b];"),
    "la_den_dropped_sin": ("den += qp[a] * ct * zc[a] + qp[a] * st * zs[a];",
                           "den += qp[a] * ct * zc[a];"),
    "la_state_transposed": ("Sc[a * d + b] += kc * v;", "Sc[b * d + a] += kc * v;"),
    "la_position_zero_based": ("double pos = (double)(pos0 + t + 1);",
                               "double pos = (double)(pos0 + t);"),
    "la_zero_den": ("O[t * d + b] = den != 0.0 ? num / den : 0.0;", "O[t * d + b] = num / den;"),
}


def _all_mutants():
    for name in sorted(MUTANTS):
        yield name, "oracle.c"
    for name in sorted(LA_MUTANTS):
        yield name, "linattn.c"


@pytest.mark.parametrize("name,fname", list(_all_mutants()))
def test_planted_mistake_fails_a_pin(name, fname, tmp_path):
    old, new = (MUTANTS if fname == "oracle.c" else LA_MUTANTS)[name]
    srcs = []
    for path in oracle_build.SRCS:
        text = open(path).read()
        if os.path.basename(path) == fname:
            assert text.count(old) == 1, f"mutant {name} no longer matches {fname}"
            text = text.replace(old, new)
        csrc = tmp_path / os.path.basename(path)
        csrc.write_text(text)
        srcs.append(str(csrc))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(so),
                    *srcs, "-lm"], check=True)
    failed = []
    with oracle.using_library(str(so)):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


def test_oracle_is_independent_of_the_cuda_path():
    """The oracle shares no code with the CUDA library: no include of the
    library's headers, no import of the package."""
    here = os.path.dirname(oracle_build.SRCS[0])
    for fn in os.listdir(here):
        if fn.endswith((".c", ".h", ".py")):
            text = open(os.path.join(here, fn)).read()
            assert "attention_prefix_scan_02_b300" not in text, fn
            assert "aaren.h" not in text and "csrc" not in text, fn
