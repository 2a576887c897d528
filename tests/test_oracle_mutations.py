"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/la_oracle.c`` (on the CPU:
a dropped term, a wrong sign, a wrong operand, a wrong order), builds it, and
runs the pin suite against it in a subprocess. Every mutant must fail a pin.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "la_oracle.c")

MUTANTS = {
    "phi_drops_plus_one": ("x > 0.0 ? x + 1.0 : exp(x)", "x > 0.0 ? x : exp(x)"),
    "phi_wrong_branch": ("x > 0.0 ? x + 1.0 : exp(x)", "x < 0.0 ? x + 1.0 : exp(x)"),
    "norm_drops_normalizer": ("ot[j] = num[j] / d;", "ot[j] = num[j];"),
    "norm_z_counts_tokens": ("z[i] += f[i];", "z[i] += 1.0;"),
    "norm_output_before_update": (
        "for (int i = 0; i < dk; ++i) p[i] = phi(qt[i]);",
        "for (int i = 0; i < dk; ++i) p[i] = phi(qt[i]);"
        " for (int i = 0; i < dk; ++i) { for (int j = 0; j < dv; ++j)"
        " S[(size_t)i * dv + j] -= f[i] * vt[j]; z[i] -= f[i]; }"),
    "decay_misses_normalizer": ("z[i] = g * z[i] + f[i];", "z[i] = z[i] + f[i];"),
    "decay_misses_state": (
        "S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + f[i] * vt[j];",
        "S[(size_t)i * dv + j] = S[(size_t)i * dv + j] + f[i] * vt[j];"),
    "decay_after_write": (
        "S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + f[i] * vt[j];",
        "S[(size_t)i * dv + j] = g * (S[(size_t)i * dv + j] + f[i] * vt[j]);"),
    "kda_decay_on_value_axis": (
        "for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] *= at[c];",
        "for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] *= at[i % dk];"),
    "kda_error_against_undecayed": (
        "for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] *= at[c];", "/* decay moved below */"),
    "gla_gate_after_write": (
        "S[(size_t)i * dv + j] = gt[i] * S[(size_t)i * dv + j] + f[i] * vt[j];",
        "S[(size_t)i * dv + j] = gt[i] * (S[(size_t)i * dv + j] + f[i] * vt[j]);"),
    "gla_gate_on_value_axis": (
        "S[(size_t)i * dv + j] = gt[i] * S[(size_t)i * dv + j] + f[i] * vt[j];",
        "S[(size_t)i * dv + j] = gt[j % dk] * S[(size_t)i * dv + j] + f[i] * vt[j];"),
    "gla_phi_on_query_dropped": ("p[i] = identity_phi ? qt[i] : phi(qt[i]);", "p[i] = qt[i];"),
    "gdn_error_sign": ("u[i] = bt * (vt[i] - sk);", "u[i] = bt * (vt[i] + sk);"),
    "gdn_error_against_undecayed": (
        "for (size_t e = 0; e < sz; ++e) S[e] *= gt;             /* S~ = g S */",
        "/* decay moved below */"),
    "gdn_reads_with_key": ("acc += S[(size_t)i * dk + c] * qt[c];", "acc += S[(size_t)i * dk + c] * kt[c];"),
    "gdn_drops_beta": ("u[i] = bt * (vt[i] - sk);", "u[i] = (vt[i] - sk);"),
}
# the undecayed-error mutants keep the decay, but apply it after the write
MUTANTS_EXTRA = {
    "kda_error_against_undecayed": (
        "/* S = S~ + u k^T (after the decay) */\n"
        "                for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] += u[i] * kt[c];\n",
        "/* S = S~ + u k^T (after the decay) */\n"
        "                for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] += u[i] * kt[c];\n"
        "            for (int i = 0; i < dv; ++i) for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] *= at[c];\n"),
    "gdn_error_against_undecayed": (
        "double* ot = o + row * dv;                               /* o = S q */",
        "for (size_t e = 0; e < sz; ++e) S[e] *= gt; double* ot = o + row * dv;"),
}


def _build(tmp, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, name
    src = src.replace(old, new, 1)
    if name in MUTANTS_EXTRA:
        o2, n2 = MUTANTS_EXTRA[name]
        assert src.count(o2) == 1, name
        src = src.replace(o2, n2, 1)
    c = os.path.join(tmp, name + ".c")
    so = os.path.join(tmp, name + ".so")
    open(c, "w").write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", c, "-o", so, "-lm"],
                   check=True, capture_output=True)
    return so


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(tmp_path, name):
    so = _build(str(tmp_path), name)
    env = dict(os.environ, LA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
