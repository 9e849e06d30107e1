"""The oracle's pins must catch plausible slips.

Each case plants one mistake in a temporary copy of the oracle's C source
(never in the committed file), builds it with gcc, points the oracle's loader
at the mutant, runs the pin suite, and requires at least one pin to fail.
CPU only.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTATIONS = {
    "decay dropped": ("const double a = exp(gt[c]);", "const double a = 1.0;"),
    "decay on the value axis": (
        "const double a = exp(gt[c]);\n            for (int64_t x = 0; x < V; ++x) S[c * V + x] *= a;",
        "for (int64_t x = 0; x < V; ++x) S[c * V + x] *= exp(gt[x % K]);"),
    "delta-rule sign": ("- bt * kt[c] * kS[x]", "+ bt * kt[c] * kS[x]"),
    "beta dropped on the write": ("+ bt * kt[c] * vt[x]", "+ kt[c] * vt[x]"),
    "erase with q instead of k": ("kS[x] += kt[c] * S[c * V + x];", "kS[x] += qt[c] * S[c * V + x];"),
    "read-out with k": ("acc += S[c * V + x] * qt[c];", "acc += S[c * V + x] * kt[c];"),
    "scale dropped": ("ot[x] = j->scale * acc;", "ot[x] = acc;"),
    "conv taps reversed": ("acc += w[c * W + j] * x[s * C + c];",
                           "acc += w[c * W + (W - 1 - j)] * x[s * C + c];"),
    "conv not restarted per sequence": ("if (s >= b) acc", "if (s >= 0) acc"),
    "dt_bias transposed": ("dt_bias[h * K + c]", "dt_bias[c * H + h]"),
    "A_log not exponentiated": ("val = -exp(A_log[c]) * softplus", "val = A_log[c] * softplus"),
    "no lower bound": ("g[i] = val > lower_bound ? val : lower_bound;", "g[i] = val;"),
    "output norm over the sum, not the mean": ("sqrt(ss / (double)V + eps)", "sqrt(ss + eps)"),
    "output gate sigmoid sign": ("exp(-gate[r * V + c])", "exp(gate[r * V + c])"),
    "output weight dropped": ("(w ? w[c] : 1.0)", "1.0"),
    "output eps outside the root": ("sqrt(ss / (double)V + eps)", "(sqrt(ss / (double)V) + eps)"),
    "backward: state gradient not decayed": ("dS[c * V + x] = ea * d;", "dS[c * V + x] = d;"),
    "backward: erase term sign": ("const double d = dS[c * V + x] + kt[c] * (-bt * ddelta[x]);",
                                  "const double d = dS[c * V + x] + kt[c] * (bt * ddelta[x]);"),
    "backward: dq from the pre-update state": ("(Sp[c * V + x] + kt[c] * delta[x]) * dot[x]",
                                               "Sp[c * V + x] * dot[x]"),
    "backward: dbeta without the erase": ("db += ddelta[x] * (vt[x] - kS[x]);", "db += ddelta[x] * vt[x];"),
    "gate projection: f_b transposed": ("acc += f_b[j * R + i] * y[i];", "acc += f_b[i * HK + j] * y[i];"),
    "gate projection: low-rank step skipped": ("acc += f_a[i * D + d] * xt[d];", "acc += xt[d];"),
    "gate projection: b_proj transposed": ("z += b_proj[h * D + d] * xt[d];", "z += b_proj[d * NH + h] * xt[d];"),
    "gate projection: sigmoid sign": ("beta[t * NH + h] = 1.0 / (1.0 + exp(-z));",
                                      "beta[t * NH + h] = 1.0 / (1.0 + exp(z));"),
}

PINS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and n != "test_thread_count_does_not_change_results"]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for '{name}' not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(path), "-o", str(so), "-lm"],
                   check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(tmp_path, name, monkeypatch):
    old, new = MUTATIONS[name]
    so = _build_mutant(tmp_path, name, old, new)
    real = oracle._load()
    mutant = ctypes.CDLL(so)
    for fn in ("kda_oracle_forward", "kda_oracle_short_conv", "kda_oracle_l2norm", "kda_oracle_gate",
               "kda_oracle_output_gate", "kda_oracle_backward", "kda_oracle_gate_proj"):
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
        getattr(mutant, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", mutant)
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the mutation '{name}'"


def test_committed_oracle_passes_all_pins():
    for pin in PINS:
        pin()
