"""Planted mistakes in the oracle must be caught by the pins (CPU only).

Each case copies the oracle's C source, plants one plausible mistake (a wrong
sign, a dropped term, a wrong index, a wrong direction), compiles the copy and
checks that the closed-form pin of ``test_oracle`` rejects it.  The planted
copies live in a temporary directory; the oracle itself is never modified.
"""
import os

import numpy as np
import pytest

import oracle
from test_oracle import (_rand_diag, _rand_ssd, _rel, _rng, diag_closed_form,
                         ssd_closed_form)

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

MUTANTS = {
    # diagonal scan
    "decay_sign": ("diag", "exp(dl * A[e * N + n])", "exp(-dl * A[e * N + n])"),
    "decay_wrong_state": ("diag", "exp(dl * A[e * N + n])", "exp(dl * A[e * N + (N - 1 - n)])"),
    "input_drops_delta": ("diag", "h[n] = a * h[n] + dl * B[r + n] * xv;",
                          "h[n] = a * h[n] + B[r + n] * xv;"),
    "readout_uses_B": ("diag", "acc += C[r + n] * h[n];", "acc += B[r + n] * h[n];"),
    "drops_D": ("diag", "const double out = acc + (D ? D[e] * xv : 0.0);", "const double out = acc;"),
    "decay_uses_previous_delta": ("diag", "prep_delta(delta[i], dt_bias",
                                  "prep_delta(delta[t > 0 ? i - ED : i], dt_bias"),
    # SSD / bidirectional
    "ssd_no_decay": ("ssd", "*s = a * (*s) + d * xt[p] * Bt[n];", "*s = (*s) + d * xt[p] * Bt[n];"),
    "ssd_readout_uses_B": ("ssd", "acc += (*s) * Ct[n];", "acc += (*s) * Bt[n];"),
    "ssd_reverse_runs_forward": ("ssd", "const int64_t t = rev ? (L - 1 - k) : k;",
                                 "const int64_t t = k;"),
    "ssd_drops_D": ("ssd", "y[o + p] = D ? D[h] * x[o + p] : 0.0;", "y[o + p] = 0.0;"),
    "ssd_decay_sign": ("ssd", "const double a = exp(d * Ah);", "const double a = exp(-d * Ah);"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    kind, old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = os.path.join(str(mutant_dir), name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(str(mutant_dir), name + ".so"))
    if kind == "diag":
        args = _rand_diag(_rng(1), 2, 7, 3, 4)
        y = oracle.diag_scan(*args, library=lib)
        err = _rel(y, diag_closed_form(*args))
    else:
        args = _rand_ssd(_rng(1), 2, 6, 2, 3, 4)
        y = oracle.ssd_scan(*args, bidirectional=True, library=lib)
        err = _rel(y, ssd_closed_form(*args, bidirectional=True))
    assert err > 1e-6, "planted mistake %s was not caught (err %.3g)" % (name, err)
