"""Pins of the oracle's gradients of the diagonal scan (CPU only).

Reverse mode is written out by hand in the oracle; here every gradient entry
is checked against central finite differences of the oracle's forward scan
(fp64, step 1e-6: truncation error ~1e-12), on tiny random inputs.  Planted
mistakes in the adjoint code are caught by the same check.
"""
import os

import numpy as np
import pytest

import oracle
from test_oracle import _rand_diag, _rng

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")
EPS = 1e-6


def _fd_grads(x, delta, A, B, C, D, dy, library=None):
    """d(sum(dy * y)) / d(each input) by central differences of the forward oracle."""
    args = dict(x=x, delta=delta, A=A, B=B, C=C, D=D)
    out = {}
    for name in ("x", "delta", "A", "B", "C", "D"):
        base = args[name]
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            plus, minus = dict(args), dict(args)
            p, m = base.copy(), base.copy()
            p[idx] += EPS
            m[idx] -= EPS
            plus[name], minus[name] = p, m
            lp = float(np.sum(dy * oracle.diag_scan(**plus, library=library)))
            lm = float(np.sum(dy * oracle.diag_scan(**minus, library=library)))
            g[idx] = (lp - lm) / (2 * EPS)
        out["d" + name] = g
    return out


def _case(seed, Bs=2, L=5, ED=2, N=3):
    rng = _rng(seed)
    x, delta, A, B, C, D = _rand_diag(rng, Bs, L, ED, N)
    dy = rng.standard_normal(x.shape)
    return x, delta, A, B, C, D, dy


def _worst(an, fd):
    return max(float(np.max(np.abs(an[k] - fd[k]))) / max(1.0, float(np.max(np.abs(fd[k]))))
               for k in fd)


@pytest.mark.parametrize("seed,shape", [(1, (2, 5, 2, 3)), (2, (1, 7, 3, 4)), (3, (1, 1, 2, 2))])
def test_gradients_match_finite_differences(seed, shape):
    x, delta, A, B, C, D, dy = _case(seed, *shape)
    an = oracle.diag_scan_bwd(x, delta, A, B, C, D, dy)
    fd = _fd_grads(x, delta, A, B, C, D, dy)
    assert set(an) == set(fd)
    assert _worst(an, fd) < 1e-7


def test_gradients_without_D():
    x, delta, A, B, C, D, dy = _case(4)
    g = oracle.diag_scan_bwd(x, delta, A, B, C, None, dy)
    assert g["dD"] is None
    g2 = oracle.diag_scan_bwd(x, delta, A, B, C, np.zeros_like(D), dy)
    assert np.array_equal(g["dx"], g2["dx"]) and np.array_equal(g["ddelta"], g2["ddelta"])


BWD_MUTANTS = {
    "decay_term_sign": ("sdd += g[n] * (A[e * N + n] * a * hprev + B[r + n] * xv);",
                        "sdd += g[n] * (-A[e * N + n] * a * hprev + B[r + n] * xv);"),
    "adjoint_not_decayed": ("g[n] *= a;                             /* a_t g_t",
                            "g[n] *= 1.0;                           /* a_t g_t"),
    "dC_uses_entering_state": ("lC[t * N + n] += gy * hist[(t + 1) * N + n];",
                               "lC[t * N + n] += gy * hist[t * N + n];"),
    "dx_drops_D": ("dx[i] = sdx + (D ? D[e] * gy : 0.0);", "dx[i] = sdx;"),
    "dA_misses_delta": ("lA[n] += g[n] * dl * a * hprev;", "lA[n] += g[n] * a * hprev;"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_planted_gradient_mistake_is_caught(name, tmp_path):
    old, new = BWD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = str(tmp_path / (name + ".c"))
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, str(tmp_path / (name + ".so")))
    x, delta, A, B, C, D, dy = _case(5)
    an = oracle.diag_scan_bwd(x, delta, A, B, C, D, dy, library=lib)
    fd = _fd_grads(x, delta, A, B, C, D, dy)    # the real forward oracle
    assert _worst(an, fd) > 1e-6, "planted mistake %s was not caught" % name
