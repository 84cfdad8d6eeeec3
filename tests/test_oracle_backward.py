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


# ---- gradients of the scan with its options --------------------------------

def _case_opts(seed, Bs, L, ED, N, opts):
    rng = _rng(seed)
    x, _, A, B, C, D = _rand_diag(rng, Bs, L, ED, N)
    args = dict(x=x, delta=rng.standard_normal(x.shape) - 1.0, A=A, B=B, C=C, D=D)
    kw = {}
    if "bias" in opts:
        args["dt_bias"] = 0.5 * rng.standard_normal(ED)
    if "softplus" in opts:
        kw["dt_softplus"] = True
    if "limit" in opts:
        kw["dt_limit"] = (0.2, 0.8)      # clamps some steps at either bound
    if "z" in opts:
        args["z"] = rng.standard_normal(x.shape)
    if "h0" in opts:
        args["h0"] = 0.5 * rng.standard_normal((Bs, ED, N))
    return args, kw, rng.standard_normal(x.shape)


def _fd_grads_opts(args, kw, dy, library=None):
    out = {}
    for name, base in args.items():
        if base is None:
            continue
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            plus, minus = dict(args), dict(args)
            p, m = base.copy(), base.copy()
            p[idx] += EPS
            m[idx] -= EPS
            plus[name], minus[name] = p, m
            lp = float(np.sum(dy * oracle.diag_scan(**plus, **kw)))
            lm = float(np.sum(dy * oracle.diag_scan(**minus, **kw)))
            g[idx] = (lp - lm) / (2 * EPS)
        out[{"dt_bias": "ddt_bias"}.get(name, "d" + name)] = g
    return out


@pytest.mark.parametrize("seed,shape,opts", [
    (11, (2, 5, 2, 3), ("bias", "softplus", "limit", "z", "h0")),
    (12, (1, 6, 3, 2), ("softplus", "z")),
    (13, (2, 4, 2, 2), ("limit", "h0")),
    (14, (1, 5, 2, 3), ("bias", "limit")),   # the clamp keeps delta > 0 (in contract)
])
def test_option_gradients_match_finite_differences(seed, shape, opts):
    """dz, ddt_bias, dh0 and the gradient with respect to the delta given
    (through the bias, softplus and clamp) against central differences of
    the forward oracle with the same options."""
    args, kw, dy = _case_opts(seed, *shape, opts)
    an = oracle.diag_scan_bwd_ex(**args, dy=dy, **kw)
    fd = _fd_grads_opts(args, kw, dy)
    for k in an:
        assert (an[k] is None) == (k not in fd), k
    assert _worst({k: an[k] for k in fd}, fd) < 1e-7


def test_option_gradients_without_options_equal_plain_ones():
    args, kw, dy = _case_opts(15, 2, 5, 2, 3, ())
    an = oracle.diag_scan_bwd_ex(**args, dy=dy)
    plain = oracle.diag_scan_bwd(**args, dy=dy)
    for k in plain:
        assert np.array_equal(an[k], plain[k]), k


BWD_OPT_MUTANTS = {
    "gate_derivative_drops_term": (
        "if (dz) dz[i] = dy[i] * u[i] * sgm * (1.0 + z[i] * (1.0 - sgm));",
        "if (dz) dz[i] = dy[i] * u[i] * sgm;"),
    "softplus_derivative_dropped": ("fac = 1.0 / (1.0 + exp(-w));", "fac = 1.0;"),
    "clamp_passes_gradient": ("if (sv < dt_min || sv > dt_max) fac = 0.0;", "if (0) fac = 0.0;"),
    "backward_ignores_initial_state": ("for (int64_t n = 0; n < N; ++n) hist[n] = h0[c * N + n];",
                                       "for (int64_t n = 0; n < N; ++n) hist[n] = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(BWD_OPT_MUTANTS))
def test_planted_option_gradient_mistake_is_caught(name, tmp_path):
    old, new = BWD_OPT_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = str(tmp_path / (name + ".c"))
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, str(tmp_path / (name + ".so")))
    args, kw, dy = _case_opts(16, 2, 5, 2, 3, ("bias", "softplus", "limit", "z", "h0"))
    an = oracle.diag_scan_bwd_ex(**args, dy=dy, **kw, library=lib)
    fd = _fd_grads_opts(args, kw, dy)   # the real forward oracle
    assert _worst({k: an[k] for k in fd}, fd) > 1e-6, "planted mistake %s was not caught" % name
