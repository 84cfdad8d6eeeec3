"""Pins of the oracle's gradients of the SSD scan (CPU only).

Reverse mode is written out by hand in the oracle; every gradient entry is
checked here against central finite differences of the oracle's forward
scan (fp64, step 1e-6: truncation error ~1e-12), on tiny random inputs --
unidirectional, bidirectional, with groups of B, C, and without D.  Planted
mistakes in the adjoint code are caught by the same check.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import forms
from test_oracle import _rand_ssd, _rng

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")
EPS = 1e-6


def _case(seed, Bs, L, H, P, N, G=1, bidir=False):
    rng = _rng(seed)
    x, dt, A, B, C, D = _rand_ssd(rng, Bs, L, H, P, N)
    if G > 1:
        B = rng.standard_normal((Bs, L, G, N)) / np.sqrt(N)
        C = rng.standard_normal((Bs, L, G, N)) / np.sqrt(N)
    dy = rng.standard_normal(x.shape)
    return dict(x=x, dt=dt, A_head=A, B=B, C=C, D=D), dy, bidir


def _fd_grads(args, dy, bidir):
    """d(sum(dy * y)) / d(each input) by central differences of the forward oracle."""
    out = {}
    for name in ("x", "dt", "A_head", "B", "C", "D"):
        base = args[name]
        if base is None:
            continue
        g = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            plus, minus = dict(args), dict(args)
            p, m = base.copy(), base.copy()
            p[idx] += EPS
            m[idx] -= EPS
            plus[name], minus[name] = p, m
            lp = float(np.sum(dy * oracle.ssd_scan(**plus, bidirectional=bidir)))
            lm = float(np.sum(dy * oracle.ssd_scan(**minus, bidirectional=bidir)))
            g[idx] = (lp - lm) / (2 * EPS)
        out[{"A_head": "dA"}.get(name, "d" + name)] = g
    return out


def _worst(an, fd):
    return max(float(np.max(np.abs(an[k] - fd[k]))) / max(1.0, float(np.max(np.abs(fd[k]))))
               for k in fd)


CASES = [
    # seed, Bs, L, H, P, N, G, bidirectional
    (1, 1, 5, 2, 2, 3, 1, False),
    (2, 2, 4, 1, 3, 2, 1, False),
    (3, 1, 6, 2, 2, 3, 1, True),
    (4, 1, 4, 4, 2, 2, 2, False),    # groups of B, C: dB, dC sum over a group's heads
    (5, 1, 5, 2, 2, 2, 2, True),     # one group per head, both directions
    (6, 1, 1, 1, 2, 2, 1, True),     # L = 1
]


@pytest.mark.parametrize("seed,Bs,L,H,P,N,G,bidir", CASES)
def test_gradients_match_finite_differences(seed, Bs, L, H, P, N, G, bidir):
    args, dy, bidir = _case(seed, Bs, L, H, P, N, G, bidir)
    an = oracle.ssd_scan_bwd(**args, dy=dy, bidirectional=bidir)
    fd = _fd_grads(args, dy, bidir)
    assert set(an) == set(fd)
    assert _worst(an, fd) < 1e-7


def test_gradients_without_D():
    args, dy, _ = _case(7, 1, 5, 2, 2, 3)
    args["D"] = None
    g = oracle.ssd_scan_bwd(**args, dy=dy)
    assert g["dD"] is None
    fd = _fd_grads(args, dy, False)
    assert _worst({k: g[k] for k in fd}, fd) < 1e-7


def test_single_head_width_one_equals_diagonal_gradients():
    """With P = 1 and one head the SSD scan is the diagonal scan with ED = 1,
    N states sharing one decay: the two oracles' gradients agree."""
    rng = _rng(8)
    Bs, L, N = 2, 6, 3
    x = rng.standard_normal((Bs, L, 1, 1))
    dt = np.log1p(np.exp(rng.standard_normal((Bs, L, 1)) - 1.0))
    Ah = np.array([-1.7])
    B = rng.standard_normal((Bs, L, N))
    C = rng.standard_normal((Bs, L, N))
    D = rng.standard_normal(1)
    dy = rng.standard_normal((Bs, L, 1, 1))
    s = oracle.ssd_scan_bwd(x, dt, Ah, B, C, D, dy)
    d = oracle.diag_scan_bwd(x[:, :, :, 0], dt, np.full((1, N), Ah[0]), B, C, D, dy[:, :, :, 0])
    assert np.allclose(s["dx"][:, :, :, 0], d["dx"], rtol=1e-12, atol=1e-12)
    assert np.allclose(s["ddt"], d["ddelta"], rtol=1e-12, atol=1e-12)
    assert np.allclose(s["dA"], d["dA"].sum(), rtol=1e-12, atol=1e-12)
    assert np.allclose(s["dB"], d["dB"], rtol=1e-12, atol=1e-12)
    assert np.allclose(s["dC"], d["dC"], rtol=1e-12, atol=1e-12)
    assert np.allclose(s["dD"], d["dD"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed,Bs,L,H,P,N,G,bidir,chunk", [
    (11, 1, 9, 2, 3, 4, 1, False, 4),      # ragged last chunk
    (12, 2, 13, 2, 2, 3, 1, True, 5),
    (13, 1, 17, 4, 3, 2, 2, False, 1),     # one step per chunk: the recurrence itself
    (14, 1, 11, 2, 2, 3, 2, True, 11),     # one chunk: the quadratic masked form
    (15, 1, 20, 2, 3, 4, 1, True, 64),     # chunk longer than L
    (16, 1, 24, 1, 2, 2, 1, False, 8),     # whole chunks only
])
def test_chunked_gradient_form_matches_sequential(seed, Bs, L, H, P, N, G, bidir, chunk):
    """The chunked form of the gradients (transposed chunk products, state
    gradient passed from the last chunk back) reaches the sequential
    reverse-mode result for every chunk size, to rounding."""
    rng = _rng(seed)
    x, dt, A, B, C, D = _rand_ssd(rng, Bs, L, H, P, N)
    if G > 1:
        B = rng.standard_normal((Bs, L, G, N)) / np.sqrt(N)
        C = rng.standard_normal((Bs, L, G, N)) / np.sqrt(N)
    dy = rng.standard_normal(x.shape)
    ref = oracle.ssd_scan_bwd(x, dt, A, B, C, D, dy, bidirectional=bidir)
    got = forms.ssd_scan_bwd_chunked(x, dt, A, B, C, D, dy, chunk=chunk, bidirectional=bidir)
    assert set(got) == set(ref)
    for k in ref:
        assert got[k].shape == ref[k].shape, k
        scale = max(1.0, float(np.max(np.abs(ref[k]))))
        assert float(np.max(np.abs(got[k] - ref[k]))) <= 1e-12 * scale, k


SSD_BWD_MUTANTS = {
    "adjoint_not_decayed": ("*gpn *= a;                             /* a_k Gb_k, carried to step k - 1 */",
                            "*gpn *= 1.0;                           /* a_k Gb_k, carried to step k - 1 */"),
    "dC_uses_entering_state": ("dcr[n] += gy[p] * hk[p * N + n];",
                               "dcr[n] += gy[p] * hprev[p * N + n];"),
    "ddt_decay_sign": ("ddt[(b * L + t) * H + h] += sdt + Ah * a * sda;",
                       "ddt[(b * L + t) * H + h] += sdt - Ah * a * sda;"),
    "dA_misses_dt": ("*dAh += dtv * a * sda;", "*dAh += a * sda;"),
    "dB_misses_dt": ("dbr[n] += dtv * *gpn * xr[p];", "dbr[n] += *gpn * xr[p];"),
    "dx_drops_D": ("if (D) dx[i] += D[h] * dy[i];", "if (D) dx[i] += 0.0 * dy[i];"),
    "reverse_direction_skipped": ("for (int dir = 0; dir < (bidirectional ? 2 : 1); ++dir)",
                                  "for (int dir = 0; dir < 1; ++dir)"),
}


@pytest.mark.parametrize("name", sorted(SSD_BWD_MUTANTS))
def test_planted_gradient_mistake_is_caught(name, tmp_path):
    old, new = SSD_BWD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = str(tmp_path / (name + ".c"))
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, str(tmp_path / (name + ".so")))
    args, dy, bidir = _case(9, 1, 5, 2, 2, 2, 2, True)
    an = oracle.ssd_scan_bwd(**args, dy=dy, bidirectional=bidir, library=lib)
    fd = _fd_grads(args, dy, bidir)    # the real forward oracle
    assert _worst(an, fd) > 1e-6, "planted mistake %s was not caught" % name


# ---- gradients of the scan with its options --------------------------------

def _case_opts(seed, Bs, L, H, P, N, G, bidir, opts):
    rng = _rng(seed)
    x, dt, A, B, C, D = _rand_ssd(rng, Bs, L, H, P, N)
    if G > 1:
        B = rng.standard_normal((Bs, L, G, N)) / np.sqrt(N)
        C = rng.standard_normal((Bs, L, G, N)) / np.sqrt(N)
    args = dict(x=x, dt=rng.standard_normal((Bs, L, H)) - 1.0, A_head=A, B=B, C=C, D=D)
    kw = dict(bidirectional=bidir)
    if "bias" in opts:
        args["dt_bias"] = 0.5 * rng.standard_normal(H)
    if "softplus" in opts:
        kw["dt_softplus"] = True
    if "limit" in opts:
        kw["dt_limit"] = (0.2, 0.8)      # clamps some steps at either bound
    if "z" in opts:
        args["z"] = rng.standard_normal(x.shape)
    if "h0" in opts:
        args["h0"] = 0.5 * rng.standard_normal((Bs, H, P, N))
    return args, kw, rng.standard_normal(x.shape)


def _fd_grads_opts(args, kw, dy):
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
            lp = float(np.sum(dy * oracle.ssd_scan(**plus, **kw)))
            lm = float(np.sum(dy * oracle.ssd_scan(**minus, **kw)))
            g[idx] = (lp - lm) / (2 * EPS)
        out[{"A_head": "dA", "dt_bias": "ddt_bias"}.get(name, "d" + name)] = g
    return out


OPT_CASES = [
    # seed, Bs, L, H, P, N, G, bidirectional, options
    (21, 1, 5, 2, 2, 3, 1, False, ("bias", "softplus", "limit", "z", "h0")),
    (22, 2, 4, 2, 2, 2, 2, True, ("bias", "softplus", "z")),
    (23, 1, 6, 1, 3, 2, 1, False, ("softplus", "h0")),
    (24, 1, 5, 2, 2, 2, 1, True, ("limit", "z")),
]


@pytest.mark.parametrize("seed,Bs,L,H,P,N,G,bidir,opts", OPT_CASES)
def test_option_gradients_match_finite_differences(seed, Bs, L, H, P, N, G, bidir, opts):
    """dz, ddt_bias, dh0 and the gradient with respect to the dt given
    (through the bias, softplus and clamp) against central differences of
    the forward oracle with the same options."""
    args, kw, dy = _case_opts(seed, Bs, L, H, P, N, G, bidir, opts)
    an = oracle.ssd_scan_bwd_ex(**args, dy=dy, **kw)
    fd = _fd_grads_opts(args, kw, dy)
    for k in an:
        assert (an[k] is None) == (k not in fd), k
    assert _worst({k: an[k] for k in fd}, fd) < 1e-7


def test_option_gradients_without_options_equal_plain_ones():
    args, kw, dy = _case_opts(25, 2, 5, 2, 2, 3, 1, True, ())
    an = oracle.ssd_scan_bwd_ex(**args, dy=dy, **kw)
    plain = oracle.ssd_scan_bwd(**args, dy=dy, **kw)
    for k in plain:
        assert np.array_equal(an[k], plain[k]), k


SSD_BWD_OPT_MUTANTS = {
    "gate_derivative_drops_term": (
        "if (dz) dz[i] = dy[i] * u[i] * sg * (1.0 + z[i] * (1.0 - sg));",
        "if (dz) dz[i] = dy[i] * u[i] * sg;"),
    "softplus_derivative_dropped": ("f = 1.0 / (1.0 + exp(-v));", "f = 1.0;"),
    "clamp_passes_gradient": ("if (s < dt_min || s > dt_max) f = 0.0;", "if (0) f = 0.0;"),
    "backward_ignores_initial_state": ("for (int64_t i = 0; i < PN; ++i) hist[i] = init ? init[i] : 0.0;",
                                       "for (int64_t i = 0; i < PN; ++i) hist[i] = 0.0;"),
}


@pytest.mark.parametrize("name", sorted(SSD_BWD_OPT_MUTANTS))
def test_planted_option_gradient_mistake_is_caught(name, tmp_path):
    old, new = SSD_BWD_OPT_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = str(tmp_path / (name + ".c"))
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, str(tmp_path / (name + ".so")))
    args, kw, dy = _case_opts(26, 1, 5, 2, 2, 2, 1, False, ("bias", "softplus", "limit", "z", "h0"))
    an = oracle.ssd_scan_bwd_ex(**args, dy=dy, **kw, library=lib)
    fd = _fd_grads_opts(args, kw, dy)   # the real forward oracle
    assert _worst({k: an[k] for k in fd}, fd) > 1e-6, "planted mistake %s was not caught" % name
