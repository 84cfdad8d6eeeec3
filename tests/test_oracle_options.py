"""Pins of the oracle's scan options (CPU only).

The chunked scan's argument list in "Some questions of Bi-Mamba2 and Hydra"
(Bi-Mamba2 issue 1) carries dt_bias, dt_softplus, dt_limit, the gate z and
initial / final states.  Their plainest reading (the Mamba convention):
delta' = clamp(softplus(delta + dt_bias)); y = (scan + D x) * silu(z);
h_{-1} = h0; the final state is h_{L-1}.

The pins below do not re-call the oracle's own arithmetic: the closed forms
are written non-recursively (sums over sources with explicit decay spans),
softplus is numpy's logaddexp, the gate uses scipy's expit, the clamp is
np.clip.  Planted mistakes in the option code are caught by them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from test_oracle import _rand_diag, _rand_ssd, _rel, _rng

expit = pytest.importorskip("scipy.special").expit

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")


def _prep(delta, bias, lo, hi):
    """delta' = clip(softplus(delta + bias), lo, hi) with library routines."""
    return np.clip(np.logaddexp(0.0, delta + bias), lo, hi)


def diag_closed_form_ex(x, delta, A, B, C, D, h0, z):
    """Non-recursive form with an initial state:
    h_t[n] = exp(A[e,n] sum_{r<=t} d_r) h0[n] + sum_{s<=t} exp(A[e,n] sum_{s<r<=t} d_r) d_s B_s[n] x_s,
    y_t = (C_t . h_t + D x_t) * z_t * expit(z_t); returns (y, h_{L-1})."""
    Bs, L, ED = x.shape
    N = A.shape[1]
    y = np.zeros((Bs, L, ED))
    hf = np.zeros((Bs, ED, N))
    for b in range(Bs):
        for e in range(ED):
            for t in range(L):
                h = np.zeros(N)
                for n in range(N):
                    span0 = sum(delta[b, r, e] for r in range(0, t + 1))
                    h[n] = math.exp(A[e, n] * span0) * h0[b, e, n]
                    for s in range(t + 1):
                        span = sum(delta[b, r, e] for r in range(s + 1, t + 1))
                        h[n] += math.exp(A[e, n] * span) * delta[b, s, e] * B[b, s, n] * x[b, s, e]
                out = float(np.dot(C[b, t], h)) + D[e] * x[b, t, e]
                y[b, t, e] = out * z[b, t, e] * expit(z[b, t, e])
                if t == L - 1:
                    hf[b, e] = h
    return y, hf


def ssd_closed_form_ex(x, dt, A, B, C, D, h0, z):
    """Non-recursive single-direction SSD with an initial state (P x N per head):
    H_t = exp(A_h sum_{r<=t} dt_r) H0 + sum_{s<=t} exp(A_h sum_{s<r<=t} dt_r) dt_s x_s B_s^T,
    y_t = (H_t C_t + D_h x_t) * silu(z_t); returns (y, H_{L-1})."""
    Bs, L, H, P = x.shape
    N = B.shape[-1]
    y = np.zeros((Bs, L, H, P))
    hf = np.zeros((Bs, H, P, N))
    for b in range(Bs):
        for h in range(H):
            for t in range(L):
                span0 = sum(dt[b, r, h] for r in range(0, t + 1))
                St = math.exp(A[h] * span0) * h0[b, h]
                for s in range(t + 1):
                    span = sum(dt[b, r, h] for r in range(s + 1, t + 1))
                    St = St + math.exp(A[h] * span) * dt[b, s, h] * np.outer(x[b, s, h], B[b, s])
                out = St @ C[b, t] + D[h] * x[b, t, h]
                y[b, t, h] = out * z[b, t, h] * expit(z[b, t, h])
                if t == L - 1:
                    hf[b, h] = St
    return y, hf


def _diag_case(seed, Bs=2, L=6, ED=3, N=4):
    rng = _rng(seed)
    x, delta, A, B, C, D = _rand_diag(rng, Bs, L, ED, N)
    raw = rng.standard_normal((Bs, L, ED))          # delta before preprocessing
    bias = 0.5 * rng.standard_normal(ED)
    z = rng.standard_normal((Bs, L, ED))
    h0 = rng.standard_normal((Bs, ED, N))
    return x, raw, A, B, C, D, bias, z, h0


def _ssd_case(seed, Bs=2, L=6, H=2, P=3, N=4):
    rng = _rng(seed)
    x, dt, A, B, C, D = _rand_ssd(rng, Bs, L, H, P, N)
    raw = rng.standard_normal((Bs, L, H)) - 1.0
    bias = 0.5 * rng.standard_normal(H)
    z = rng.standard_normal((Bs, L, H, P))
    h0 = rng.standard_normal((Bs, H, P, N))
    return x, raw, A, B, C, D, bias, z, h0


LIMIT = (0.2, 1.2)


def _check_diag(library=None, seed=3):
    x, raw, A, B, C, D, bias, z, h0 = _diag_case(seed)
    y, hf = oracle.diag_scan(x, raw, A, B, C, D, dt_bias=bias, dt_softplus=True, dt_limit=LIMIT,
                             z=z, h0=h0, return_final_state=True, library=library)
    yr, hr = diag_closed_form_ex(x, _prep(raw, bias[None, None, :], *LIMIT), A, B, C, D, h0, z)
    return max(_rel(y, yr), _rel(hf, hr))


def _check_ssd(library=None, seed=4):
    x, raw, A, B, C, D, bias, z, h0 = _ssd_case(seed)
    y, hf = oracle.ssd_scan(x, raw, A, B, C, D, dt_bias=bias, dt_softplus=True, dt_limit=LIMIT,
                            z=z, h0=h0, return_final_state=True, library=library)
    yr, hr = ssd_closed_form_ex(x, _prep(raw, bias[None, None, :], *LIMIT), A, B, C, D, h0, z)
    return max(_rel(y, yr), _rel(hf, hr))


@pytest.mark.parametrize("seed", [3, 5])
def test_diag_options_match_closed_form(seed):
    assert _check_diag(seed=seed) < 1e-12


@pytest.mark.parametrize("seed", [4, 6])
def test_ssd_options_match_closed_form(seed):
    assert _check_ssd(seed=seed) < 1e-12


def test_limit_is_active_in_the_pins():
    """The pin inputs exercise both ends of the clamp and the softplus."""
    x, raw, A, B, C, D, bias, z, h0 = _diag_case(3)
    sp = np.logaddexp(0.0, raw + bias)
    assert (sp < LIMIT[0]).any() and (sp > LIMIT[1]).any()


def test_no_options_is_the_plain_scan():
    x, delta, A, B, C, D = _rand_diag(_rng(7), 2, 5, 3, 4)
    y0 = oracle.diag_scan(x, delta, A, B, C, D)
    y1, hf = oracle.diag_scan(x, delta, A, B, C, D, h0=np.zeros((2, 3, 4)), return_final_state=True)
    assert np.array_equal(y0, y1)


@pytest.mark.parametrize("split", [1, 3, 5])
def test_diag_state_io_splits_the_sequence(split):
    """Running [0, split) and then [split, L) from its final state equals one run."""
    x, delta, A, B, C, D = _rand_diag(_rng(8), 2, 7, 3, 4)
    h0 = _rng(9).standard_normal((2, 3, 4))
    y, hf = oracle.diag_scan(x, delta, A, B, C, D, h0=h0, return_final_state=True)
    sl, sr = slice(0, split), slice(split, None)
    ya, ha = oracle.diag_scan(x[:, sl], delta[:, sl], A, B[:, sl], C[:, sl], D, h0=h0,
                              return_final_state=True)
    yb, hb = oracle.diag_scan(x[:, sr], delta[:, sr], A, B[:, sr], C[:, sr], D, h0=ha,
                              return_final_state=True)
    assert _rel(np.concatenate([ya, yb], axis=1), y) < 1e-13
    assert _rel(hb, hf) < 1e-13


@pytest.mark.parametrize("split", [1, 4])
def test_ssd_state_io_splits_the_sequence(split):
    x, dt, A, B, C, D = _rand_ssd(_rng(10), 2, 6, 2, 3, 4)
    h0 = _rng(11).standard_normal((2, 2, 3, 4))
    y, hf = oracle.ssd_scan(x, dt, A, B, C, D, h0=h0, return_final_state=True)
    sl, sr = slice(0, split), slice(split, None)
    ya, ha = oracle.ssd_scan(x[:, sl], dt[:, sl], A, B[:, sl], C[:, sl], D, h0=h0,
                             return_final_state=True)
    yb, hb = oracle.ssd_scan(x[:, sr], dt[:, sr], A, B[:, sr], C[:, sr], D, h0=ha,
                             return_final_state=True)
    assert _rel(np.concatenate([ya, yb], axis=1), y) < 1e-13
    assert _rel(hb, hf) < 1e-13


def test_ssd_state_io_is_single_direction_only():
    x, dt, A, B, C, D = _rand_ssd(_rng(12), 1, 4, 1, 2, 3)
    with pytest.raises(ValueError):
        oracle.ssd_scan(x, dt, A, B, C, D, bidirectional=True, return_final_state=True)


def test_bidirectional_gate_and_dt_options():
    """Bidirectional with the pointwise options: equals the plain bidirectional
    scan of the preprocessed dt, gated afterwards (library softplus / expit)."""
    x, raw, A, B, C, D, bias, z, _ = _ssd_case(13)
    y = oracle.ssd_scan(x, raw, A, B, C, D, bidirectional=True, dt_bias=bias, dt_softplus=True,
                        z=z)
    plain = oracle.ssd_scan(x, np.logaddexp(0.0, raw + bias), A, B, C, D, bidirectional=True)
    assert _rel(y, plain * z * expit(z)) < 1e-13


OPTION_MUTANTS = {
    "bias_after_softplus": ("if (bias) d += bias[k];\n    if (softplus) d = log1p(exp(d));",
                            "if (softplus) d = log1p(exp(d));\n    if (bias) d += bias[k];"),
    "limit_bounds_swapped": ("d = fmin(fmax(d, dmin), dmax);", "d = fmax(fmin(d, dmin), dmax);"),
    "gate_is_sigmoid": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "diag_gate_skips_D": ("y[i] = z ? out * silu(z[i]) : out;",
                          "y[i] = z ? acc * silu(z[i]) + (out - acc) : out;"),
    "diag_h0_ignored": ("for (int64_t n = 0; n < N; ++n) h[n] = h0[(b * ED + e) * N + n];",
                        "for (int64_t n = 0; n < N; ++n) h[n] = 0.0 * h0[(b * ED + e) * N + n];"),
    "diag_h0_transposed": ("h[n] = h0[(b * ED + e) * N + n];", "h[n] = h0[(b * N + n) * ED + e];"),
    "ssd_h0_ignored": ("state[i] = h0 ? h0[u * P * N + i] : 0.0;", "state[i] = 0.0;"),
    "ssd_final_state_stale": ("h_final[u * P * N + i] = state[i];",
                              "h_final[u * P * N + i] = h0 ? h0[u * P * N + i] : 0.0;"),
    "ssd_gate_before_D": ("y[o + p] = D ? D[h] * x[o + p] : 0.0;",
                          "y[o + p] = D ? D[h] * x[o + p] / (z ? silu(z[o + p]) : 1.0) : 0.0;"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_option_mutants")


@pytest.mark.parametrize("name", sorted(OPTION_MUTANTS))
def test_planted_option_mistake_is_caught(name, mutant_dir):
    old, new = OPTION_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = os.path.join(str(mutant_dir), name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(str(mutant_dir), name + ".so"))
    err = max(_check_diag(library=lib), _check_ssd(library=lib))
    assert err > 1e-6, "planted mistake %s was not caught (err %.3g)" % (name, err)
