"""Pins for the fp64 oracle (CPU only).

Every check here compares the oracle with something other than itself: the
worked example printed on the pages, closed forms of the recurrence evaluated
by brute force, the other forms the pages compare (Blelloch, chunkwise,
parallel retention), invariances, and special cases with textbook answers.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import forms
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = np.array([float(t) for t in v.split()])
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_diag(rng, Bs, L, ED, N):
    x = rng.standard_normal((Bs, L, ED))
    delta = np.log1p(np.exp(rng.standard_normal((Bs, L, ED)) - 1.0))
    A = -(np.arange(N) + 1.0)[None, :] * np.exp(0.1 * rng.standard_normal((ED, N)))
    B = rng.standard_normal((Bs, L, N))
    C = rng.standard_normal((Bs, L, N))
    D = rng.standard_normal(ED)
    return x, delta, A, B, C, D


def _rand_ssd(rng, Bs, L, H, P, N):
    x = rng.standard_normal((Bs, L, H, P))
    dt = np.log1p(np.exp(rng.standard_normal((Bs, L, H)) - 2.0))
    A = -np.exp(rng.uniform(0.0, math.log(16.0), H))
    B = rng.standard_normal((Bs, L, N)) / math.sqrt(N)
    C = rng.standard_normal((Bs, L, N)) / math.sqrt(N)
    D = rng.standard_normal(H)
    return x, dt, A, B, C, D


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))


# ---------------------------------------------------------------------------
# The worked example printed on the pages
# ---------------------------------------------------------------------------

def test_cumsum_worked_example_blelloch_sweeps():
    g = _read_golden("cumsum_worked_example.txt")
    up = forms.blelloch_upsweep_cumsum(g["input"])
    np.testing.assert_array_equal(up, g["after_upsweep"])
    down = forms.blelloch_downsweep_cumsum(up)
    np.testing.assert_array_equal(down, g["after_downsweep"])


def test_cumsum_worked_example_through_diag_oracle():
    # a = exp(delta*A) = 1 and b = delta*B*x = x: the recurrence is a cumsum.
    g = _read_golden("cumsum_worked_example.txt")
    L = g["input"].shape[0]
    x = g["input"].reshape(1, L, 1)
    ones = np.ones((1, L, 1))
    y = oracle.diag_scan(x, ones, np.zeros((1, 1)), ones, ones, None)
    np.testing.assert_array_equal(y.ravel(), g["after_downsweep"])


def test_cumsum_worked_example_through_pair_scan():
    g = _read_golden("cumsum_worked_example.txt")
    h = forms.blelloch_linear_scan(np.ones(8), g["input"])
    np.testing.assert_array_equal(h, g["after_downsweep"])


def test_page_upsweep_needs_power_of_two():
    with pytest.raises(ValueError):
        forms.blelloch_upsweep_cumsum(np.arange(6.0))


# ---------------------------------------------------------------------------
# Closed forms, brute force on tiny inputs
# ---------------------------------------------------------------------------

def diag_closed_form(x, delta, A, B, C, D):
    """y_t = sum_{s<=t} sum_n C_t[n] exp(A[e,n] sum_{s<r<=t} delta_r) delta_s B_s[n] x_s + D x_t."""
    Bs, L, ED = x.shape
    N = A.shape[1]
    y = np.zeros((Bs, L, ED))
    for b in range(Bs):
        for e in range(ED):
            for t in range(L):
                acc = 0.0
                for s in range(t + 1):
                    span = sum(delta[b, r, e] for r in range(s + 1, t + 1))
                    for n in range(N):
                        acc += (C[b, t, n] * math.exp(A[e, n] * span) * delta[b, s, e]
                                * B[b, s, n] * x[b, s, e])
                y[b, t, e] = acc + (D[e] * x[b, t, e] if D is not None else 0.0)
    return y


def ssd_closed_form(x, dt, A, B, C, D, bidirectional):
    """Forward: sum_{s<=t} (C_t.B_s) exp(A_h sum_{s<r<=t} dt_r) dt_s x_s.
    Reverse:    sum_{s>=t} (C_t.B_s) exp(A_h sum_{t<=r<s} dt_r) dt_s x_s.
    Plus D_h x_t once."""
    Bs, L, H, P = x.shape
    y = np.zeros((Bs, L, H, P))
    for b in range(Bs):
        for h in range(H):
            for t in range(L):
                acc = np.zeros(P)
                for s in range(L):
                    cb = float(np.dot(C[b, t], B[b, s]))
                    if s <= t:
                        span = sum(dt[b, r, h] for r in range(s + 1, t + 1))
                        acc += cb * math.exp(A[h] * span) * dt[b, s, h] * x[b, s, h]
                    if bidirectional and s >= t:
                        span = sum(dt[b, r, h] for r in range(t, s))
                        acc += cb * math.exp(A[h] * span) * dt[b, s, h] * x[b, s, h]
                y[b, t, h] = acc + (D[h] * x[b, t, h] if D is not None else 0.0)
    return y


@pytest.mark.parametrize("seed,Bs,L,ED,N", [(0, 1, 1, 1, 1), (1, 2, 5, 3, 4), (2, 1, 9, 2, 3),
                                             (3, 2, 7, 3, 2)])
def test_diag_matches_closed_form(seed, Bs, L, ED, N):
    args = _rand_diag(_rng(seed), Bs, L, ED, N)
    assert _rel(oracle.diag_scan(*args), diag_closed_form(*args)) < 1e-12


@pytest.mark.parametrize("bidir", [False, True])
@pytest.mark.parametrize("seed,Bs,L,H,P,N", [(0, 1, 1, 1, 1, 1), (1, 2, 6, 2, 3, 4),
                                              (2, 1, 9, 3, 2, 2)])
def test_ssd_matches_closed_form(seed, Bs, L, H, P, N, bidir):
    args = _rand_ssd(_rng(seed), Bs, L, H, P, N)
    y = oracle.ssd_scan(*args, bidirectional=bidir)
    assert _rel(y, ssd_closed_form(*args, bidirectional=bidir)) < 1e-12


# ---------------------------------------------------------------------------
# Agreement of the sequential, Blelloch and chunkwise forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L", [1, 2, 6, 8, 13, 64, 100])
def test_diag_blelloch_form_agrees(L):
    args = _rand_diag(_rng(L), 2, L, 5, 4)
    assert _rel(forms.diag_scan_blelloch(*args), oracle.diag_scan(*args)) < 1e-12


@pytest.mark.parametrize("chunk", [1, 2, 3, 5, 37])
def test_diag_chunked_form_agrees(chunk):
    args = _rand_diag(_rng(100 + chunk), 2, 37, 4, 6)
    assert _rel(forms.diag_scan_chunked(*args, chunk=chunk), oracle.diag_scan(*args)) < 1e-12


@pytest.mark.parametrize("bidir", [False, True])
@pytest.mark.parametrize("chunk", [1, 7, 16, 64, 128, 150])
def test_ssd_chunked_form_agrees(chunk, bidir):
    args = _rand_ssd(_rng(7 + chunk), 2, 150, 2, 3, 8)
    y_seq = oracle.ssd_scan(*args, bidirectional=bidir)
    y_chk = forms.ssd_scan_chunked(*args, chunk=chunk, bidirectional=bidir)
    assert _rel(y_chk, y_seq) < 1e-12


def test_ssd_chunk_size_invariance_long_chunks():
    # Chunks as long as the benchmark's (256) over a ragged length.
    args = _rand_ssd(_rng(11), 1, 300, 1, 4, 16)
    ys = [forms.ssd_scan_chunked(*args, chunk=q) for q in (64, 128, 256, 300)]
    for y in ys[1:]:
        assert _rel(y, ys[0]) < 1e-12
    assert _rel(ys[0], oracle.ssd_scan(*args)) < 1e-12


# ---------------------------------------------------------------------------
# Invariances and special cases
# ---------------------------------------------------------------------------

def test_bidirectional_reversal_equivariance():
    x, dt, A, B, C, D = _rand_ssd(_rng(5), 2, 23, 3, 4, 5)
    y = oracle.ssd_scan(x, dt, A, B, C, D, bidirectional=True)
    f = lambda t: np.ascontiguousarray(t[:, ::-1])
    y_flip = oracle.ssd_scan(f(x), f(dt), A, f(B), f(C), D, bidirectional=True)
    assert _rel(f(y_flip), y) < 1e-12


def test_bidirectional_is_forward_plus_flipped_forward():
    x, dt, A, B, C, D = _rand_ssd(_rng(6), 1, 17, 2, 3, 4)
    f = lambda t: np.ascontiguousarray(t[:, ::-1])
    fwd = oracle.ssd_scan(x, dt, A, B, C, None)
    rev = f(oracle.ssd_scan(f(x), f(dt), A, f(B), f(C), None))
    y = oracle.ssd_scan(x, dt, A, B, C, D, bidirectional=True)
    assert _rel(y, fwd + rev + D[None, None, :, None] * x) < 1e-12


def test_single_step():
    x, delta, A, B, C, D = _rand_diag(_rng(8), 3, 1, 4, 5)
    y = oracle.diag_scan(x, delta, A, B, C, D)
    want = delta * x * np.einsum("bln,bln->bl", C, B)[:, :, None] + D * x
    assert _rel(y, want) < 1e-14


def test_memoryless_limit():
    # A -> -inf with delta > 0: exp(delta A) underflows to 0, no memory.
    x, delta, A, B, C, D = _rand_diag(_rng(9), 2, 11, 3, 4)
    delta = 0.5 + 0.5 * np.abs(delta)
    A = np.full_like(A, -1e4)
    y = oracle.diag_scan(x, delta, A, B, C, D)
    want = delta * x * np.einsum("bln,bln->bl", C, B)[:, :, None] + D * x
    assert _rel(y, want) < 1e-14


def test_memoryless_limit_bidirectional_counts_diagonal_twice():
    x, dt, A, B, C, D = _rand_ssd(_rng(10), 2, 9, 2, 3, 4)
    dt = 0.5 + np.abs(dt)
    A = np.full_like(A, -1e4)
    y = oracle.ssd_scan(x, dt, A, B, C, D, bidirectional=True)
    cb = np.einsum("bln,bln->bl", C, B)
    want = 2.0 * dt[..., None] * x * cb[:, :, None, None] + D[None, None, :, None] * x
    assert _rel(y, want) < 1e-14


def test_linear_attention_limit():
    # A = 0, delta = 1: y = tril(C B^T) x + D x (unnormalised causal linear attention).
    x, _, A, B, C, D = _rand_diag(_rng(12), 2, 13, 3, 4)
    y = oracle.diag_scan(x, np.ones_like(x), np.zeros_like(A), B, C, D)
    G = np.tril(np.einsum("btn,bsn->bts", C, B))
    want = np.einsum("bts,bse->bte", G, x) + D * x
    assert _rel(y, want) < 1e-12


def test_retention_parallel_form():
    # SSD with dt = 1 and A_h = log(gamma_h) is retention: the parallel form
    # (Q K^T * D_gamma) V with D_gamma[t, s] = gamma^(t-s) for s <= t.
    rng = _rng(13)
    Bs, L, H, P, N = 2, 16, 4, 3, 4
    x, _, _, B, C, _ = _rand_ssd(rng, Bs, L, H, P, N)
    gamma = 1.0 - 2.0 ** (-5.0 - np.arange(H))
    y = oracle.ssd_scan(x, np.ones((Bs, L, H)), np.log(gamma), B, C, None)
    t = np.arange(L)
    for h in range(H):
        Dg = np.where(t[:, None] >= t[None, :], gamma[h] ** (t[:, None] - t[None, :]), 0.0)
        want = np.einsum("bts,bsp->btp", np.einsum("btn,bsn->bts", C, B) * Dg, x[:, :, h])
        assert _rel(y[:, :, h], want) < 1e-12


def test_ssd_single_head_width_one_equals_diag():
    # P = 1, one head: the SSD recurrence is the diagonal scan with ED = 1 and
    # the same decay for every state.
    x, dt, A, B, C, D = _rand_ssd(_rng(14), 2, 21, 1, 1, 6)
    y_ssd = oracle.ssd_scan(x, dt, A, B, C, D)
    y_diag = oracle.diag_scan(x[:, :, :, 0], dt, np.full((1, 6), A[0]), B, C, D)
    assert _rel(y_ssd[:, :, :, 0], y_diag) < 1e-14


def test_zero_input_gives_zero_output():
    x, delta, A, B, C, D = _rand_diag(_rng(15), 1, 8, 2, 3)
    y = oracle.diag_scan(np.zeros_like(x), delta, A, B, C, D)
    assert np.all(y == 0.0)


def test_sampled_channels_match_full_run():
    x, delta, A, B, C, D = _rand_diag(_rng(16), 2, 10, 5, 3)
    full = oracle.diag_scan(x, delta, A, B, C, D)
    part = oracle.diag_scan(x, delta, A, B, C, D, channels=(3, 7))
    flat = lambda y: y.transpose(0, 2, 1).reshape(10, 10)
    assert np.array_equal(flat(part)[3:7], flat(full)[3:7])
    assert np.isnan(flat(part)[:3]).all() and np.isnan(flat(part)[7:]).all()


def test_workload_inputs_feed_the_oracle():
    inp = workloads.diag_inputs(2, 9, 3, 4, "bf16", seed=0)
    y = oracle.diag_scan(**inp)
    args = [inp[k].double().numpy() for k in ("x", "delta", "A", "B", "C", "D")]
    assert _rel(y, diag_closed_form(*args)) < 1e-12
