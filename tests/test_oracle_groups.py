"""Pins of the oracle's groups of B, C for the SSD scan (CPU only).

The chunked scan's interface in "Some questions of Bi-Mamba2 and Hydra"
(Bi-Mamba2 issue 1) takes B, C of shape (Bs, L, ngroups, N); heads are split
evenly over the groups, head h reading group h // (H // G) (the Mamba
convention).  Pins: a non-recursive closed form indexed by group (both
directions), replicated groups reduce to one shared group, and planted
mistakes in the group indexing are caught.
"""
import math
import os

import numpy as np
import pytest

import oracle
from test_oracle import _rand_ssd, _rel, _rng

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")


def ssd_grouped_closed_form(x, dt, A, B, C, D, bidirectional):
    """sum_s (C_t^g . B_s^g) exp(A_h * span) dt_s x_s (+ reverse) + D_h x_t, g = h // (H // G)."""
    Bs, L, H, P = x.shape
    G = B.shape[2]
    y = np.zeros((Bs, L, H, P))
    for b in range(Bs):
        for h in range(H):
            g = h // (H // G)
            for t in range(L):
                acc = np.zeros(P)
                for s in range(L):
                    cb = float(np.dot(C[b, t, g], B[b, s, g]))
                    if s <= t:
                        span = sum(dt[b, r, h] for r in range(s + 1, t + 1))
                        acc += cb * math.exp(A[h] * span) * dt[b, s, h] * x[b, s, h]
                    if bidirectional and s >= t:
                        span = sum(dt[b, r, h] for r in range(t, s))
                        acc += cb * math.exp(A[h] * span) * dt[b, s, h] * x[b, s, h]
                y[b, t, h] = acc + D[h] * x[b, t, h]
    return y


def _grouped(seed, Bs=2, L=5, H=4, P=3, N=4, G=2):
    rng = _rng(seed)
    x, dt, A, _, _, D = _rand_ssd(rng, Bs, L, H, P, N)
    B = rng.standard_normal((Bs, L, G, N)) / math.sqrt(N)
    C = rng.standard_normal((Bs, L, G, N)) / math.sqrt(N)
    return x, dt, A, B, C, D


@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("bidir", [False, True])
def test_grouped_matches_closed_form(G, bidir):
    args = _grouped(20 + G, G=G)
    y = oracle.ssd_scan(*args, bidirectional=bidir)
    assert _rel(y, ssd_grouped_closed_form(*args, bidir)) < 1e-12


def test_replicated_groups_equal_one_group():
    x, dt, A, B, C, D = _grouped(31, G=1)
    B4, C4 = np.repeat(B, 4, axis=2), np.repeat(C, 4, axis=2)
    assert np.array_equal(oracle.ssd_scan(x, dt, A, B4, C4, D), oracle.ssd_scan(x, dt, A, B, C, D))


def test_heads_must_split_evenly():
    x, dt, A, B, C, D = _grouped(32, H=4, G=2)
    B3 = np.concatenate([B, B[:, :, :1]], axis=2)
    with pytest.raises(AssertionError):
        oracle.ssd_scan(x, dt, A, B3, B3, D)


GROUP_MUTANTS = {
    "group_index_modulo": ("const int64_t g = h / (H / G);", "const int64_t g = h % G;"),
    "C_from_group_zero": ("const double *Ct = C + ((b * L + t) * G + g) * N;",
                          "const double *Ct = C + ((b * L + t) * G + 0) * N;"),
}


@pytest.mark.parametrize("name", sorted(GROUP_MUTANTS))
def test_planted_group_mistake_is_caught(name, tmp_path):
    old, new = GROUP_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    path = str(tmp_path / (name + ".c"))
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, str(tmp_path / (name + ".so")))
    args = _grouped(40, G=2)
    err = _rel(oracle.ssd_scan(*args, library=lib), ssd_grouped_closed_form(*args, False))
    assert err > 1e-6, "planted mistake %s was not caught (err %.3g)" % (name, err)
