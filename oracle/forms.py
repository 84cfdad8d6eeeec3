"""Second and third forms of the scan, in fp64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  These exist to pin the
sequential oracle: the pages compare a sequential form, a Blelloch parallel
scan and a chunkwise form, and state that their results must agree.

* ``blelloch_cumsum`` -- the scalar up-sweep / down-sweep on a power-of-two
  array, step for step as described in "scan output is different between
  sequential and parallel versions" (mamba.py issue 26, the two answers that
  describe the reduction step and the down-sweep).  Its worked example turns
  [1..8] into the prefix sums [1, 3, 6, 10, 15, 21, 28, 36].
* ``blelloch_linear_scan`` -- the same two sweeps over (a, b) pairs of the
  first-order recurrence h_t = a_t h_{t-1} + b_t, using the associative
  operator (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2).  Any length is handled
  by padding with the identity (1, 0) (the page's version needs a power of
  two).
* ``diag_scan_blelloch`` / ``diag_scan_chunked`` -- the diagonal selective scan
  through those two forms.
* ``ssd_scan_chunked`` -- the chunked scalar-decay (SSD) form: per-chunk
  cumulative sums of dt*A, the masked C B^T intra-chunk product built from
  differences of cumulative sums (the numerically stable segment sum that
  "Some questions of Bi-Mamba2 and Hydra" discusses), per-chunk states,
  state passing across chunks and
  the inter-chunk output; optionally with the reversed direction computed from
  the same chunks (no flipped copy), as that page describes.
* ``ssd_scan_bwd_chunked`` -- the gradients of the SSD scan in the same
  chunked shape (the chunked backward pass that page names): transposed chunk
  products and a state gradient passed from the last chunk to the first.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Blelloch up-sweep / down-sweep
# ---------------------------------------------------------------------------

def blelloch_upsweep_cumsum(X):
    """Reduction (up-sweep) step on a 1-D power-of-two array, in place order.

    Level k pairs the elements at stride 2**k and adds each pair's first
    element into its second.  Returns the array after all log2(L) levels.
    """
    X = np.array(X, dtype=np.float64)
    L = X.shape[0]
    levels = int(math.log2(L))
    if 2 ** levels != L:
        raise ValueError("the page's up-sweep needs a power-of-two length")
    for k in range(levels):
        right = np.arange(2 ** (k + 1) - 1, L, 2 ** (k + 1))
        left = right - 2 ** k
        X[right] += X[left]
    return X


def blelloch_downsweep_cumsum(X):
    """Down-sweep on the output of the up-sweep; gives the inclusive prefix sum.

    For k = log2(L)-1 .. 0 take the sub-array of every 2**k-th element
    starting at index 2**k - 1, view it as pairs, and add to the first element
    of every pair (but the first) the second element of the previous pair.
    """
    X = np.array(X, dtype=np.float64)
    L = X.shape[0]
    levels = int(math.log2(L))
    for k in range(levels - 1, -1, -1):
        sub = np.arange(2 ** k - 1, L, 2 ** k)
        npairs = sub.shape[0] // 2
        firsts = sub[2:2 * npairs:2]          # first element of pairs 1..npairs-1
        prev_seconds = sub[1:2 * npairs - 2:2]  # second element of pairs 0..npairs-2
        X[firsts] += X[prev_seconds]
    return X


def blelloch_cumsum(X):
    return blelloch_downsweep_cumsum(blelloch_upsweep_cumsum(X))


def _combine(a1, b1, a2, b2):
    """(a1, b1) o (a2, b2): apply step 1 then step 2 of h -> a h + b."""
    return a1 * a2, a2 * b1 + b2


def blelloch_linear_scan(a, b):
    """Inclusive scan of h_t = a_t h_{t-1} + b_t (h_{-1} = 0) along the last axis.

    a, b: arrays of equal shape (..., L).  Returns h (..., L).  The two sweeps
    are the page's, with '+' replaced by the operator above; lengths that are
    not a power of two are padded at the end with the identity (1, 0).
    """
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    L = a.shape[-1]
    P2 = 1 if L <= 1 else 2 ** int(math.ceil(math.log2(L)))
    pad = [(0, 0)] * (a.ndim - 1) + [(0, P2 - L)]
    A = np.pad(a, pad, constant_values=1.0)
    Bv = np.pad(b, pad, constant_values=0.0)
    levels = int(math.log2(P2)) if P2 > 1 else 0
    for k in range(levels):  # up-sweep
        right = np.arange(2 ** (k + 1) - 1, P2, 2 ** (k + 1))
        left = right - 2 ** k
        A[..., right], Bv[..., right] = _combine(A[..., left], Bv[..., left],
                                                 A[..., right], Bv[..., right])
    for k in range(levels - 1, -1, -1):  # down-sweep
        sub = np.arange(2 ** k - 1, P2, 2 ** k)
        npairs = sub.shape[0] // 2
        firsts = sub[2:2 * npairs:2]
        prev_seconds = sub[1:2 * npairs - 2:2]
        A[..., firsts], Bv[..., firsts] = _combine(A[..., prev_seconds], Bv[..., prev_seconds],
                                                   A[..., firsts], Bv[..., firsts])
    return Bv[..., :L]


# ---------------------------------------------------------------------------
# Diagonal selective scan through the parallel and chunkwise forms
# ---------------------------------------------------------------------------

def _f64(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def diag_scan_blelloch(x, delta, A, B, C, D=None):
    """Diagonal scan with the state recurrence solved by ``blelloch_linear_scan``."""
    x, delta, A, B, C, D = map(_f64, (x, delta, A, B, C, D))
    # a, b over (Bs, ED, N, L)
    a = np.exp(np.einsum("ble,en->benl", delta, A))
    u = np.einsum("ble,ble,bln->benl", delta, x, B)
    h = blelloch_linear_scan(a, u)
    y = np.einsum("bln,benl->ble", C, h)
    if D is not None:
        y = y + D[None, None, :] * x
    return y


def diag_scan_chunked(x, delta, A, B, C, D=None, chunk: int = 16):
    """Chunkwise diagonal scan with a carried state.

    Each chunk runs the recurrence from a zero state, then adds the carried
    state's contribution C_t . (prod of decays since the chunk start) * h_in,
    and passes h_out = (prod of all decays in the chunk) * h_in + h_local_end.
    """
    x, delta, A, B, C, D = map(_f64, (x, delta, A, B, C, D))
    Bs, L, ED = x.shape
    N = A.shape[1]
    y = np.zeros((Bs, L, ED))
    h_in = np.zeros((Bs, ED, N))
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        h_loc = np.zeros((Bs, ED, N))
        decay = np.ones((Bs, ED, N))
        for t in range(c0, c1):
            a = np.exp(delta[:, t, :, None] * A[None])
            h_loc = a * h_loc + (delta[:, t, :] * x[:, t, :])[:, :, None] * B[:, t, None, :]
            decay = decay * a
            y[:, t, :] = np.einsum("bn,ben->be", C[:, t, :], h_loc + decay * h_in)
        h_in = decay * h_in + h_loc
    if D is not None:
        y = y + D[None, None, :] * x
    return y


# ---------------------------------------------------------------------------
# Chunked scalar-decay (SSD) form
# ---------------------------------------------------------------------------

def ssd_scan_chunked(x, dt, A_head, B, C, D=None, chunk: int = 64, bidirectional: bool = False):
    """Chunked SSD scan, steps in the order of the chunked pipeline.

    x: (Bs, L, H, P); dt: (Bs, L, H); A_head: (H); B, C: (Bs, L, N) or
    (Bs, L, 1, N); D: (H) or None.  For every (b, h) and chunk of Q rows:

    1. dA_r = dt_r A_h, cum = inclusive prefix sum of dA inside the chunk,
       excl = cum - dA (exclusive prefix), tot = cum at the chunk's end.
    2. G = C_chunk B_chunk^T                            (Q x Q)
    3. forward intra-chunk:  Y[t] += sum_{s<=t} G[t,s] exp(cum_t - cum_s) dt_s x_s
       reverse intra-chunk:  Y[t] += sum_{s>=t} G[t,s] exp(excl_s - excl_t) dt_s x_s
    4. chunk states:  S_f = sum_s exp(tot - cum_s) dt_s x_s (x) B_s
                      S_r = sum_s exp(excl_s) dt_s x_s (x) B_s
    5. state passing: forward chunks in order, S_in <- exp(tot) S_in + S_f;
                      reverse chunks from the last, R_in <- exp(tot) R_in + S_r
    6. inter-chunk output: forward  Y[t] += exp(cum_t) C_t S_in^T
                           reverse  Y[t] += exp(tot - excl_t) C_t R_in^T
    7. y = Y (+ D_h x)
    Every exponent above is <= 0 when dt A_h <= 0.
    """
    x, dt, A_head, B, C, D = map(_f64, (x, dt, A_head, B, C, D))
    if B.ndim == 4:
        B, C = B[:, :, 0, :], C[:, :, 0, :]
    Bs, L, H, P = x.shape
    N = B.shape[-1]
    y = np.zeros((Bs, L, H, P))
    bounds = [(c0, min(L, c0 + chunk)) for c0 in range(0, L, chunk)]
    for b in range(Bs):
        for h in range(H):
            pieces = []
            for (c0, c1) in bounds:
                dA = dt[b, c0:c1, h] * A_head[h]
                cum = np.cumsum(dA)
                excl = cum - dA
                tot = cum[-1]
                G = C[b, c0:c1] @ B[b, c0:c1].T
                xs = dt[b, c0:c1, h, None] * x[b, c0:c1, h]          # dt_s x_s
                tt, ss = np.meshgrid(np.arange(c1 - c0), np.arange(c1 - c0), indexing="ij")
                with np.errstate(over="ignore", invalid="ignore"):
                    Lf = np.where(ss <= tt, np.exp(cum[:, None] - cum[None, :]), 0.0)
                Y = (G * Lf) @ xs
                Sf = (np.exp(tot - cum)[:, None] * xs).T @ B[b, c0:c1]   # (P, N)
                piece = dict(c0=c0, c1=c1, cum=cum, excl=excl, tot=tot, Y=Y, Sf=Sf)
                if bidirectional:
                    with np.errstate(over="ignore", invalid="ignore"):
                        Lr = np.where(ss >= tt, np.exp(excl[None, :] - excl[:, None]), 0.0)
                    piece["Y"] = Y + (G * Lr) @ xs
                    piece["Sr"] = (np.exp(excl)[:, None] * xs).T @ B[b, c0:c1]
                pieces.append(piece)
            S_in = np.zeros((P, N))
            for pc in pieces:  # forward state passing + inter-chunk output
                Cc = C[b, pc["c0"]:pc["c1"]]
                pc["Y"] = pc["Y"] + np.exp(pc["cum"])[:, None] * (Cc @ S_in.T)
                S_in = np.exp(pc["tot"]) * S_in + pc["Sf"]
            if bidirectional:
                R_in = np.zeros((P, N))
                for pc in reversed(pieces):
                    Cc = C[b, pc["c0"]:pc["c1"]]
                    pc["Y"] = pc["Y"] + np.exp(pc["tot"] - pc["excl"])[:, None] * (Cc @ R_in.T)
                    R_in = np.exp(pc["tot"]) * R_in + pc["Sr"]
            for pc in pieces:
                y[b, pc["c0"]:pc["c1"], h] = pc["Y"]
    if D is not None:
        y = y + D[None, None, :, None] * x
    return y


# ---------------------------------------------------------------------------
# Chunked form of the SSD gradients
# ---------------------------------------------------------------------------

def _ssd_bwd_chunked_one_direction(x, dt, A_head, B, C, dy, chunk):
    """Gradients of the forward-direction chunked scan (no D term).

    B, C: (Bs, L, G, N).  Per (b, h) the forward chunk recursion is run to get
    the state S_in entering each chunk; then, from the last chunk to the first,
    with dS the gradient of the state leaving the chunk (0 after the last):

      du_s   = sum_{t>=s} G[t,s] e^{cum_t-cum_s} dY_t + e^{tot-cum_s} dS B_s
      dG     = Lf o (dY u^T)  ->  dC += dG B,  dB += dG^T C
      dC_t  += e^{cum_t} dY_t S_in,      dB_s += e^{tot-cum_s} dS^T u_s
      dcum_t = sum_s W[t,s] - sum_s W[s,t] + e^{cum_t} dY_t . (S_in C_t)
               - e^{tot-cum_t} u_t . (dS B_t),     W = G o dG
      dtot   = <dS, S_out>
      d(dt_r A_h) = sum_{i>=r} dcum_i + dtot
      dS_in  = e^{tot} dS + sum_t e^{cum_t} dY_t (x) C_t

    with u_s = dt_s x_s, so dx_s = dt_s du_s, ddt_s = x_s . du_s + A_h d(dA_s)
    and dA_h = sum_r dt_r d(dA_r).
    """
    Bs, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    out = dict(dx=np.zeros_like(x), ddt=np.zeros_like(dt), dA=np.zeros(H),
               dB=np.zeros_like(B), dC=np.zeros_like(C))
    bounds = [(c0, min(L, c0 + chunk)) for c0 in range(0, L, chunk)]
    for b in range(Bs):
        for h in range(H):
            g = h // hpg
            Ah = A_head[h]
            pieces = []
            S = np.zeros((P, N))
            for (c0, c1) in bounds:          # forward: the state entering each chunk
                dA = dt[b, c0:c1, h] * Ah
                cum = np.cumsum(dA)
                tot = cum[-1]
                u = dt[b, c0:c1, h, None] * x[b, c0:c1, h]
                S_out = np.exp(tot) * S + (np.exp(tot - cum)[:, None] * u).T @ B[b, c0:c1, g]
                pieces.append((c0, c1, cum, tot, u, S, S_out))
                S = S_out
            dS = np.zeros((P, N))
            for (c0, c1, cum, tot, u, S_in, S_out) in reversed(pieces):
                Bc, Cc, dY = B[b, c0:c1, g], C[b, c0:c1, g], dy[b, c0:c1, h]
                Gm = Cc @ Bc.T
                q = c1 - c0
                tt, ss = np.meshgrid(np.arange(q), np.arange(q), indexing="ij")
                with np.errstate(over="ignore", invalid="ignore"):
                    Lf = np.where(ss <= tt, np.exp(cum[:, None] - cum[None, :]), 0.0)
                dSB = Bc @ dS.T                                   # (Q, P): dS B_s
                du = (Gm * Lf).T @ dY + np.exp(tot - cum)[:, None] * dSB
                dG = Lf * (dY @ u.T)
                out["dC"][b, c0:c1, g] += dG @ Bc + np.exp(cum)[:, None] * (dY @ S_in)
                out["dB"][b, c0:c1, g] += dG.T @ Cc + np.exp(tot - cum)[:, None] * (u @ dS)
                W = Gm * dG
                dcum = (W.sum(axis=1) - W.sum(axis=0)
                        + np.exp(cum) * np.sum(dY * (Cc @ S_in.T), axis=1)
                        - np.exp(tot - cum) * np.sum(u * dSB, axis=1))
                dtot = float(np.sum(dS * S_out))
                d_dA = np.cumsum(dcum[::-1])[::-1] + dtot
                out["dx"][b, c0:c1, h] += dt[b, c0:c1, h, None] * du
                out["ddt"][b, c0:c1, h] += np.sum(x[b, c0:c1, h] * du, axis=1) + Ah * d_dA
                out["dA"][h] += float(np.sum(dt[b, c0:c1, h] * d_dA))
                dS = np.exp(tot) * dS + (np.exp(cum)[:, None] * dY).T @ Cc
    return out


def ssd_scan_bwd_chunked(x, dt, A_head, B, C, D, dy, chunk: int = 64, bidirectional: bool = False):
    """Gradients (dx, ddt, dA, dB, dC, dD) of sum(dy * y) for the SSD scan,
    chunk by chunk: the transposed products of the chunked pipeline and the
    state gradient passed from the last chunk to the first.

    B, C: (Bs, L, N) or (Bs, L, G, N) (groups of heads sharing B, C; dB, dC
    are summed over a group's heads).  The reversed direction of the
    bidirectional scan is the forward direction's gradient on time-reversed
    inputs and upstream gradient, reversed back; D x enters once.
    """
    x, dt, A_head, B, C, D, dy = map(_f64, (x, dt, A_head, B, C, D, dy))
    grouped = B.ndim == 4
    if not grouped:
        B, C = B[:, :, None, :], C[:, :, None, :]
    out = _ssd_bwd_chunked_one_direction(x, dt, A_head, B, C, dy, chunk)
    if bidirectional:
        rev = lambda a: a[:, ::-1]
        r = _ssd_bwd_chunked_one_direction(rev(x), rev(dt), A_head, rev(B), rev(C), rev(dy), chunk)
        for k in ("dx", "ddt", "dB", "dC"):
            out[k] = out[k] + rev(r[k])
        out["dA"] = out["dA"] + r["dA"]
    out["dD"] = None
    if D is not None:
        out["dx"] = out["dx"] + D[None, None, :, None] * dy
        out["dD"] = np.sum(dy * x, axis=(0, 1, 3))
    if not grouped:
        out["dB"], out["dC"] = out["dB"][:, :, 0], out["dC"][:, :, 0]
    return out
