"""The algebra of the chunked SSD backward on the GPU, pinned on the CPU.

The CUDA path (ssd_bwd_chunk.cu) forms the SSD scan's gradients chunk by
chunk: states entering each chunk and adjoints leaving it by two recursions
over the chunks, products inside each chunk, and -- for dA and the dt A part
of ddt -- a suffix sum of one per-step scalar, from the identity

    dL/d(dA_r) = a_r <G_r, H_{r-1}> = <G_r, H_r> - dt_r x_r . (G_r B_r)
               = sum_{u >= r} (dy_u . yt_u - dt_u x_u . (G_u B_u)),

yt the scan output without D, G the state adjoint.  This test restates those
formulas in numpy (fp64, written from the definitions above, not from the
kernel) and requires them to equal the oracle's sequential reverse mode
(itself pinned by finite differences) to 1e-10, in both directions, with a
ragged last chunk and groups of B, C.
"""
import numpy as np
import pytest

import oracle
import workloads


def _chunked_grads(x, dt, A, B, C, D, dy, heads_per_group, Q, bidir):
    Bs, L, H, P = x.shape
    N = B.shape[-1]
    out = {k: np.zeros(s) for k, s in (("dx", x.shape), ("ddt", dt.shape), ("dA", (H,)),
                                        ("dB", B.shape), ("dC", C.shape), ("dD", (H,)))}
    nc = (L + Q - 1) // Q
    for d in range(2 if bidir else 1):
        order = np.arange(L)[::-1] if d else np.arange(L)    # walk step -> time index
        for b in range(Bs):
            for h in range(H):
                g = h // heads_per_group
                X = np.zeros((nc * Q, P)); Y = np.zeros((nc * Q, P))
                Bm = np.zeros((nc * Q, N)); Cm = np.zeros((nc * Q, N)); dv = np.zeros(nc * Q)
                X[:L] = x[b, order, h]; Y[:L] = dy[b, order, h]
                Bm[:L] = B[b, order, g]; Cm[:L] = C[b, order, g]; dv[:L] = dt[b, order, h]
                cum = [np.cumsum(dv[k * Q:(k + 1) * Q] * A[h]) for k in range(nc)]
                rows = [slice(k * Q, (k + 1) * Q) for k in range(nc)]
                # states entering each chunk, adjoints leaving it
                S = [np.zeros((P, N)) for _ in range(nc)]
                for k in range(nc - 1):
                    w = dv[rows[k]] * np.exp(cum[k][-1] - cum[k])
                    S[k + 1] = np.exp(cum[k][-1]) * S[k] + (X[rows[k]] * w[:, None]).T @ Bm[rows[k]]
                Gin = [np.zeros((P, N)) for _ in range(nc)]
                for k in range(nc - 2, -1, -1):
                    e = np.exp(cum[k + 1])
                    Gin[k] = np.exp(cum[k + 1][-1]) * Gin[k + 1] + (Y[rows[k + 1]] * e[:, None]).T @ Cm[rows[k + 1]]
                q = np.zeros(nc * Q)
                for k in range(nc):
                    r, c = rows[k], cum[k]
                    Lm = np.tril(np.exp(c[:, None] - c[None, :]))
                    GL = (Cm[r] @ Bm[r].T) * Lm
                    WL = (Y[r] @ X[r].T) * Lm
                    eo, ec, dtk = np.exp(c[-1] - c), np.exp(c), dv[r]
                    v = GL.T @ Y[r] + eo[:, None] * (Bm[r] @ Gin[k].T)
                    d1 = (X[r] * v).sum(1)
                    dxk = dtk[:, None] * v + (D[h] if d == 0 else 0.0) * Y[r]
                    dBk = dtk[:, None] * (WL.T @ Cm[r] + eo[:, None] * (X[r] @ Gin[k]))
                    dCk = (WL * dtk[None, :]) @ Bm[r] + ec[:, None] * (Y[r] @ S[k])
                    yt = (GL * dtk[None, :]) @ X[r] + ec[:, None] * (Cm[r] @ S[k].T)
                    q[r] = (Y[r] * yt).sum(1) - dtk * d1
                    for i in range(Q):
                        lam = k * Q + i
                        if lam >= L:
                            continue
                        t = order[lam]
                        out["dx"][b, t, h] += dxk[i]
                        out["dB"][b, t, g] += dBk[i]
                        out["dC"][b, t, g] += dCk[i]
                        out["ddt"][b, t, h] += d1[i]
                    if d == 0:
                        out["dD"][h] += (Y[r] * X[r]).sum()
                suffix = np.cumsum(q[:L][::-1])[::-1]      # dL/d(dA_r), walk order
                out["ddt"][b, order, h] += A[h] * suffix
                out["dA"][h] += (dv[:L] * suffix).sum()
    return out


@pytest.mark.parametrize("bidir", [False, True])
@pytest.mark.parametrize("groups", [1, 2])
def test_chunked_algebra_equals_sequential_gradients(bidir, groups):
    Bs, L, H, P, N, Q = 1, 45, 2, 8, 6, 16           # a ragged last chunk (45 = 2 x 16 + 13)
    inp = workloads.ssd_inputs(Bs, L, H, P, N, "f32", seed=11 + groups, groups=groups)
    dy = workloads.grad_output((Bs, L, H, P), seed=5)
    ref = oracle.ssd_scan_bwd(**inp, dy=dy, bidirectional=bidir)
    n = {k: (v.double().numpy() if v is not None else None) for k, v in inp.items()}
    got = _chunked_grads(n["x"], n["dt"], n["A_head"], n["B"], n["C"], n["D"],
                         dy.double().numpy(), H // groups, Q, bidir)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        r = np.asarray(ref[k], dtype=np.float64).reshape(got[k].shape)
        assert np.max(np.abs(got[k] - r)) <= 1e-10 * max(1.0, np.max(np.abs(r))), k
