"""fp64 CPU oracle for the selective-scan backward.

TEST INFRASTRUCTURE ONLY: the tests and the bench's CPU-baseline leg use it;
the product path never does. It shares no code with the CUDA library.

The page "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南"
(section 4.1) routes the backward of ``selective_scan_fn`` to a CUDA ``bwd``
kernel that returns the gradient of every input; it prints neither formula nor
code. The gradients are therefore the plain definition: the derivatives of
L = sum(dout * out) with respect to u, delta, A, B, C, D, z, delta_bias (and
the start state), for the forward

    dt_t  = softplus(v_t), v_t = delta_t + delta_bias   (dt_t = v_t without softplus)
    a_t   = exp(dt_t A_n),  h_t = a_t h_{t-1} + dt_t B_t u_t   (h_{-1} = start state or 0)
    y_t   = sum_n C_t h_t + D u_t,   out_t = y_t silu(z_t)

taken by reverse-mode differentiation (the chain rule in reverse step order):

    dy_t      = dout_t silu(z_t)                  dz_t = dout_t y_t silu'(z_t)
    lam_t     = dy_t C_t + a_{t+1} lam_{t+1}      (lam = dL/dh_t; lam_l = 0)
    dC_t     += dy_t h_t                          dB_t += lam_t dt_t u_t
    du_t      = dy_t D + sum_n lam_t dt_t B_t     dD   += dy_t u_t
    ddt_t     = sum_n lam_t (A a_t h_{t-1} + B_t u_t)
    dA       += lam_t a_t h_{t-1} dt_t            dstart = a_0 lam_0
    ddelta_t  = ddt_t sigmoid(v_t)  (ddt_t without softplus)
    ddelta_bias = sum_{b, t} ddelta_t

with the sums over batch and step for the per-channel weights (A, D,
delta_bias, fixed B/C) and over the channels of a group for variable B/C.
silu'(z) = s (1 + z (1 - s)), s = sigmoid(z). Everything is fp64 numpy,
vectorised over (batch, channel, state) with an explicit loop over steps.

Pins (``tests/test_oracle_bwd.py``): central finite differences of the
independent C forward oracle, torch.autograd through a plain torch forward,
and planted slips in the helpers below.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _sigmoid(v):
    """1 / (1 + e^-v), evaluated without overflow for either sign."""
    e = np.exp(-np.abs(v))
    return np.where(v >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _softplus(v):
    return np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v)))


def _dsilu(z):
    """d silu(z) / dz = s (1 + z (1 - s)), s = sigmoid(z)."""
    s = _sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def _dsoftplus(v):
    """d softplus(v) / dv = sigmoid(v)."""
    return _sigmoid(v)


# The adjoint at step t decays by the factor of step t + _DECAY_OFFSET: the
# factor that carried h_t into h_{t+1}.
_DECAY_OFFSET = 1


def _adjoint(a, g):
    """lam_t = g_t + a_{t+1} lam_{t+1} for t = l-1 .. 0, with lam_{l-1} = g_{l-1}."""
    l_ = g.shape[-1]
    lam = np.empty_like(g)
    nxt = np.zeros(g.shape[:-1])
    for t in range(l_ - 1, -1, -1):
        k = t + _DECAY_OFFSET
        nxt = g[..., t] + (a[..., k] * nxt if k < l_ else 0.0)
        lam[..., t] = nxt
    return lam


def _group_sum(x, ngroups):
    """(b, d, n, l) per-channel terms -> (b, g, n, l): sum over each group's
    dim / ngroups consecutive channels."""
    b, d, n, l = x.shape
    return x.reshape(b, ngroups, d // ngroups, n, l).sum(axis=2)


def selective_scan_bwd_ref(dout, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                           delta_softplus=False, initial_state=None):
    """Gradients of sum(dout * out) for the selective-scan forward.

    Shapes as for the forward: u, delta, z, dout (b, d, l); A (d, n); B, C
    fixed (d, n), 3-D (b, n, l) or 4-D (b, g, n, l); D, delta_bias (d,);
    initial_state (b, d, n). Returns a dict of fp64 arrays with keys du,
    ddelta, dA, dB, dC (each in its input's shape), and dD, dz, ddelta_bias,
    dinitial_state when the matching input was given (else None)."""
    dout, u, delta, A, B, C = (_f64(t) for t in (dout, u, delta, A, B, C))
    D, z, bias, x0 = _f64(D), _f64(z), _f64(delta_bias), _f64(initial_state)
    b_, d_, l_ = u.shape
    n_ = A.shape[1]
    fixed = B.ndim == 2
    three_d = B.ndim == 3
    if fixed:
        Bt = np.broadcast_to(B[None, :, :, None], (b_, d_, n_, l_))
        Ct = np.broadcast_to(C[None, :, :, None], (b_, d_, n_, l_))
        ng = 1
    else:
        B4, C4 = (B[:, None], C[:, None]) if three_d else (B, C)
        ng = B4.shape[1]
        grp = np.arange(d_) // (d_ // ng)
        Bt, Ct = B4[:, grp], C4[:, grp]                     # (b, d, n, l)

    if l_ == 0:  # nothing depends on the weights; the start state passes through unchanged
        zero = lambda t: None if t is None else np.zeros_like(t)
        return dict(du=zero(u), ddelta=zero(delta), dA=zero(A), dB=zero(B), dC=zero(C), dD=zero(D),
                    dz=zero(z), ddelta_bias=zero(bias), dinitial_state=zero(x0))

    # forward, keeping every state
    v = delta + (bias[None, :, None] if bias is not None else 0.0)
    dt = _softplus(v) if delta_softplus else v
    a = np.exp(dt[:, :, None, :] * A[None, :, :, None])      # (b, d, n, l)
    bu = (dt * u)[:, :, None, :] * Bt
    h = np.empty((b_, d_, n_, l_))
    x = np.zeros((b_, d_, n_)) if x0 is None else x0.copy()
    for t in range(l_):
        x = a[..., t] * x + bu[..., t]
        h[..., t] = x
    y = np.sum(Ct * h, axis=2)
    if D is not None:
        y = y + D[None, :, None] * u

    # output gate
    if z is not None:
        dy = dout * z * _sigmoid(z)
        dz = dout * y * _dsilu(z)
    else:
        dy, dz = dout, None

    # state adjoint, in reverse step order
    lam = _adjoint(a, dy[:, :, None, :] * Ct)

    h_prev = np.concatenate([(np.zeros((b_, d_, n_)) if x0 is None else x0)[..., None], h[..., :-1]], axis=3)
    a_hprev = a * h_prev
    ddt = np.sum(lam * (A[None, :, :, None] * a_hprev + Bt * u[:, :, None, :]), axis=2)
    du = np.sum(lam * dt[:, :, None, :] * Bt, axis=2)
    if D is not None:
        du = du + dy * D[None, :, None]
    dA = np.sum(lam * a_hprev * dt[:, :, None, :], axis=(0, 3))
    dB_full = lam * (dt * u)[:, :, None, :]
    dC_full = dy[:, :, None, :] * h
    if fixed:
        dB, dC = dB_full.sum(axis=(0, 3)), dC_full.sum(axis=(0, 3))
    else:
        dB, dC = _group_sum(dB_full, ng), _group_sum(dC_full, ng)
        if three_d:
            dB, dC = dB[:, 0], dC[:, 0]
    dv = ddt * _dsoftplus(v) if delta_softplus else ddt
    return dict(du=du, ddelta=dv, dA=dA, dB=dB, dC=dC,
                dD=None if D is None else np.sum(dy * u, axis=(0, 2)),
                dz=dz,
                ddelta_bias=None if bias is None else np.sum(dv, axis=(0, 2)),
                dinitial_state=None if x0 is None else a[..., 0] * lam[..., 0])


def selective_scan_bwd_rows(rows, dout, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                            delta_softplus=False, initial_state=None):
    """Per-row parts of the backward for selected (b, d) rows, each solved as a
    one-row problem (rows do not interact except through the sums over rows).
    Returns a list of dicts: du, ddelta, dz (l,), and the row's own
    contributions to dA (n,), dD, ddelta_bias (scalars), dB, dC ((n, l), or
    (n,) for fixed B/C) and dinitial_state (n,)."""
    dout, u, delta, A, B, C = (_f64(t) for t in (dout, u, delta, A, B, C))
    D, z, bias, x0 = _f64(D), _f64(z), _f64(delta_bias), _f64(initial_state)
    dim = u.shape[1]
    fixed = B.ndim == 2
    ng = 1 if B.ndim <= 3 else B.shape[1]
    res = []
    for b, d in rows:
        if fixed:
            Bi, Ci = B[d:d + 1], C[d:d + 1]
        elif B.ndim == 3:
            Bi, Ci = B[b:b + 1], C[b:b + 1]
        else:
            gi = d // (dim // ng)
            Bi, Ci = B[b:b + 1, gi:gi + 1], C[b:b + 1, gi:gi + 1]
        sl = lambda t: None if t is None else t[b:b + 1, d:d + 1]
        r = selective_scan_bwd_ref(sl(dout), sl(u), sl(delta), A[d:d + 1], Bi, Ci,
                                   None if D is None else D[d:d + 1], sl(z),
                                   None if bias is None else bias[d:d + 1], delta_softplus, sl(x0))
        one = dict(du=r["du"][0, 0], ddelta=r["ddelta"][0, 0], dA=r["dA"][0],
                   dz=None if r["dz"] is None else r["dz"][0, 0],
                   dD=None if r["dD"] is None else r["dD"][0],
                   ddelta_bias=None if r["ddelta_bias"] is None else r["ddelta_bias"][0],
                   dinitial_state=None if r["dinitial_state"] is None else r["dinitial_state"][0, 0])
        if fixed:
            one["dB"], one["dC"] = r["dB"][0], r["dC"][0]
        elif B.ndim == 3:
            one["dB"], one["dC"] = r["dB"][0], r["dC"][0]
        else:
            one["dB"], one["dC"] = r["dB"][0, 0], r["dC"][0, 0]
        res.append(one)
    return res
