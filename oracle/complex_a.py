"""fp64 CPU oracle for the complex-A variant of the selective-scan forward.

TEST INFRASTRUCTURE ONLY: the tests and the bench's CPU-baseline leg use it;
the product path never does. It shares no code with the CUDA library.

The page "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南"
(section 4.1) says that A, of shape (dim, dstate), may be real or complex, and
gives B and C only the real shapes (fixed (dim, dstate), or varying
(batch, [groups,] dstate, seqlen)). The plain reading taken here: A complex,
everything else as for real A (u, delta, z, B, C, D, delta_bias real), the
state complex, and the real output the real part of the contraction:

    dt   = softplus(delta_t + delta_bias)           (or the sum itself)
    x_n  = exp(dt A_n) x_n + dt B_{n,t} u_t          (complex x, complex exp)
    y    = Re(sum_n C_{n,t} x_n) + D u_t
    out  = y silu(z_t)                               (when z is given)

with x = initial_state before step 0 (complex; zero when absent) and
last_state = x after the last step (complex). Everything is complex128 /
float64 numpy, vectorised over (batch, channel, state) with an explicit loop
over steps.

Pins (``tests/test_oracle_complex.py``): with Im(A) = 0 it equals the
independently written C oracle for real A; a brute-force unrolling with cmath
and math.fsum on tiny problems; the closed-form geometric sum for constant
inputs; the 2x2 real rotation form of one complex state.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu()
        if x.is_complex():
            return np.ascontiguousarray(x.to(torch.complex128).numpy())
        return np.ascontiguousarray(x.to(torch.float64).numpy())
    a = np.asarray(x)
    return np.ascontiguousarray(a.astype(np.complex128 if np.iscomplexobj(a) else np.float64))


def selective_scan_complex_ref(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                               return_last_state=False, initial_state=None):
    """Returns out (b, d, l) float64, and last_state (b, d, n) complex128 when
    return_last_state."""
    u, delta, B, C = (_f64(t) for t in (u, delta, B, C))
    A = _f64(A).astype(np.complex128)
    D, z, bias = _f64(D), _f64(z), _f64(delta_bias)
    x0 = _f64(initial_state)
    b_, d_, l_ = u.shape
    n_ = A.shape[1]
    if B.ndim == 2:                                   # fixed (d, n)
        Bt = np.broadcast_to(B[None, :, :, None], (b_, d_, n_, l_))
        Ct = np.broadcast_to(C[None, :, :, None], (b_, d_, n_, l_))
    else:
        B4, C4 = (B[:, None], C[:, None]) if B.ndim == 3 else (B, C)
        grp = np.arange(d_) // (d_ // B4.shape[1])
        Bt, Ct = B4[:, grp], C4[:, grp]
    v = delta + (bias[None, :, None] if bias is not None else 0.0)
    dt = np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v))) if delta_softplus else v
    x = np.zeros((b_, d_, n_), np.complex128) if x0 is None else x0.astype(np.complex128).copy()
    out = np.empty((b_, d_, l_))
    for t in range(l_):
        a = np.exp(dt[:, :, t, None] * A[None])
        x = a * x + (dt[:, :, t] * u[:, :, t])[:, :, None] * Bt[..., t]
        y = np.sum(Ct[..., t] * x, axis=2).real
        if D is not None:
            y = y + D[None, :] * u[:, :, t]
        out[:, :, t] = y
    if z is not None:
        out = out * (z / (1.0 + np.exp(-z)))
    return (out, x) if return_last_state else out
