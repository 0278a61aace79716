"""Pins for the complex-A oracle (``oracle/complex_a.py``; page "PaddleNLP
Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南", section 4.1: A
"real or complex"), each against something other than the oracle itself:
the C oracle for real A, a brute-force cmath unrolling, a closed-form
geometric sum, and the 2x2 real rotation form of a complex state.
"""
import cmath
import math

import numpy as np
import pytest

import oracle
from oracle import complex_a


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _problem(seed, b, d, l, n, g=1, fixed=False, im_scale=3.0):
    rng = np.random.default_rng(seed)
    A = -rng.uniform(0.2, 2.0, (d, n)) + 1j * rng.uniform(-im_scale, im_scale, (d, n))
    p = dict(u=rng.standard_normal((b, d, l)), delta=rng.standard_normal((b, d, l)) * 0.7, A=A,
             D=rng.standard_normal(d), z=rng.standard_normal((b, d, l)), delta_bias=rng.uniform(-2, 0.5, d))
    if fixed:
        p["B"], p["C"] = rng.standard_normal((d, n)), rng.standard_normal((d, n))
    else:
        p["B"], p["C"] = rng.standard_normal((b, g, n, l)), rng.standard_normal((b, g, n, l))
    return p


@pytest.mark.parametrize("fixed", [False, True])
def test_real_A_equals_the_c_oracle(fixed):
    p = _problem(1, 2, 4, 30, 3, g=2, fixed=fixed)
    p["A"] = p["A"].real + 0j
    x0 = np.random.default_rng(2).standard_normal((2, 4, 3))
    out, last = complex_a.selective_scan_complex_ref(**p, delta_softplus=True, return_last_state=True,
                                                     initial_state=x0 + 0j)
    pr = dict(p, A=p["A"].real)
    ref, ref_last = oracle.selective_scan_ref(**pr, delta_softplus=True, return_last_state=True, initial_state=x0)
    assert _rel(out, ref) < 1e-13
    assert _rel(last.real, ref_last) < 1e-13 and not np.any(last.imag)


def _brute(p, x0):
    """x_t = prod_{j<=t} a_j x0 + sum_k prod_{j=k+1..t} a_j dt_k B_k u_k with
    complex a_j = e^{dt_j A}, cmath; the real and imaginary parts summed with
    math.fsum."""
    u, delta, A, B, C, D, z, bias = (p[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias"))
    b_, d_, l_ = u.shape
    n_ = A.shape[1]
    g_ = B.shape[1]
    out = np.zeros((b_, d_, l_))
    for b in range(b_):
        for d in range(d_):
            gi = d // (d_ // g_)
            dt = [math.log1p(math.exp(float(delta[b, d, t] + bias[d]))) for t in range(l_)]
            for t in range(l_):
                ys = []
                for n in range(n_):
                    terms = [cmath.exp(A[d, n] * math.fsum(dt[:t + 1])) * x0[b, d, n]]
                    for k in range(t + 1):
                        terms.append(cmath.exp(A[d, n] * math.fsum(dt[k + 1:t + 1])) * dt[k] * B[b, gi, n, k] * u[b, d, k])
                    x = complex(math.fsum(c.real for c in terms), math.fsum(c.imag for c in terms))
                    ys.append(C[b, gi, n, t] * x.real)
                y = math.fsum(ys) + D[d] * u[b, d, t]
                out[b, d, t] = y * z[b, d, t] / (1.0 + math.exp(-z[b, d, t]))
    return out


def test_brute_force():
    p = _problem(3, 1, 2, 7, 3, g=1)
    x0 = np.random.default_rng(4).standard_normal((1, 2, 3)) + 1j * np.random.default_rng(5).standard_normal((1, 2, 3))
    out = complex_a.selective_scan_complex_ref(**p, delta_softplus=True, initial_state=x0)
    assert _rel(out, _brute(p, x0)) < 1e-12


def test_geometric_closed_form():
    """Constant dt, u, B and a start x0: x_t = a^{t+1} x0 + dt B u (1 - a^{t+1}) / (1 - a)."""
    d, l, n = 1, 25, 2
    A = np.array([[-0.3 + 2.0j, -1.0 - 0.5j]])
    Bf, Cf = np.array([[0.7, -1.2]]), np.array([[1.0, 0.4]])
    x0 = np.array([[[0.5 - 0.25j, -1.0 + 2.0j]]])
    dt, uval = 0.37, -1.3
    u = np.full((1, d, l), uval)
    out, last = complex_a.selective_scan_complex_ref(u, np.full((1, d, l), dt), A, Bf, Cf, return_last_state=True,
                                                     initial_state=x0)
    t = np.arange(l)
    a = np.exp(dt * A[0])[:, None]
    pw = a ** (t[None, :] + 1)
    x = pw * x0[0, 0][:, None] + dt * Bf[0][:, None] * uval * (1 - pw) / (1 - a)
    assert _rel(out[0, 0], (Cf[0][:, None] * x).sum(0).real) < 1e-13
    assert _rel(last[0, 0], x[:, -1]) < 1e-13


def test_rotation_form():
    """One complex state A = alpha + i omega is the real 2x2 system
    [xr, xi] <- e^{alpha dt} R(omega dt) [xr, xi] + [dt B u, 0]. The output is
    the same for conj(A) (real B, C, u: the rotation's sense does not reach
    Re x), while dropping the rotation's cross term changes it."""
    rng = np.random.default_rng(6)
    l = 40
    alpha, omega = -0.4, 2.5
    A = np.array([[alpha + 1j * omega]])
    u, delta = rng.standard_normal((1, 1, l)), rng.standard_normal((1, 1, l)) * 0.5
    Bv, Cv = rng.standard_normal((1, 1, 1, l)), rng.standard_normal((1, 1, 1, l))
    out = complex_a.selective_scan_complex_ref(u, delta, A, Bv, Cv, delta_softplus=True)

    def rot(sign):
        xr = xi = 0.0
        ys = []
        for t in range(l):
            dt = math.log1p(math.exp(delta[0, 0, t]))
            e, c, s = math.exp(alpha * dt), math.cos(omega * dt), sign * math.sin(omega * dt)
            xr, xi = e * (c * xr - s * xi) + dt * Bv[0, 0, 0, t] * u[0, 0, t], e * (s * xr + c * xi)
            ys.append(Cv[0, 0, 0, t] * xr)
        return np.array(ys)

    assert _rel(out[0, 0], rot(+1)) < 1e-13
    assert _rel(out[0, 0], rot(-1)) < 1e-13
    conj = complex_a.selective_scan_complex_ref(u, delta, np.conj(A), Bv, Cv, delta_softplus=True)
    assert _rel(conj, out) < 1e-13
    assert _rel(rot(0), out[0, 0]) > 1e-3
