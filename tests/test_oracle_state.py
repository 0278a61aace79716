"""Pins for the oracle's initial-state input and for the one-step state-update
oracle (the decode step the page "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能
NLP GPU 算子实战指南" lists in section 4.4 as "selective_state_update"; it prints
no signature, so the operands are those of the section 4.1 scan at one step).

Each pin checks against something other than the function itself: a brute-force
unrolling with the initial-state term, a closed-form geometric sum, the
independently written C sequence oracle (for the numpy step function) and the
composition law of the recurrence (a run split in two with the state handed
over equals the whole run).
"""
import math

import numpy as np
import pytest

import oracle

RTOL = 1e-12


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _problem(rng, b, d, l, n, g=1, fixed=False):
    p = dict(u=rng.standard_normal((b, d, l)),
             delta=rng.standard_normal((b, d, l)) * 0.7,
             A=-rng.uniform(0.2, 3.0, (d, n)),
             D=rng.standard_normal(d),
             z=rng.standard_normal((b, d, l)),
             delta_bias=rng.uniform(-3, 0.5, d))
    if fixed:
        p["B"], p["C"] = rng.standard_normal((d, n)), rng.standard_normal((d, n))
    else:
        p["B"], p["C"] = rng.standard_normal((b, g, n, l)), rng.standard_normal((b, g, n, l))
    return p


def _brute_with_init(p, x0):
    """x_{n,t} = exp(A_n sum_{j<=t} dt_j) x0_n
               + sum_{k<=t} exp(A_n sum_{j=k+1..t} dt_j) dt_k B_{n,k} u_k,
    with softplus written as log(1 + e^v), summed with math.fsum."""
    u, delta, A, B, C, D, z, bias = (p[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias"))
    b_, d_, l_ = u.shape
    n_ = A.shape[1]
    fixed = B.ndim == 2
    g_ = 1 if fixed else B.shape[1]
    out = np.zeros((b_, d_, l_))
    last = np.zeros((b_, d_, n_))
    for b in range(b_):
        for d in range(d_):
            gi = 0 if fixed else d // (d_ // g_)
            dt = [math.log(1.0 + math.exp(float(delta[b, d, t]) + float(bias[d]))) for t in range(l_)]
            for t in range(l_):
                ys = []
                for n in range(n_):
                    terms = [math.exp(A[d, n] * math.fsum(dt[0:t + 1])) * x0[b, d, n]]
                    for k in range(t + 1):
                        Bk = B[d, n] if fixed else B[b, gi, n, k]
                        terms.append(math.exp(A[d, n] * math.fsum(dt[k + 1:t + 1])) * dt[k] * Bk * u[b, d, k])
                    x = math.fsum(terms)
                    ys.append((C[d, n] if fixed else C[b, gi, n, t]) * x)
                    if t == l_ - 1:
                        last[b, d, n] = x
                y = math.fsum(ys) + D[d] * u[b, d, t]
                out[b, d, t] = y * z[b, d, t] / (1.0 + math.exp(-z[b, d, t]))
    return out, last


@pytest.mark.parametrize("case", [dict(b=1, d=2, l=8, n=3), dict(b=2, d=4, l=6, n=2, g=2),
                                  dict(b=1, d=3, l=7, n=3, fixed=True)])
def test_initial_state_brute_force(case):
    rng = np.random.default_rng(3 + case["l"])
    p = _problem(rng, **case)
    x0 = rng.standard_normal((case["b"], case["d"], case["n"]))
    out, last = oracle.selective_scan_ref(**p, delta_softplus=True, return_last_state=True, initial_state=x0)
    bout, blast = _brute_with_init(p, x0)
    assert _rel(out, bout) < RTOL
    assert _rel(last, blast) < RTOL


def test_initial_state_geometric_closed_form():
    """Constant dt, A, B, u and a start x0: x_t = a^{t+1} x0 + dt B u (1 - a^{t+1}) / (1 - a)."""
    d, l, n = 2, 30, 3
    A = -np.array([[0.5, 1.0, 2.0], [0.1, 0.7, 3.0]])
    Bf = np.array([[1.0, -0.5, 0.25], [0.3, 0.1, -1.0]])
    Cf = np.array([[0.7, 0.2, -0.4], [1.0, -1.0, 0.5]])
    x0 = np.array([[[2.0, -1.0, 0.5], [0.25, 3.0, -2.0]]])
    dt, uval = 0.29, np.array([0.8, -1.7])
    u = np.broadcast_to(uval[None, :, None], (1, d, l)).copy()
    out, last = oracle.selective_scan_ref(u, np.full((1, d, l), dt), A, Bf, Cf,
                                          return_last_state=True, initial_state=x0)
    t = np.arange(l)
    for di in range(d):
        a = np.exp(dt * A[di])[:, None]
        p = a ** (t[None, :] + 1)
        x = p * x0[0, di][:, None] + dt * Bf[di][:, None] * uval[di] * (1 - p) / (1 - a)
        assert _rel(out[0, di], (Cf[di][:, None] * x).sum(0)) < 1e-13
        assert _rel(last[0, di], x[:, -1]) < 1e-13


@pytest.mark.parametrize("fixed", [False, True])
def test_split_run_composes(fixed):
    """A run over l1 + l2 steps equals a run over l1 steps followed by a run over
    the last l2 steps started from the first run's last_state."""
    rng = np.random.default_rng(17)
    b, d, l1, l2, n, g = 2, 6, 23, 17, 4, 3
    p = _problem(rng, b, d, l1 + l2, n, g=g, fixed=fixed)
    full, last = oracle.selective_scan_ref(**p, delta_softplus=True, return_last_state=True)

    def part(sl):
        q = dict(p)
        for k in ("u", "delta", "z"):
            q[k] = np.ascontiguousarray(p[k][:, :, sl])
        if not fixed:
            for k in ("B", "C"):
                q[k] = np.ascontiguousarray(p[k][..., sl])
        return q

    o1, s1 = oracle.selective_scan_ref(**part(slice(0, l1)), delta_softplus=True, return_last_state=True)
    o2, s2 = oracle.selective_scan_ref(**part(slice(l1, None)), delta_softplus=True, return_last_state=True,
                                       initial_state=s1)
    assert _rel(o1, full[:, :, :l1]) < 1e-14
    assert _rel(o2, full[:, :, l1:]) < RTOL
    assert _rel(s2, last) < RTOL


def _step_inputs(rng, b, d, n, g, fixed):
    st = rng.standard_normal((b, d, n))
    u, delta, z = rng.standard_normal((b, d)), rng.standard_normal((b, d)) * 0.7, rng.standard_normal((b, d))
    A, D, bias = -rng.uniform(0.2, 3.0, (d, n)), rng.standard_normal(d), rng.uniform(-3, 0.5, d)
    if fixed:
        B, C = rng.standard_normal((d, n)), rng.standard_normal((d, n))
    elif g == 0:
        B, C = rng.standard_normal((b, n)), rng.standard_normal((b, n))
    else:
        B, C = rng.standard_normal((b, g, n)), rng.standard_normal((b, g, n))
    return st, u, delta, A, B, C, D, z, bias


@pytest.mark.parametrize("form", ["per_token", "grouped", "fixed"])
@pytest.mark.parametrize("softplus", [True, False])
def test_state_update_equals_one_step_of_the_scan(form, softplus):
    """The numpy step function against the C sequence oracle run for one step
    from the same state (two independent implementations)."""
    rng = np.random.default_rng(23 + softplus)
    b, d, n = 3, 8, 5
    g = {"per_token": 0, "grouped": 4, "fixed": 1}[form]
    st, u, delta, A, B, C, D, z, bias = _step_inputs(rng, b, d, n, g, form == "fixed")
    out, new = oracle.selective_state_update_ref(st, u, delta, A, B, C, D=D, z=z, delta_bias=bias,
                                                 delta_softplus=softplus, bc_fixed=form == "fixed")
    if form == "fixed":
        Bs, Cs = B, C
    elif form == "per_token":
        Bs, Cs = B[:, :, None], C[:, :, None]          # (b, n, 1): 3-D, one group
    else:
        Bs, Cs = B[..., None], C[..., None]             # (b, g, n, 1)
    o, s = oracle.selective_scan_ref(u[..., None], delta[..., None], A, Bs, Cs, D=D, z=z[..., None],
                                     delta_bias=bias, delta_softplus=softplus, return_last_state=True,
                                     initial_state=st)
    assert _rel(out, o[..., 0]) < 1e-13
    assert _rel(new, s) < 1e-13


def test_state_updates_chain_to_the_scan():
    """k successive steps from a state reproduce the scan over k steps from it."""
    rng = np.random.default_rng(29)
    b, d, l, n, g = 2, 6, 9, 4, 2
    p = _problem(rng, b, d, l, n, g=g)
    x0 = rng.standard_normal((b, d, n))
    out, last = oracle.selective_scan_ref(**p, delta_softplus=True, return_last_state=True, initial_state=x0)
    st = x0
    for t in range(l):
        o, st = oracle.selective_state_update_ref(st, p["u"][:, :, t], p["delta"][:, :, t], p["A"],
                                                  p["B"][..., t], p["C"][..., t], D=p["D"], z=p["z"][:, :, t],
                                                  delta_bias=p["delta_bias"], delta_softplus=True)
        assert _rel(o, out[:, :, t]) < 1e-12, t
    assert _rel(st, last) < 1e-12


def test_planted_initial_state_mistakes_are_caught():
    """Plausible slips in the initial-state path (ignored start, start not
    decayed at the first step, start added after the step) fail the brute-force pin."""
    rng = np.random.default_rng(41)
    p = _problem(rng, 1, 2, 6, 3)
    x0 = rng.standard_normal((1, 2, 3))
    bout, _ = _brute_with_init(p, x0)

    def scan(variant):
        u, delta, A, B, C, D, z, bias = (p[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias"))
        out = np.zeros_like(u)
        for d in range(2):
            x = np.zeros(3) if variant == "ignored" else x0[0, d].copy()
            for t in range(u.shape[2]):
                dt = np.log1p(np.exp(delta[0, d, t] + bias[d]))
                a = np.exp(dt * A[d])
                if variant == "undecayed" and t == 0:
                    x = x + dt * B[0, 0, :, t] * u[0, d, t]
                else:
                    x = a * x + dt * B[0, 0, :, t] * u[0, d, t]
                xs = x + x0[0, d] if (variant == "added_after" and t == 0) else x
                y = (C[0, 0, :, t] * xs).sum() + D[d] * u[0, d, t]
                out[0, d, t] = y * z[0, d, t] / (1 + np.exp(-z[0, d, t]))
        return out

    assert _rel(scan("none"), bout) < 1e-12
    for v in ("ignored", "undecayed", "added_after"):
        assert _rel(scan(v), bout) > 1e-3, v
