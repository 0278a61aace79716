"""Pins for the fp64 oracle, each checked against something other than the
oracle itself: brute-force unrolling, closed forms, a library routine
(numpy.convolve), invariants and special cases of the recurrence.

The operation (page "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU
算子实战指南", section 4.1, operands of selective_scan_fn) is
  dt = softplus(delta + delta_bias), x_t = exp(dt A) x_{t-1} + dt B_t u_t,
  y_t = sum_n C_t x_t + D u_t, out = y silu(z).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from state_space_model_03_gb300 import workloads

RTOL = 1e-12


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _rand_problem(rng, b, d, l, n, g=1, bc="variable", z=True, D=True, bias=True):
    u = rng.standard_normal((b, d, l))
    delta = rng.standard_normal((b, d, l)) * 0.7
    A = -rng.uniform(0.2, 3.0, (d, n))
    if bc == "fixed":
        B = rng.standard_normal((d, n))
        C = rng.standard_normal((d, n))
    else:
        B = rng.standard_normal((b, g, n, l))
        C = rng.standard_normal((b, g, n, l))
    return dict(u=u, delta=delta, A=A, B=B, C=C,
                D=rng.standard_normal(d) if D else None,
                z=rng.standard_normal((b, d, l)) if z else None,
                delta_bias=rng.uniform(-3, 0.5, d) if bias else None)


# --------------------------------------------------------------------------
# Independent brute force: the recurrence unrolled into its closed sum,
#   x_{n,t} = sum_{k<=t} exp(A_n * sum_{j=k+1..t} dt_j) * dt_k * B_{n,k} * u_k,
# evaluated with math.fsum, and softplus written as log(1 + e^v) directly.
# --------------------------------------------------------------------------
def _brute(p, softplus=True):
    u, delta, A, B, C = p["u"], p["delta"], p["A"], p["B"], p["C"]
    D, z, bias = p["D"], p["z"], p["delta_bias"]
    b_, d_, l_ = u.shape
    n_ = A.shape[1]
    fixed = B.ndim == 2
    g_ = 1 if fixed else B.shape[1]
    out = np.zeros((b_, d_, l_))
    last = np.zeros((b_, d_, n_))
    for b in range(b_):
        for d in range(d_):
            gi = 0 if fixed else d // (d_ // g_)
            v = [float(delta[b, d, t]) + (float(bias[d]) if bias is not None else 0.0) for t in range(l_)]
            dt = [math.log(1.0 + math.exp(x)) if softplus else x for x in v]
            for t in range(l_):
                ys = []
                for n in range(n_):
                    terms = []
                    for k in range(t + 1):
                        s = math.fsum(dt[k + 1:t + 1])
                        Bk = B[d, n] if fixed else B[b, gi, n, k]
                        terms.append(math.exp(A[d, n] * s) * dt[k] * Bk * u[b, d, k])
                    x = math.fsum(terms)
                    Ct = C[d, n] if fixed else C[b, gi, n, t]
                    ys.append(Ct * x)
                    if t == l_ - 1:
                        last[b, d, n] = x
                y = math.fsum(ys) + (D[d] * u[b, d, t] if D is not None else 0.0)
                if z is not None:
                    zz = z[b, d, t]
                    y = y * zz / (1.0 + math.exp(-zz))
                out[b, d, t] = y
    return out, last


@pytest.mark.parametrize("case", [
    dict(b=1, d=2, l=9, n=3, g=1, bc="variable"),
    dict(b=2, d=3, l=7, n=2, g=3, bc="variable"),
    dict(b=2, d=4, l=6, n=4, g=2, bc="variable", z=False),
    dict(b=1, d=3, l=12, n=2, bc="fixed", D=False),
    dict(b=1, d=2, l=5, n=3, bc="fixed", bias=False),
])
@pytest.mark.parametrize("softplus", [True, False])
def test_brute_force(case, softplus):
    case = dict(case)
    rng = np.random.default_rng(7 + case["l"] + 100 * softplus)
    p = _rand_problem(rng, **case)
    if not softplus:  # keep dt positive when the raw delta is the step
        p["delta"] = np.abs(p["delta"]) * 0.3 + 0.01
        p["delta_bias"] = None if p["delta_bias"] is None else np.abs(p["delta_bias"]) * 0.1
    out, last = oracle.selective_scan_ref(**p, delta_softplus=softplus, return_last_state=True)
    bout, blast = _brute(p, softplus)
    assert _rel(out, bout) < RTOL
    assert _rel(last, blast) < RTOL


def test_geometric_closed_form():
    """Constant dt, A, B, C and u: x_t = dt B u (1 - a^{t+1}) / (1 - a), a = e^{dt A}."""
    d, l, n = 3, 40, 4
    A = -np.array([[0.5, 1.0, 2.0, 4.0], [0.1, 0.2, 0.3, 0.4], [3.0, 1.5, 0.75, 0.25]])
    Bf = np.array([[1.0, -0.5, 0.25, 2.0], [0.3, 0.1, -1.0, 1.0], [-2.0, 0.5, 0.5, 1.0]])
    Cf = np.array([[0.7, 0.2, -0.4, 1.1], [1.0, 1.0, 1.0, 1.0], [0.1, -0.3, 0.8, 0.6]])
    delta = np.full((1, d, l), 0.37)
    uval = np.array([1.3, -0.6, 2.0])
    u = np.broadcast_to(uval[None, :, None], (1, d, l)).copy()
    Dv = np.array([0.5, -1.0, 0.0])
    out, last = oracle.selective_scan_ref(u, delta, A, Bf, Cf, D=Dv, return_last_state=True)
    t = np.arange(l)
    for di in range(d):
        dt = 0.37
        a = np.exp(dt * A[di])
        x = dt * Bf[di][:, None] * uval[di] * (1 - a[:, None] ** (t[None, :] + 1)) / (1 - a[:, None])
        y = (Cf[di][:, None] * x).sum(0) + Dv[di] * uval[di]
        assert _rel(out[0, di], y) < 1e-13
        assert _rel(last[0, di], x[:, -1]) < 1e-13


def test_lti_convolution_numpy():
    """Constant step and fixed B/C make the scan LTI: y = conv(u, K) + D u with
    K_k = sum_n C_n a_n^k dt B_n, checked by numpy.convolve."""
    rng = np.random.default_rng(11)
    d, l, n = 4, 300, 8
    A = -rng.uniform(0.01, 2.0, (d, n))
    Bf, Cf = rng.standard_normal((d, n)), rng.standard_normal((d, n))
    Dv = rng.standard_normal(d)
    u = rng.standard_normal((1, d, l))
    v = -1.3
    delta = np.full((1, d, l), v)
    dt = math.log1p(math.exp(v))
    out = oracle.selective_scan_ref(u, delta, A, Bf, Cf, D=Dv, delta_softplus=True)
    for di in range(d):
        a = np.exp(dt * A[di])
        K = (Cf[di][:, None] * (a[:, None] ** np.arange(l)[None, :]) * dt * Bf[di][:, None]).sum(0)
        y = np.convolve(u[0, di], K)[:l] + Dv[di] * u[0, di]
        assert _rel(out[0, di], y) < 1e-11


def test_b_zero_gives_skip_and_gate():
    rng = np.random.default_rng(3)
    p = _rand_problem(rng, 2, 5, 33, 4, g=1)
    p["B"] = np.zeros_like(p["B"])
    out, last = oracle.selective_scan_ref(**p, delta_softplus=True, return_last_state=True)
    zz = p["z"]
    expect = p["D"][None, :, None] * p["u"] * zz / (1 + np.exp(-zz))
    assert _rel(out, expect) < 1e-15
    assert np.all(last == 0.0)


def test_linearity_in_u():
    rng = np.random.default_rng(5)
    p = _rand_problem(rng, 2, 3, 50, 4, g=3)
    u1, u2 = p["u"], rng.standard_normal(p["u"].shape)
    al, be = 0.75, -1.25
    f = lambda uu: oracle.selective_scan_ref(**{**p, "u": uu}, delta_softplus=True, return_last_state=True)
    o1, s1 = f(u1)
    o2, s2 = f(u2)
    o3, s3 = f(al * u1 + be * u2)
    assert _rel(o3, al * o1 + be * o2) < 1e-12
    assert _rel(s3, al * s1 + be * s2) < 1e-12


def test_causality():
    rng = np.random.default_rng(9)
    p = _rand_problem(rng, 1, 3, 64, 4)
    o1 = oracle.selective_scan_ref(**p, delta_softplus=True)
    t0 = 37
    p2 = dict(p)
    for key in ("u", "delta", "z"):
        p2[key] = p[key].copy()
        p2[key][:, :, t0] += 1.5
    B2 = p["B"].copy()
    B2[..., t0] -= 2.0
    p2["B"] = B2
    o2 = oracle.selective_scan_ref(**p2, delta_softplus=True)
    assert np.array_equal(o1[..., :t0], o2[..., :t0])
    assert not np.array_equal(o1[..., t0], o2[..., t0])


def test_last_state_is_prefix_state():
    """last_state of a run on the first L steps equals the brute-force state
    after step L-1 of the longer sequence, and outputs agree on the prefix."""
    rng = np.random.default_rng(13)
    p = _rand_problem(rng, 1, 2, 20, 3, z=False)
    L = 8
    pre = {k: (v[..., :L] if (v is not None and k in ("u", "delta", "z", "B", "C")) else v) for k, v in p.items()}
    o_full = oracle.selective_scan_ref(**p, delta_softplus=True)
    o_pre, s_pre = oracle.selective_scan_ref(**pre, delta_softplus=True, return_last_state=True)
    assert np.array_equal(o_full[..., :L], o_pre)
    _, blast = _brute(pre)
    assert _rel(s_pre, blast) < RTOL


def test_fixed_equals_grouped_per_channel():
    """Fixed (d, n) B/C equal the grouped form with one group per channel and
    B/C constant over time."""
    rng = np.random.default_rng(17)
    b, d, l, n = 2, 6, 25, 4
    p = _rand_problem(rng, b, d, l, n, bc="fixed")
    o1, s1 = oracle.selective_scan_ref(**p, delta_softplus=True, return_last_state=True)
    Bg = np.broadcast_to(p["B"][None, :, :, None], (b, d, n, l)).copy()
    Cg = np.broadcast_to(p["C"][None, :, :, None], (b, d, n, l)).copy()
    o2, s2 = oracle.selective_scan_ref(**{**p, "B": Bg, "C": Cg}, delta_softplus=True, return_last_state=True)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_three_d_equals_four_d_one_group():
    rng = np.random.default_rng(19)
    p = _rand_problem(rng, 2, 4, 30, 3, g=1)
    o4 = oracle.selective_scan_ref(**p, delta_softplus=True)
    o3 = oracle.selective_scan_ref(**{**p, "B": p["B"][:, 0], "C": p["C"][:, 0]}, delta_softplus=True)
    assert np.array_equal(o3, o4)


def test_group_mapping_contiguous_channels():
    """Channel d of a g-group problem behaves as a one-group problem over that
    group's B/C: group index = d // (dim / g)."""
    rng = np.random.default_rng(23)
    b, d, l, n, g = 2, 8, 20, 3, 4
    p = _rand_problem(rng, b, d, l, n, g=g)
    out = oracle.selective_scan_ref(**p, delta_softplus=True)
    dpg = d // g
    for gi in range(g):
        sl = slice(gi * dpg, (gi + 1) * dpg)
        sub = dict(u=p["u"][:, sl], delta=p["delta"][:, sl], A=p["A"][sl],
                   B=p["B"][:, gi:gi + 1], C=p["C"][:, gi:gi + 1], D=p["D"][sl],
                   z=p["z"][:, sl], delta_bias=p["delta_bias"][sl])
        assert np.array_equal(out[:, sl], oracle.selective_scan_ref(**sub, delta_softplus=True))


def test_memoryless_limit():
    """A -> -inf leaves only the current step: y_t = dt u sum_n C B + D u."""
    rng = np.random.default_rng(29)
    p = _rand_problem(rng, 1, 3, 40, 4, z=False)
    p["A"] = np.full_like(p["A"], -1e4)
    p["delta_bias"] = np.full(3, 2.0)  # dt >= ~0.1 so exp(dt A) underflows to 0
    out = oracle.selective_scan_ref(**p, delta_softplus=True)
    v = p["delta"] + p["delta_bias"][None, :, None]
    dt = np.log1p(np.exp(v))
    cb = (p["C"][:, 0] * p["B"][:, 0]).sum(1)  # (b, l)
    expect = dt * p["u"] * cb[:, None, :] + p["D"][None, :, None] * p["u"]
    assert _rel(out, expect) < 1e-13


def test_softplus_and_silu_against_libraries():
    """Single-step, single-state problems isolate softplus and silu:
    out = C dt B u silu(z) with dt = softplus(v). Checked against mpmath at
    40 digits, and against torch's fp64 softplus/silu (threshold lifted: by
    default torch returns v itself for v > 20)."""
    mp = pytest.importorskip("mpmath")
    vs = np.array([-40.0, -20.0, -5.0, -0.5, 0.0, 0.3, 4.0, 19.0, 25.0, 60.0])
    zs = np.array([-30.0, -3.0, -0.2, 0.0, 0.1, 1.0, 5.0, 12.0, -12.0, 40.0])
    m = len(vs)
    u = np.ones((1, m, 1))
    delta = vs.reshape(1, m, 1)
    A = -np.ones((m, 1))
    B = np.ones((m, 1))
    C = np.ones((m, 1))
    out = oracle.selective_scan_ref(u, delta, A, B, C, z=zs.reshape(1, m, 1), delta_softplus=True)
    mp.mp.dps = 40
    exact = [float(mp.log(1 + mp.e ** mp.mpf(v)) * mp.mpf(z) / (1 + mp.e ** (-mp.mpf(z)))) for v, z in zip(vs, zs)]
    np.testing.assert_allclose(out[0, :, 0], exact, rtol=2e-15, atol=0)
    sp = torch.nn.functional.softplus(torch.tensor(vs, dtype=torch.float64), threshold=1e4).numpy()
    si = torch.nn.functional.silu(torch.tensor(zs, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(out[0, :, 0], sp * si, rtol=1e-14, atol=0)


def test_rows_match_whole_problem():
    w = workloads.Workload("t", 2, 8, 48, 4, groups=2, bc_4d=True, dtype="bf16",
                           return_last_state=True, seed=3)
    x = workloads.make_inputs(w)
    args = {k: x[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")}
    full, last = oracle.selective_scan_ref(**args, delta_softplus=True, return_last_state=True)
    rows = [(0, 0), (1, 7), (1, 3), (0, 5)]
    o, s = oracle.selective_scan_rows(rows, **args, delta_softplus=True, threads=2)
    for i, (b, d) in enumerate(rows):
        assert np.array_equal(o[i], full[b, d])
        assert np.array_equal(s[i], last[b, d])


def test_threads_bit_identical():
    w = workloads.WORKLOADS["tiny_fp32"]
    x = workloads.make_inputs(w)
    args = {k: x[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")}
    o1, s1 = oracle.selective_scan_ref(**args, delta_softplus=True, return_last_state=True, threads=1)
    o4, s4 = oracle.selective_scan_ref(**args, delta_softplus=True, return_last_state=True, threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


def test_oracle_rejects_bad_groups():
    rng = np.random.default_rng(1)
    p = _rand_problem(rng, 1, 6, 4, 2, g=1)
    p["B"] = rng.standard_normal((1, 4, 2, 4))
    p["C"] = rng.standard_normal((1, 4, 2, 4))
    with pytest.raises(ValueError):
        oracle.selective_scan_ref(**p)


def test_planted_mistakes_are_caught():
    """Each plausible slip in the recurrence, planted in a CPU copy of the
    per-row loop, fails the brute-force pin (so the pins can see such slips)."""
    rng = np.random.default_rng(31)
    p = _rand_problem(rng, 1, 2, 10, 3, g=1)
    bout, _ = _brute(p)

    def scan(variant):
        u, delta, A, B, C, D, z, bias = (p[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias"))
        out = np.zeros_like(u)
        for d in range(u.shape[1]):
            x = np.zeros(A.shape[1])
            for t in range(u.shape[2]):
                v = delta[0, d, t] + bias[d]
                dt = np.log1p(np.exp(v)) if variant != "no_softplus" else v
                Bt = B[0, 0, :, t]
                Ct = C[0, 0, :, t] if variant != "C_prev" else C[0, 0, :, max(t - 1, 0)]
                a = np.exp(dt * A[d]) if variant != "sign" else np.exp(-dt * A[d])
                xn = a * x + dt * Bt * u[0, d, t]
                y = (Ct * (x if variant == "y_before_update" else xn)).sum()
                x = xn
                y += D[d] * u[0, d, t] * (0 if variant == "no_D" else 1)
                gate = z[0, d, t] / (1 + np.exp(-z[0, d, t]))
                out[0, d, t] = y * (gate if variant != "no_gate" else 1.0)
        return out

    assert _rel(scan("none"), bout) < 1e-12
    for v in ("no_softplus", "C_prev", "sign", "y_before_update", "no_D", "no_gate"):
        assert _rel(scan(v), bout) > 1e-3, v
