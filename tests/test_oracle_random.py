"""Randomised pins for the oracles (CPU): the same independent checks as the
fixed cases, over shapes, group counts, options and value ranges drawn by
hypothesis, so that a slip that only shows for some shape or option
combination still fails. Each example is small enough for finite differences.

- backward: central finite differences of the C forward oracle;
- forward: a run split in two at a random step, the second part started from
  the first part's last_state, equals the whole run (composition law);
- complex A: the same composition law, and conj(A) invariance of the output;
- conv1d: numpy.convolve of each row with the reversed taps;
- decode step: k one-step updates (numpy) equal the C forward over k steps.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import backward as bwd  # noqa: E402
from oracle import complex_a  # noqa: E402


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


@st.composite
def problems(draw, max_l=6, complex_A=False):
    b = draw(st.integers(1, 2))
    g = draw(st.sampled_from([1, 2]))
    d = g * draw(st.integers(1, 2))
    l = draw(st.integers(1, max_l))
    n = draw(st.integers(1, 3))
    form = draw(st.sampled_from(["fixed", "3d", "4d"]))
    if form == "3d":
        g = 1
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    p = dict(u=rng.standard_normal((b, d, l)),
             delta=rng.standard_normal((b, d, l)) * draw(st.sampled_from([0.3, 1.0])),
             A=-rng.uniform(0.1, 2.5, (d, n)))
    if complex_A:
        p["A"] = p["A"] + 1j * rng.uniform(-4, 4, (d, n))
    if form == "fixed":
        p["B"], p["C"] = rng.standard_normal((d, n)), rng.standard_normal((d, n))
    elif form == "3d":
        p["B"], p["C"] = rng.standard_normal((b, n, l)), rng.standard_normal((b, n, l))
    else:
        p["B"], p["C"] = rng.standard_normal((b, g, n, l)), rng.standard_normal((b, g, n, l))
    p["D"] = rng.standard_normal(d) if draw(st.booleans()) else None
    p["z"] = rng.standard_normal((b, d, l)) if draw(st.booleans()) else None
    p["delta_bias"] = rng.uniform(-1.5, 0.5, d) if draw(st.booleans()) else None
    if draw(st.booleans()):
        x0 = rng.standard_normal((b, d, n))
        p["initial_state"] = x0 + 1j * rng.standard_normal((b, d, n)) if complex_A else x0
    else:
        p["initial_state"] = None
    softplus = draw(st.booleans())
    if not softplus:  # the raw sum is the step: keep it positive
        p["delta"] = np.abs(p["delta"]) * 0.3 + 0.05
        if p["delta_bias"] is not None:
            p["delta_bias"] = np.abs(p["delta_bias"]) * 0.1
    return p, softplus, rng.standard_normal((b, d, l))


def _loss(p, dout, softplus):
    out = oracle.selective_scan_ref(**p, delta_softplus=softplus)
    return float(np.sum(dout * out))


@settings(max_examples=25, deadline=None)
@given(problems())
def test_backward_against_finite_differences(case):
    p, softplus, dout = case
    got = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=softplus)
    names = {"du": "u", "ddelta": "delta", "dA": "A", "dB": "B", "dC": "C", "dD": "D", "dz": "z",
             "ddelta_bias": "delta_bias", "dinitial_state": "initial_state"}
    for key, name in names.items():
        if p[name] is None:
            assert got[key] is None
            continue
        x = p[name]
        fd = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            old = x[i]
            h = 1e-5 * max(1.0, abs(old))
            x[i] = old + h
            lp = _loss(p, dout, softplus)
            x[i] = old - h
            lm = _loss(p, dout, softplus)
            x[i] = old
            fd[i] = (lp - lm) / (2 * h)
        assert _rel(got[key], fd) < 1e-6, key


def _split(p, l1, fixed):
    def part(sl):
        q = dict(p)
        for k in ("u", "delta", "z"):
            if p[k] is not None:
                q[k] = np.ascontiguousarray(p[k][:, :, sl])
        if not fixed:
            for k in ("B", "C"):
                q[k] = np.ascontiguousarray(p[k][..., sl])
        return q
    return part(slice(0, l1)), part(slice(l1, None))


@settings(max_examples=25, deadline=None)
@given(problems(max_l=12), st.data())
def test_forward_split_run_composes(case, data):
    p, softplus, _ = case
    l = p["u"].shape[2]
    l1 = data.draw(st.integers(0, l))
    full, last = oracle.selective_scan_ref(**p, delta_softplus=softplus, return_last_state=True)
    first, second = _split(p, l1, p["B"].ndim == 2)
    o1, s1 = oracle.selective_scan_ref(**first, delta_softplus=softplus, return_last_state=True)
    second["initial_state"] = s1
    o2, s2 = oracle.selective_scan_ref(**second, delta_softplus=softplus, return_last_state=True)
    assert _rel(np.concatenate([o1, o2], axis=2), full) < 1e-12
    assert _rel(s2, last) < 1e-12


@settings(max_examples=25, deadline=None)
@given(problems(max_l=12, complex_A=True), st.data())
def test_complex_split_run_composes_and_is_conjugation_invariant(case, data):
    p, softplus, _ = case
    l = p["u"].shape[2]
    l1 = data.draw(st.integers(0, l))
    full, last = complex_a.selective_scan_complex_ref(**p, delta_softplus=softplus, return_last_state=True)
    first, second = _split(p, l1, p["B"].ndim == 2)
    o1, s1 = complex_a.selective_scan_complex_ref(**first, delta_softplus=softplus, return_last_state=True)
    second["initial_state"] = s1
    o2, s2 = complex_a.selective_scan_complex_ref(**second, delta_softplus=softplus, return_last_state=True)
    assert _rel(np.concatenate([o1, o2], axis=2), full) < 1e-12
    assert _rel(s2, last) < 1e-12
    conj = dict(p, A=np.conj(p["A"]))
    if p["initial_state"] is not None:
        conj["initial_state"] = np.conj(p["initial_state"])
    out_c = complex_a.selective_scan_complex_ref(**conj, delta_softplus=softplus)
    assert _rel(out_c, full) < 1e-12


@settings(max_examples=25, deadline=None)
@given(st.integers(1, 2), st.integers(1, 4), st.integers(1, 24), st.sampled_from([2, 3, 4]),
       st.booleans(), st.booleans(), st.integers(0, 2 ** 31 - 1))
def test_conv1d_against_numpy_convolve(b, d, l, width, with_init, silu, seed):
    """The conv1d oracle equals numpy.convolve of each row (prefixed by its
    initial states) with the reversed taps, plus bias, then silu."""
    from oracle import conv1d
    rng = np.random.default_rng(seed)
    x, w, bias = rng.standard_normal((b, d, l)), rng.standard_normal((d, width)), rng.standard_normal(d)
    init = rng.standard_normal((b, d, width - 1)) if with_init else None
    out = conv1d.causal_conv1d_ref(x, w, bias, initial_states=init, activation="silu" if silu else None)
    for bi in range(b):
        for di in range(d):
            pre = init[bi, di] if with_init else np.zeros(width - 1)
            row = np.concatenate([pre, x[bi, di]])
            ref = np.convolve(row, w[di][::-1])[width - 1:width - 1 + l] + bias[di]
            if silu:
                ref = ref / (1.0 + np.exp(-ref))
            assert _rel(out[bi, di], ref) < 1e-12


@settings(max_examples=25, deadline=None)
@given(problems(max_l=8))
def test_decode_steps_equal_the_forward(case):
    """k one-step updates from a start state reproduce the forward oracle's
    k-step run from it (variable B/C: per-step slices; fixed: the same B/C)."""
    p, softplus, _ = case
    b, d, l = p["u"].shape
    n = p["A"].shape[1]
    x0 = p["initial_state"] if p["initial_state"] is not None else np.zeros((b, d, n))
    out, last = oracle.selective_scan_ref(**dict(p, initial_state=x0), delta_softplus=softplus,
                                          return_last_state=True)
    fixed = p["B"].ndim == 2
    st_ = x0
    for t in range(l):
        Bt = p["B"] if fixed else p["B"][..., t]
        Ct = p["C"] if fixed else p["C"][..., t]
        o, st_ = oracle.selective_state_update_ref(st_, p["u"][:, :, t], p["delta"][:, :, t], p["A"], Bt, Ct,
                                                   D=p["D"], z=None if p["z"] is None else p["z"][:, :, t],
                                                   delta_bias=p["delta_bias"], delta_softplus=softplus,
                                                   bc_fixed=fixed)
        assert _rel(o, out[:, :, t]) < 1e-12
    assert _rel(st_, last) < 1e-12
