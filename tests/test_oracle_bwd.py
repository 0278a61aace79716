"""Pins for the selective-scan backward oracle (``oracle/backward.py``): the
gradients of sum(dout * out) for the section 4.1 operator of the page
"PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南",
whose backward the page routes to a CUDA kernel returning every input's
gradient.

Each pin checks against something other than the oracle itself:
  - central finite differences of the independently written C forward oracle
    (truncation error O(h^2), here far below the 1e-7 bound used);
  - torch.autograd through a plain torch fp64 forward written in this file;
  - slips planted in the oracle's helpers, each of which the finite-difference
    pin must catch.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bwd

KEYS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias", "dinitial_state")
ARG_OF = {"du": "u", "ddelta": "delta", "dA": "A", "dB": "B", "dC": "C", "dD": "D", "dz": "z",
          "ddelta_bias": "delta_bias", "dinitial_state": "initial_state"}


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _problem(seed, b, d, l, n, g=1, form="grouped", z=True, D=True, bias=True, init=False):
    rng = np.random.default_rng(seed)
    p = dict(u=rng.standard_normal((b, d, l)),
             delta=rng.standard_normal((b, d, l)) * 0.7,
             A=-rng.uniform(0.2, 2.0, (d, n)))
    if form == "fixed":
        p["B"], p["C"] = rng.standard_normal((d, n)), rng.standard_normal((d, n))
    elif form == "3d":
        p["B"], p["C"] = rng.standard_normal((b, n, l)), rng.standard_normal((b, n, l))
    else:
        p["B"], p["C"] = rng.standard_normal((b, g, n, l)), rng.standard_normal((b, g, n, l))
    p["D"] = rng.standard_normal(d) if D else None
    p["z"] = rng.standard_normal((b, d, l)) if z else None
    p["delta_bias"] = rng.uniform(-1.5, 0.5, d) if bias else None
    p["initial_state"] = rng.standard_normal((b, d, n)) if init else None
    dout = rng.standard_normal((b, d, l))
    return p, dout


def _loss(p, dout, softplus):
    out = oracle.selective_scan_ref(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"],
                                    delta_bias=p["delta_bias"], delta_softplus=softplus,
                                    initial_state=p["initial_state"])
    return float(np.sum(dout * out))


def _finite_differences(p, dout, softplus, h=1e-5):
    """Central differences of sum(dout * out), one input element at a time."""
    grads = {}
    for key in KEYS:
        name = ARG_OF[key]
        if p[name] is None:
            continue
        x = p[name]
        gr = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = x[i]
            step = h * max(1.0, abs(old))
            x[i] = old + step
            lp = _loss(p, dout, softplus)
            x[i] = old - step
            lm = _loss(p, dout, softplus)
            x[i] = old
            gr[i] = (lp - lm) / (2 * step)
        grads[key] = gr
    return grads


CASES = [
    dict(seed=1, b=2, d=4, l=7, n=3, g=2, form="grouped", softplus=True),
    dict(seed=2, b=1, d=3, l=6, n=2, form="3d", z=False, softplus=True),
    dict(seed=3, b=2, d=2, l=5, n=3, form="fixed", softplus=False),
    dict(seed=4, b=1, d=2, l=6, n=2, g=1, form="grouped", D=False, bias=False, softplus=True),
    dict(seed=5, b=2, d=2, l=5, n=2, g=2, form="grouped", init=True, softplus=True),
    dict(seed=6, b=1, d=2, l=4, n=3, form="fixed", init=True, z=False, softplus=True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['form']}_s{c['seed']}")
def test_against_finite_differences(case):
    case = dict(case)
    softplus = case.pop("softplus")
    p, dout = _problem(**case)
    got = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=softplus)
    fd = _finite_differences(p, dout, softplus)
    for key, ref in fd.items():
        assert got[key] is not None, key
        assert got[key].shape == ref.shape, key
        assert _rel(got[key], ref) < 1e-7, key
    for key in KEYS:  # gradients of absent inputs are absent
        if key not in fd:
            assert got[key] is None, key


def _torch_forward(u, delta, A, B, C, D, z, bias, x0, softplus):
    """Plain torch fp64 forward (grouped B/C), written out step by step."""
    b, d, l = u.shape
    g = B.shape[1]
    grp = torch.arange(d) // (d // g)
    Bt, Ct = B[:, grp], C[:, grp]                             # (b, d, n, l)
    v = delta + bias[None, :, None]
    dt = torch.nn.functional.softplus(v) if softplus else v
    x = x0
    ys = []
    for t in range(l):
        x = torch.exp(dt[:, :, t, None] * A) * x + (dt[:, :, t] * u[:, :, t])[:, :, None] * Bt[..., t]
        ys.append((Ct[..., t] * x).sum(-1) + D * u[:, :, t])
    y = torch.stack(ys, dim=2)
    return y * torch.nn.functional.silu(z)


@pytest.mark.parametrize("softplus", [True, False])
def test_against_torch_autograd(softplus):
    p, dout = _problem(11, 2, 6, 20, 4, g=3, init=True)
    if not softplus:
        p["delta"] = np.abs(p["delta"]) * 0.3 + 0.05
        p["delta_bias"] = np.abs(p["delta_bias"]) * 0.1
    got = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=softplus)
    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "initial_state")
    ts = {k: torch.tensor(p[k], dtype=torch.float64, requires_grad=True) for k in names}
    out = _torch_forward(*(ts[k] for k in names), softplus)
    (out * torch.tensor(dout)).sum().backward()
    for key in KEYS:
        assert _rel(got[key], ts[ARG_OF[key]].grad.numpy()) < 1e-12, key


def test_rows_match_the_whole_problem():
    """Per-row parts add up to the whole-problem gradients (grouped B/C)."""
    p, dout = _problem(21, 2, 4, 9, 3, g=2, init=True)
    whole = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=True)
    rows = [(b, d) for b in range(2) for d in range(4)]
    parts = bwd.selective_scan_bwd_rows(rows, dout, **p, delta_softplus=True)
    dA, dB = np.zeros_like(whole["dA"]), np.zeros_like(whole["dB"])
    for (b, d), r in zip(rows, parts):
        assert _rel(r["du"], whole["du"][b, d]) < 1e-14
        assert _rel(r["ddelta"], whole["ddelta"][b, d]) < 1e-14
        assert _rel(r["dz"], whole["dz"][b, d]) < 1e-14
        assert _rel(r["dinitial_state"], whole["dinitial_state"][b, d]) < 1e-14
        dA[d] += r["dA"]
        dB[b, d // 2] += r["dB"]
    assert _rel(dA, whole["dA"]) < 1e-13
    assert _rel(dB, whole["dB"]) < 1e-13


def test_empty_sequence_gives_zero_gradients():
    p, dout = _problem(31, 2, 3, 0, 4, g=1, init=True)
    got = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=True)
    for key in KEYS:
        assert got[key].shape == p[ARG_OF[key]].shape
        assert not np.any(got[key]), key


@pytest.mark.parametrize("slip", ["adjoint_decays_by_own_step", "no_softplus_derivative", "one_group_sum",
                                  "silu_derivative_as_sigmoid"])
def test_planted_slips_fail_finite_differences(slip, monkeypatch):
    """Plausible slips planted in the oracle (the adjoint decaying by its own
    step's factor a_t instead of a_{t+1}, softplus' derivative dropped, the B/C
    gradient summed over all channels instead of each group's, silu's
    derivative taken as the sigmoid alone) are caught by the finite-difference
    pin."""
    p, dout = _problem(41, 2, 4, 6, 3, g=2)
    fd = _finite_differences(p, dout, True)
    got = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=True)
    assert max(_rel(got[k], fd[k]) for k in fd) < 1e-7
    if slip == "adjoint_decays_by_own_step":
        monkeypatch.setattr(bwd, "_DECAY_OFFSET", 0)
    elif slip == "no_softplus_derivative":
        monkeypatch.setattr(bwd, "_dsoftplus", lambda v: np.ones_like(v))
    elif slip == "silu_derivative_as_sigmoid":
        monkeypatch.setattr(bwd, "_dsilu", bwd._sigmoid)
    else:
        monkeypatch.setattr(bwd, "_group_sum",
                            lambda x, ng: np.repeat(x.sum(axis=1, keepdims=True), ng, axis=1)[:, :ng])
    got = bwd.selective_scan_bwd_ref(dout, **p, delta_softplus=True)
    assert max(_rel(got[k], fd[k]) for k in fd) > 1e-3


def test_golden_tiny_backward():
    """The backward oracle on the tiny workload equals the committed fixture
    (written by tests/golden/make_golden.py, which calls only the oracles); a
    guard against later changes to the oracle, the generator or dout's draw.
    libm may differ by an ulp between hosts, hence 1e-12 and not equality."""
    import json
    import os
    from state_space_model_03_gb300 import workloads
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_fp32_bwd_oracle.json")
    with open(path) as f:
        doc = json.load(f)
    w = workloads.WORKLOADS["tiny_fp32"]
    x = workloads.make_inputs(w)
    dout = workloads.make_dout(w)
    assert dout.reshape(-1)[:6].tolist() == doc["dout_head"]
    got = bwd.selective_scan_bwd_ref(dout, x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                     delta_bias=x["delta_bias"], delta_softplus=True)
    for k, vals in doc["grads"].items():
        ref = np.array([float(v) for v in vals])
        assert np.max(np.abs(got[k].reshape(-1) - ref)) <= 1e-12 * np.max(np.abs(ref)), k
