"""GPU parity of the complex-A forward (ss_fwd_complex, through
selective_scan_fn with a complex64 A) against the fp64 complex-A oracle.

Tolerance as for the real forward: max|gpu - oracle| / max|oracle| <= 1e-5
for fp32 inputs, <= 1e-2 for fp16/bf16 inputs, per output tensor (out, and
the complex last_state compared as complex numbers).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import complex_a
from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
TOL = {"fp32": 1e-5, "fp16": 1e-2, "bf16": 1e-2}


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = np.max(np.abs(b)) if b.size else 0.0
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a), initial=0.0))


def _np(t):
    t = t.detach().cpu()
    return t.to(torch.complex128).numpy() if t.is_complex() else t.to(torch.float64).numpy()


def _inputs(w, seed, im=3.0):
    x = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(seed)
    re = -(torch.rand(w.dim, w.dstate, generator=g) * 1.8 + 0.2)
    imag = (torch.rand(w.dim, w.dstate, generator=g) * 2 - 1) * im
    x["A"] = torch.complex(re, imag)
    return x


W = workloads.Workload
CASES = [
    (W("cx_bf16_g2", 2, 24, 300, 16, groups=2, bc_4d=True, dtype="bf16", seed=101), False),
    (W("cx_fixed_fp32_n13", 2, 20, 333, 13, bc="fixed", bc_std=0.25, dtype="fp32", seed=102), True),
    (W("cx_fp16_n40", 1, 16, 100, 40, dtype="fp16", bc_dtype="fp32", seed=103), True),
    (W("cx_fp32_n64", 2, 20, 70, 64, dtype="fp32", seed=104), False),
    (W("cx_fp32_plain", 1, 8, 50, 4, dtype="fp32", has_z=False, D_mode="none", has_bias=False,
       delta_softplus=False, delta_std=0.1, seed=105), False),
]
# large imaginary parts: rotation angles dt Im A of tens of radians per step
FAST_ROTATION = W("cx_fp32_fast_rotation", 2, 16, 200, 16, dtype="fp32", seed=109)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_complex_matches_oracle(case):
    w, with_init = case
    x = _inputs(w, w.seed)
    if not w.delta_softplus:  # the raw sum is the step: keep it positive
        x["delta"] = (x["delta"].float().abs() + 0.01).to(x["delta"].dtype)
    x0 = None
    if with_init:
        g = torch.Generator().manual_seed(w.seed + 1)
        x0 = torch.complex(torch.randn(w.batch, w.dim, w.dstate, generator=g),
                           torch.randn(w.batch, w.dim, w.dstate, generator=g))
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    out, last = api.selective_scan_fn(**dev, delta_softplus=w.delta_softplus, return_last_state=True,
                                      initial_state=None if x0 is None else x0.cuda())
    torch.cuda.synchronize()
    assert last.dtype == torch.complex64
    ref_out, ref_last = complex_a.selective_scan_complex_ref(**{k: x[k] for k in NAMES},
                                                             delta_softplus=w.delta_softplus,
                                                             return_last_state=True, initial_state=x0)
    assert _rel(_np(out), ref_out) <= TOL[w.dtype]
    assert _rel(_np(last), ref_last) <= (1e-5 if w.dtype == "fp32" else 1e-3)


def test_fast_rotations():
    """|Im A| up to 300: per-step angles dt Im A of tens of radians, so any
    relative error of the step or of the angle becomes a phase error that
    grows with |angle|. Held to the fp32 bound like every other fp32 case."""
    w = FAST_ROTATION
    x = _inputs(w, w.seed, im=300.0)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    out, last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True)
    torch.cuda.synchronize()
    ref_out, ref_last = complex_a.selective_scan_complex_ref(**{k: x[k] for k in NAMES}, delta_softplus=True,
                                                             return_last_state=True)
    v = x["delta"].double() + x["delta_bias"].double()[None, :, None]
    dt_max = float(torch.nn.functional.softplus(v).max())
    angle = dt_max * float(x["A"].imag.abs().max())
    assert angle > 20.0  # the case does exercise the range reduction
    assert _rel(_np(out), ref_out) <= TOL["fp32"]
    assert _rel(_np(last), ref_last) <= TOL["fp32"]


def test_real_valued_A_equals_the_real_forward():
    """A complex A with zero imaginary part gives the real forward's result
    (the two kernels share no code) within the fp32 bound."""
    w = W("cx_vs_real", 2, 32, 500, 16, dtype="fp32", seed=106)
    x = workloads.make_inputs(w)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    out_r, last_r = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True)
    dev["A"] = torch.complex(dev["A"], torch.zeros_like(dev["A"]))
    out_c, last_c = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True)
    torch.cuda.synchronize()
    assert _rel(_np(out_c), _np(out_r)) <= 1e-5
    assert _rel(_np(last_c).real, _np(last_r)) <= 1e-5 and not torch.any(last_c.imag)


def test_empty_sequence_and_in_place_start():
    w = W("cx_empty", 2, 16, 0, 8, dtype="bf16", seed=107)
    x = _inputs(w, 7)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    x0 = torch.complex(torch.randn(2, 16, 8), torch.randn(2, 16, 8)).cuda()
    _, last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True, initial_state=x0)
    torch.cuda.synchronize()
    assert torch.equal(last, x0)


def test_complex_full_size_sampled():
    """mamba130m_bf16's shape with an S4D-Lin-like complex A (-1/2 + i pi n):
    sampled (batch, channel) rows of out and last_state against the oracle."""
    w = workloads.WORKLOADS["mamba130m_bf16"]
    x = workloads.make_inputs(w)
    n = torch.arange(w.dstate, dtype=torch.float32)
    x["A"] = torch.complex(torch.full((w.dim, w.dstate), -0.5), (np.pi * n).expand(w.dim, w.dstate).contiguous())
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    out, last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True)
    torch.cuda.synchronize()
    o, s = _np(out), _np(last)
    for b, d in [(0, 0), (3, 517), (7, 1535), (5, 1024)]:
        sl = {k: (x[k][b:b + 1, d:d + 1] if k in ("u", "delta", "z") else x[k]) for k in NAMES}
        sl["A"], sl["D"], sl["delta_bias"] = x["A"][d:d + 1], x["D"][d:d + 1], x["delta_bias"][d:d + 1]
        sl["B"], sl["C"] = x["B"][b:b + 1], x["C"][b:b + 1]
        ro, rl = complex_a.selective_scan_complex_ref(**sl, delta_softplus=True, return_last_state=True)
        assert _rel(o[b, d], ro[0, 0]) <= 1e-2, (b, d)
        assert _rel(s[b, d], rl[0, 0]) <= 1e-3, (b, d)


def test_complex_forward_has_no_gradient():
    w = W("cx_grad", 1, 8, 16, 4, dtype="fp32", seed=108)
    x = _inputs(w, 8)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    dev["u"].requires_grad_(True)
    with pytest.raises(NotImplementedError):
        api.selective_scan_fn(**dev, delta_softplus=True)
