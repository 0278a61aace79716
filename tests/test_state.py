"""GPU parity of the start-state input of the forward and of the decode step
(selective_state_update) against the fp64 oracle, on seeded inputs.

Tolerances as for the forward: max|gpu - oracle| / max|oracle| <= 1e-5 for
fp32 inputs, <= 1e-2 for fp16/bf16 inputs, per output tensor.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "fp16": 1e-2, "bf16": 1e-2}
TDT = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}
NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


# ---------------------------------------------------------------------------
# forward with a start state
# ---------------------------------------------------------------------------
INIT_CASES = [
    workloads.Workload("init_bf16", 2, 96, 300, 16, groups=2, bc_4d=True, dtype="bf16", return_last_state=True, seed=61),
    workloads.Workload("init_fp16_n13", 2, 40, 257, 13, dtype="fp16", return_last_state=True, seed=62),
    workloads.Workload("init_fp32", 1, 48, 200, 16, dtype="fp32", return_last_state=True, seed=63),
    workloads.Workload("init_fixed_fp32", 1, 64, 333, 16, bc="fixed", bc_std=0.25, dtype="fp32",
                       has_z=False, return_last_state=True, seed=64),
    # few channels, long sequence: the split-sequence schedule folds the start in
    workloads.Workload("init_segmented_fp32", 1, 64, 9000, 16, dtype="fp32", return_last_state=True, seed=65),
    workloads.Workload("init_segmented_fixed", 1, 64, 9000, 8, bc="fixed", bc_std=0.25, dtype="fp32",
                       has_z=False, return_last_state=True, seed=66),
]


def _start_state(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((w.batch, w.dim, w.dstate), generator=g, dtype=torch.float32)


@pytest.mark.parametrize("w", INIT_CASES, ids=lambda w: w.name)
def test_forward_with_initial_state(w):
    x = workloads.make_inputs(w)
    x0 = _start_state(w, w.seed)
    if w.bc == "fixed":
        x["B"][3, 5] = 0.0  # a zero B entry: the start state must still decay there
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    out, last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True,
                                      initial_state=x0.cuda())
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref_out, ref_last = oracle.selective_scan_ref(**{k: x[k] for k in NAMES}, delta_softplus=True,
                                                  return_last_state=True, initial_state=x0, threads=8)
    assert _rel(_np(out), ref_out) <= TOL[w.dtype]
    assert _rel(_np(last), ref_last) <= TOL[w.dtype]


def test_forward_chained_in_place_equals_one_run():
    """Two calls, the second started from the first's last_state in place
    (initial_state is last_state), equal the oracle over the whole sequence."""
    w = workloads.Workload("chain", 2, 64, 400, 16, dtype="fp32", return_last_state=True, seed=67)
    x = workloads.make_inputs(w)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    l1 = 160

    def part(sl):
        d = dict(dev)
        for k in ("u", "delta", "z"):
            d[k] = dev[k][:, :, sl].contiguous()
        for k in ("B", "C"):
            d[k] = dev[k][..., sl].contiguous()
        return d

    o1, st = api.selective_scan_fn(**part(slice(0, l1)), delta_softplus=True, return_last_state=True)
    p2 = part(slice(l1, None))
    u, delta, A, B, C, D, z, bias = api.normalise(*(p2[k] for k in NAMES))
    o2 = torch.empty_like(u)
    p = api.make_params(u, delta, A, B, C, D, z, bias, True, o2, st, st)  # last_state == initial_state
    api._check(api.load_library().ss_fwd(api.ctypes.byref(p), torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    ref_out, ref_last = oracle.selective_scan_ref(**{k: x[k] for k in NAMES}, delta_softplus=True,
                                                  return_last_state=True)
    assert _rel(_np(torch.cat([o1, o2], dim=2)), ref_out) <= 1e-5
    assert _rel(_np(st), ref_last) <= 1e-5


def test_forward_empty_sequence_returns_start_state():
    w = workloads.Workload("empty", 2, 16, 0, 8, dtype="bf16", return_last_state=True, seed=68)
    x = workloads.make_inputs(w)
    x0 = _start_state(w, 3).cuda()
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    _, last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True, initial_state=x0)
    torch.cuda.synchronize()
    assert torch.equal(last, x0)


# ---------------------------------------------------------------------------
# decode step
# ---------------------------------------------------------------------------
def _step_inputs(batch, dim, n, g, dtype, form, seed, bc_f32=False, softplus=True):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=gen)
    dt = TDT[dtype]
    st = r(batch, dim, n)
    u, delta, z = r(batch, dim).to(dt), (0.7 * r(batch, dim)).to(dt), r(batch, dim).to(dt)
    A = -torch.rand(dim, n, generator=gen) * 2.8 - 0.2
    D = r(dim)
    dt0 = torch.rand(dim, generator=gen) * 0.099 + 0.001
    bias = torch.log(torch.expm1(dt0))
    if not softplus:  # the raw sum is the step: keep it positive (a step size)
        delta = (delta.float().abs() * 0.3 + 0.01).to(dt)
        bias = dt0
    bdt = torch.float32 if (bc_f32 or dtype == "fp32" or form == "fixed") else dt
    if form == "fixed":
        B, C = r(dim, n), r(dim, n)
    elif form == "per_token":
        B, C = r(batch, n).to(bdt), r(batch, n).to(bdt)
    else:
        B, C = r(batch, g, n).to(bdt), r(batch, g, n).to(bdt)
    return st, u, delta, A, B, C, D, z, bias


STEP_CASES = [
    # (batch, dim, dstate, groups, dtype, form, bc_f32)
    (4, 1536, 16, 1, "bf16", "per_token", False),
    (3, 520, 16, 4, "bf16", "grouped", False),
    (2, 136, 13, 2, "fp16", "grouped", True),
    (5, 72, 64, 1, "fp32", "per_token", False),
    (2, 96, 1, 1, "fp32", "per_token", False),
    (3, 64, 7, 1, "bf16", "fixed", False),
    (1, 33, 32, 1, "fp16", "per_token", False),
    # larger states and contiguous decode-like shapes
    (2, 256, 64, 1, "fp32", "per_token", False),
    (3, 384, 32, 3, "fp16", "grouped", False),
    (2, 512, 8, 1, "bf16", "per_token", True),
    (1, 1024, 4, 1, "fp32", "per_token", False),
    (2, 128, 16, 1, "bf16", "fixed", False),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: f"{c[4]}_{c[5]}_b{c[0]}d{c[1]}n{c[2]}g{c[3]}")
@pytest.mark.parametrize("softplus", [True, False])
def test_state_update_matches_oracle(case, softplus):
    batch, dim, n, g, dtype, form, bc_f32 = case
    st, u, delta, A, B, C, D, z, bias = _step_inputs(batch, dim, n, g, dtype, form, 70 + n, bc_f32, softplus)
    ref_out, ref_state = oracle.selective_state_update_ref(st, u, delta, A, B, C, D=D, z=z, delta_bias=bias,
                                                           delta_softplus=softplus, bc_fixed=form == "fixed")
    s = st.cuda()
    out = api.selective_state_update(s, u.cuda(), delta.cuda(), A.cuda(), B.cuda(), C.cuda(), D=D.cuda(),
                                     z=z.cuda(), delta_bias=bias.cuda(), delta_softplus=softplus,
                                     bc_fixed=form == "fixed")
    torch.cuda.synchronize()
    assert _rel(_np(out), ref_out) <= TOL[dtype]
    assert _rel(_np(s), ref_state) <= (1e-5 if dtype == "fp32" else 1e-3)


@pytest.mark.parametrize("q", [1, 2, 4])
@pytest.mark.parametrize("case", [c for c in STEP_CASES if c[2] in (13, 16, 32, 64)],
                         ids=lambda c: f"{c[4]}_{c[5]}_n{c[2]}")
def test_state_update_every_lane_split(case, q, monkeypatch):
    """Every split of a channel's states over lanes (4, 8 or 16 states a lane;
    the default is 8) gives the oracle's result."""
    monkeypatch.setenv("SSFWD_SU_Q", str(q))
    batch, dim, n, g, dtype, form, bc_f32 = case
    st, u, delta, A, B, C, D, z, bias = _step_inputs(batch, dim, n, g, dtype, form, 90 + n, bc_f32)
    ref_out, ref_state = oracle.selective_state_update_ref(st, u, delta, A, B, C, D=D, z=z, delta_bias=bias,
                                                           delta_softplus=True, bc_fixed=form == "fixed")
    s = st.cuda()
    out = api.selective_state_update(s, u.cuda(), delta.cuda(), A.cuda(), B.cuda(), C.cuda(), D=D.cuda(),
                                     z=z.cuda(), delta_bias=bias.cuda(), delta_softplus=True,
                                     bc_fixed=form == "fixed")
    torch.cuda.synchronize()
    assert _rel(_np(out), ref_out) <= TOL[dtype]
    assert _rel(_np(s), ref_state) <= (1e-5 if dtype == "fp32" else 1e-3)


def test_state_update_optional_operands_and_views():
    """No z, D or bias; state as a strided view (odd row stride: the scalar path)."""
    batch, dim, n = 3, 80, 16
    st, u, delta, A, B, C, D, z, bias = _step_inputs(batch, dim, n, 1, "fp32", "per_token", 91)
    big = torch.zeros(batch, dim, n + 3)
    big[:, :, :n] = st
    s = big.cuda()[:, :, :n]
    out = api.selective_state_update(s, u.cuda(), delta.cuda(), A.cuda(), B.cuda(), C.cuda(), delta_softplus=True)
    torch.cuda.synchronize()
    ref_out, ref_state = oracle.selective_state_update_ref(st, u, delta, A, B, C, delta_softplus=True)
    assert _rel(_np(out), ref_out) <= 1e-5
    assert _rel(_np(s), ref_state) <= 1e-5


def test_state_updates_chain_to_the_forward():
    """k decode steps on the GPU from a start state agree with the forward
    oracle over the same k steps from that state."""
    w = workloads.Workload("decode_chain", 2, 256, 12, 16, dtype="bf16", return_last_state=True, seed=93)
    x = workloads.make_inputs(w)
    x0 = _start_state(w, 5)
    ref_out, ref_last = oracle.selective_scan_ref(**{k: x[k] for k in NAMES}, delta_softplus=True,
                                                  return_last_state=True, initial_state=x0)
    s = x0.cuda()
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    outs = []
    for t in range(w.seqlen):
        outs.append(api.selective_state_update(
            s, dev["u"][:, :, t], dev["delta"][:, :, t], dev["A"], dev["B"][..., t], dev["C"][..., t],
            D=dev["D"], z=dev["z"][:, :, t], delta_bias=dev["delta_bias"], delta_softplus=True))
    torch.cuda.synchronize()
    assert _rel(_np(torch.stack(outs, dim=2)), ref_out) <= 1e-2
    assert _rel(_np(s), ref_last) <= 1e-3


def test_state_update_errors_raise_and_empty_is_noop():
    st, u, delta, A, B, C, D, z, bias = _step_inputs(2, 32, 16, 1, "bf16", "per_token", 95)
    s = st.cuda()
    out = torch.empty(2, 32, dtype=torch.bfloat16, device="cuda")
    p = api.make_state_update_params(s, u.cuda(), delta.cuda(), A.cuda(), B.cuda(), C.cuda(), None, None, None,
                                     True, out)
    p.out = s.data_ptr()  # out inside the state: rejected, nothing launched
    with pytest.raises(api.SSError):
        api._check(api.load_library().ss_state_update(api.ctypes.byref(p), None))
    before = s.clone()
    torch.cuda.synchronize()
    assert torch.equal(s, before)
    e = torch.empty(0, 32, 16, device="cuda")
    out = api.selective_state_update(e, torch.empty(0, 32, device="cuda"), torch.empty(0, 32, device="cuda"),
                                     A.cuda(), torch.empty(0, 16, device="cuda"), torch.empty(0, 16, device="cuda"))
    torch.cuda.synchronize()
    assert out.shape == (0, 32)

