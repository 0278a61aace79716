"""GPU parity of the selective-scan backward (ss_bwd, and autograd through
selective_scan_fn) against the fp64 backward oracle, on seeded inputs.

Tolerance, per gradient tensor: max|gpu - oracle| / max|oracle|
  <= 1e-5 for fp32 inputs, the forward's bound. The kernel works in fp32
     throughout; the reduced gradients (dA, dD, ddelta_bias and dB/dC) are
     sums of up to batch x seqlen x dim/groups fp32 terms of mixed sign and
     the adjoint runs through the whole sequence; measured errors stay below
     3e-6 on these cases;
  <= 1e-2 for fp16/bf16 inputs (the per-step gradients du, ddelta, dz are
     rounded once to the input dtype, relative 2^-9 for bf16; the fp32
     reduced gradients are held to the same bound).
"""
import numpy as np
import pytest
import torch

from oracle import backward as bwd_oracle
from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias", "dinitial_state")


def _tol(dtype):
    return 1e-5 if dtype == "fp32" else 1e-2


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.max(np.abs(b)) if b.size else 0.0
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a), initial=0.0))


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


W = workloads.Workload
CASES = [
    # two chunks + a ragged tail, 12 channels per group (a partial CTA of rows)
    (W("bwd_bf16_g2", 2, 24, 300, 16, groups=2, bc_4d=True, dtype="bf16", seed=81), False),
    # odd dstate (the dB/dC buffer parity crosses chunks), fp32 B/C, 3-D B/C
    (W("bwd_fp16_n13", 2, 16, 257, 13, dtype="fp16", bc_dtype="fp32", seed=82), False),
    (W("bwd_fixed_fp32", 2, 16, 520, 8, bc="fixed", bc_std=0.25, dtype="fp32", has_z=False, seed=83), False),
    (W("bwd_fp32_n64", 1, 8, 100, 64, dtype="fp32", seed=84), False),
    (W("bwd_fp32_init_g4", 2, 32, 700, 16, groups=4, bc_4d=True, dtype="fp32", seed=85), True),
    (W("bwd_bf16_plain", 3, 8, 64, 1, dtype="bf16", D_mode="none", has_bias=False, delta_softplus=False,
       delta_std=0.1, seed=86), False),
    (W("bwd_fp32_one_step", 2, 8, 1, 4, dtype="fp32", seed=87), True),
    (W("bwd_fixed_bf16_init", 1, 40, 333, 16, bc="fixed", bc_std=0.25, dtype="bf16", seed=88), True),
]


def _start_state(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((w.batch, w.dim, w.dstate), generator=g, dtype=torch.float32) * 0.5


def _inputs(w):
    x = workloads.make_inputs(w)
    if not w.delta_softplus:  # the raw sum is the step: keep it a positive step size
        x["delta"] = (x["delta"].float().abs() + 0.01).to(x["delta"].dtype)
    return x


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_bwd_matches_oracle(case):
    w, with_init = case
    x = _inputs(w)
    dout = workloads.make_dout(w)
    x0 = _start_state(w, w.seed) if with_init else None
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    got = api.selective_scan_bwd(dout.cuda(), **dev, delta_softplus=w.delta_softplus,
                                 initial_state=None if x0 is None else x0.cuda(), want_dinitial_state=True,
                                 want_dD=True, want_ddelta_bias=True)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref = bwd_oracle.selective_scan_bwd_ref(dout, **{k: x[k] for k in NAMES}, delta_softplus=w.delta_softplus,
                                            initial_state=x0 if x0 is not None else np.zeros((w.batch, w.dim, w.dstate)))
    # absent D / bias: the gradient at 0 (the oracle's with zero-valued inputs)
    if x["D"] is None or x["delta_bias"] is None:
        zD = np.zeros(w.dim) if x["D"] is None else x["D"]
        zb = np.zeros(w.dim) if x["delta_bias"] is None else x["delta_bias"]
        ref0 = bwd_oracle.selective_scan_bwd_ref(dout, x["u"], x["delta"], x["A"], x["B"], x["C"], D=zD, z=x["z"],
                                                 delta_bias=zb, delta_softplus=w.delta_softplus)
        ref["dD"], ref["ddelta_bias"] = ref0["dD"], ref0["ddelta_bias"]
    for k in GRADS:
        if ref[k] is None:
            assert got[k] is None, k
            continue
        assert tuple(got[k].shape) == ref[k].shape, k
        err = _rel(_np(got[k]), ref[k])
        print(f"{w.name} {k} {err:.2e}")
        assert err <= _tol(w.dtype), (k, err)


def test_autograd_through_selective_scan_fn():
    """Gradients of selective_scan_fn (bf16, 3-D B/C, start state) by
    loss.backward() equal the oracle's; last_state carries none."""
    w = W("bwd_autograd", 2, 32, 400, 16, dtype="bf16", seed=91)
    x = _inputs(w)
    dout = workloads.make_dout(w)
    x0 = _start_state(w, 3)
    leaves = {k: x[k].cuda().requires_grad_(True) for k in NAMES}
    s0 = x0.cuda().requires_grad_(True)
    out, last = api.selective_scan_fn(**leaves, delta_softplus=True, return_last_state=True, initial_state=s0)
    assert not last.requires_grad
    (out.float() * dout.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    ref = bwd_oracle.selective_scan_bwd_ref(dout, **{k: x[k] for k in NAMES}, delta_softplus=True, initial_state=x0)
    for k in NAMES:
        g = leaves[k].grad
        assert g is not None and g.dtype == x[k].dtype and g.shape == x[k].shape, k
        assert _rel(_np(g), ref["d" + k]) <= 1e-2, k
    assert _rel(_np(s0.grad), ref["dinitial_state"]) <= 1e-2


def test_bwd_empty_sequence_gives_zeros():
    w = W("bwd_empty", 2, 16, 0, 8, dtype="fp32", seed=92)
    x = _inputs(w)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    dout = torch.empty(2, 16, 0, device="cuda")
    got = api.selective_scan_bwd(dout, **dev, delta_softplus=True, initial_state=torch.ones(2, 16, 8, device="cuda"))
    torch.cuda.synchronize()
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias", "dinitial_state"):
        assert not torch.any(got[k]), k
    assert got["du"].shape == (2, 16, 0)


def test_bwd_strided_views():
    """u, delta, dout as strided views (batch/channel strides), B/C fp32 4-D."""
    w = W("bwd_views", 2, 16, 200, 16, groups=2, bc_4d=True, dtype="fp32", seed=93)
    x = _inputs(w)
    dout = workloads.make_dout(w)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    for k in ("u", "delta", "z"):
        big = torch.zeros(w.batch, w.dim + 3, w.seqlen + 5, device="cuda")
        big[:, :w.dim, :w.seqlen] = dev[k]
        dev[k] = big[:, :w.dim, :w.seqlen]
    got = api.selective_scan_bwd(dout.cuda(), **dev, delta_softplus=True)
    torch.cuda.synchronize()
    ref = bwd_oracle.selective_scan_bwd_ref(dout, **{k: x[k] for k in NAMES}, delta_softplus=True)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        assert _rel(_np(got[k]), ref[k]) <= 1e-5, k


def test_bwd_full_size_sampled():
    """mamba130m_bf16 (8, 1536, 2048, 16) in the launch configuration the
    bench times: batch row 0 in full against the oracle (du, ddelta, dz of all
    its channels and its dB, dC, which depend on that batch row only), and dA,
    dD, ddelta_bias of sampled channels summed over all eight batch rows."""
    w = workloads.WORKLOADS["mamba130m_bf16"]
    x = _inputs(w)
    dout = workloads.make_dout(w)
    dev = {k: (None if x[k] is None else x[k].cuda()) for k in NAMES}
    got = api.selective_scan_bwd(dout.cuda(), **dev, delta_softplus=True)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    one = {k: (x[k][:1] if k in ("u", "delta", "z", "B", "C") else x[k]) for k in NAMES}
    ref = bwd_oracle.selective_scan_bwd_ref(dout[:1], **one, delta_softplus=True)
    for k in ("du", "ddelta", "dz", "dB", "dC"):
        assert _rel(_np(got[k][:1]), ref[k]) <= 1e-2, k
    chans = [0, 517, 1023, 1535]
    rows = [(b, d) for d in chans for b in range(w.batch)]
    parts = bwd_oracle.selective_scan_bwd_rows(rows, dout, **{k: x[k] for k in NAMES}, delta_softplus=True)
    for i, d in enumerate(chans):
        mine = parts[i * w.batch:(i + 1) * w.batch]
        assert _rel(_np(got["dA"][d]), sum(r["dA"] for r in mine)) <= 1e-2
        assert _rel(_np(got["dD"][d]), sum(r["dD"] for r in mine)) <= 1e-2
        assert _rel(_np(got["ddelta_bias"][d]), sum(r["ddelta_bias"] for r in mine)) <= 1e-2


def test_bwd_errors_raise():
    """A missing workspace is refused (SS_ERR_SCRATCH) with nothing written;
    mismatched dtypes are caught by the binding."""
    w = W("bwd_err", 1, 8, 32, 4, dtype="fp32", seed=94)
    x = _inputs(w)
    u, delta, A, B, C, D, z, bias = api.normalise(*(None if x[k] is None else x[k].cuda() for k in NAMES))
    dout = torch.ones_like(u)
    du, ddelta, dz = torch.full_like(u, 7.0), torch.full_like(u, 7.0), torch.full_like(u, 7.0)
    dA = torch.full_like(A, 7.0)
    dB, dC = torch.full(B.shape, 7.0, device="cuda"), torch.full(C.shape, 7.0, device="cuda")
    p = api.make_bwd_params(dout, u, delta, A, B, C, D, z, bias, True, None, du, ddelta, dz, dA, dB, dC,
                            None, None, None)
    with pytest.raises(api.SSError) as e:
        api._check(api.load_library().ss_bwd(api.ctypes.byref(p), None))
    assert e.value.status == 11
    torch.cuda.synchronize()
    assert torch.all(du == 7.0) and torch.all(dA == 7.0) and torch.all(dB == 7.0)
    with pytest.raises(TypeError):
        api.selective_scan_bwd(torch.zeros(1, 8, 32, device="cuda", dtype=torch.float16),
                               *(None if x[k] is None else x[k].cuda() for k in NAMES), delta_softplus=True)
