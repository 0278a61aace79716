"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.

Tolerance (per output tensor, out and last_state separately):
  max|gpu - oracle| / max|oracle| <= 1e-5 for fp32 inputs, <= 1e-2 for
  fp16/bf16 inputs.
At full workload sizes the oracle is evaluated on sampled (batch, channel)
rows (first/last channels, group and tile boundaries, random rows), in the
launch configuration the bench times; everywhere the outputs must be finite.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
TOL = {"fp32": 1e-5, "fp16": 1e-2, "bf16": 1e-2}


def _rel(a, b):
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


def _to_dev(x):
    return {k: (None if x[k] is None else x[k].to("cuda")) for k in NAMES}


def _run(x, dev=None):
    dev = dev or _to_dev(x)
    res = api.selective_scan_fn(**dev, delta_softplus=x["delta_softplus"],
                                return_last_state=x["return_last_state"])
    torch.cuda.synchronize()
    assert api.device_error() == 0
    return res if x["return_last_state"] else (res, None)


def _check_full(w, x, out, last):
    ref = oracle.selective_scan_ref(**{k: x[k] for k in NAMES}, delta_softplus=x["delta_softplus"],
                                    return_last_state=x["return_last_state"], threads=8)
    ref_out, ref_last = ref if x["return_last_state"] else (ref, None)
    o = out.double().cpu().numpy()
    e = _rel(o, ref_out)
    assert np.isfinite(o).all()
    assert e <= TOL[w.dtype], f"out {e:.3e}"
    if ref_last is not None:
        s = last.double().cpu().numpy()
        el = _rel(s, ref_last)
        assert el <= TOL[w.dtype], f"last_state {el:.3e}"
        return e, el
    return e, None


def _sample_rows(w, k=24, seed=0):
    rng = np.random.default_rng(seed)
    dpg = w.dim // (w.groups if w.bc == "variable" else 1)
    rows = {(0, 0), (w.batch - 1, w.dim - 1), (0, w.dim - 1), (w.batch - 1, 0)}
    for gi in range(1, w.groups):
        rows |= {(0, gi * dpg - 1), (w.batch - 1, gi * dpg)}
    for t in (31, 32, 33, 63, 64):  # tile boundaries
        if t < w.dim:
            rows.add((0, t))
    while len(rows) < k:
        rows.add((int(rng.integers(w.batch)), int(rng.integers(w.dim))))
    return sorted(rows)


@pytest.mark.parametrize("name", ["mamba130m_bf16", "mamba130m_bf16_l2047", "grouped_bf16", "mamba2p8b_fp16",
                                  "long_fixed_fp32"])
def test_workload_full_size_sampled(name):
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    out, last = _run(x)
    assert torch.isfinite(out.float()).all()
    rows = _sample_rows(w)
    ro, rl = oracle.selective_scan_rows(rows, **{k: x[k] for k in NAMES}, delta_softplus=True, threads=8)
    bi = torch.tensor([r[0] for r in rows])
    di = torch.tensor([r[1] for r in rows])
    go = out[bi, di].double().cpu().numpy()
    e = _rel(go, ro)
    assert e <= TOL[w.dtype], f"{name} out {e:.3e}"
    if last is not None:
        assert torch.isfinite(last).all()
        gl = last[bi, di].double().cpu().numpy()
        el = _rel(gl, rl)
        assert el <= TOL[w.dtype], f"{name} last_state {el:.3e}"


def test_tiny_workload_full():
    w = workloads.WORKLOADS["tiny_fp32"]
    x = workloads.make_inputs(w)
    out, last = _run(x)
    _check_full(w, x, out, last)


SWEEP = [
    # (batch, dim, seqlen, dstate, groups, bc, dtype, bc_dtype, z, D, bias, softplus, last)
    (1, 16, 1, 16, 1, "variable", "bf16", None, True, True, True, True, True),
    (2, 37, 7, 16, 1, "variable", "bf16", None, True, True, True, True, True),
    (2, 40, 128, 16, 4, "variable", "fp16", None, True, True, True, True, True),
    (1, 33, 1000, 16, 1, "variable", "fp32", None, False, True, True, True, True),
    (2, 64, 4096, 16, 2, "variable", "bf16", None, True, True, True, True, True),
    (1, 24, 300, 4, 1, "variable", "bf16", None, True, False, True, True, True),
    (1, 24, 300, 5, 3, "variable", "fp32", None, True, True, False, True, True),
    (2, 20, 257, 8, 1, "variable", "fp16", None, False, True, True, False, True),
    (1, 36, 200, 32, 2, "variable", "bf16", None, True, True, True, True, True),
    (1, 16, 130, 64, 1, "variable", "fp32", None, True, True, True, True, True),
    (1, 20, 130, 64, 1, "variable", "bf16", None, True, True, True, True, True),
    (2, 48, 190, 16, 1, "variable", "bf16", "fp32", True, True, True, True, True),
    (2, 48, 190, 16, 2, "variable", "fp16", "fp32", False, True, True, True, True),
    (1, 40, 500, 16, 1, "fixed", "fp32", None, False, True, True, True, True),
    (2, 40, 333, 16, 1, "fixed", "bf16", None, True, True, True, True, True),
    (1, 40, 100, 3, 1, "fixed", "fp16", None, True, False, False, True, True),
    (1, 8, 64, 64, 1, "fixed", "fp32", None, True, True, True, True, True),
    (3, 5, 70, 16, 1, "variable", "fp32", None, True, True, True, True, False),
    # more CTAs than the 16-step kernel keeps resident: 8-step hand-offs
    (4, 4096, 200, 16, 4, "variable", "bf16", None, True, True, True, True, True),
    # 2.1 CTAs of 32 channels per SM: 16-channel CTAs spread the work better
    (2, 5120, 256, 16, 1, "variable", "fp16", None, True, True, True, True, True),
]


@pytest.mark.parametrize("case", SWEEP, ids=[f"{c[6]}-{c[5]}-b{c[0]}d{c[1]}l{c[2]}n{c[3]}g{c[4]}" for c in SWEEP])
def test_sweep(case):
    b, d, l, n, g, bc, dt, bcdt, z, D, bias, sp, last = case
    w = workloads.Workload("sweep", b, d, l, n, groups=g, bc=bc, dtype=dt, bc_dtype=bcdt, has_z=z,
                           D_mode="normal" if D else "none", has_bias=bias, delta_softplus=sp,
                           return_last_state=last, bc_4d=g > 1, seed=1000 + l + n)
    x = workloads.make_inputs(w)
    if not sp:  # the raw sum is the step: keep delta + delta_bias a positive step size
        x["delta"] = (x["delta"].float().abs() * 0.05 + 0.01).to(x["delta"].dtype)
        if x["delta_bias"] is not None:
            x["delta_bias"] = torch.full_like(x["delta_bias"], 0.02)
    out, lst = _run(x)
    _check_full(w, x, out, lst)


def test_seqlen_sweep_page_grid():
    """The page's test grid of sequence lengths (128 ... 4096), bf16, grouped."""
    for l in (128, 256, 512, 1024, 2048, 4096):
        w = workloads.Workload("grid", 1, 32, l, 16, groups=2, bc_4d=True, dtype="bf16",
                               return_last_state=True, seed=l)
        x = workloads.make_inputs(w)
        out, last = _run(x)
        _check_full(w, x, out, last)


def test_non_contiguous_views_and_generic_path():
    """u/delta/z/out as strided views (dim stride not a multiple of 8 elements,
    so no TMA descriptor is legal) give the same result as contiguous inputs."""
    w = workloads.Workload("views", 2, 24, 150, 16, dtype="bf16", return_last_state=True, seed=5)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    ref_out, ref_last = _run(x, dev)
    big = {}
    for k in ("u", "delta", "z"):
        t = torch.zeros(2, 24, 157, dtype=dev[k].dtype, device="cuda")
        t[:, :, 3:153] = dev[k]
        big[k] = t[:, :, 3:153]
        assert not big[k].is_contiguous()
    out, last = api.selective_scan_fn(big["u"], big["delta"], dev["A"], dev["B"], dev["C"], dev["D"], big["z"],
                                      dev["delta_bias"], delta_softplus=True, return_last_state=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(last, ref_last)


def test_three_d_and_four_d_bc_agree():
    w = workloads.Workload("bc3", 2, 32, 200, 16, dtype="bf16", seed=8)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    o3 = api.selective_scan_fn(**dev, delta_softplus=True)
    dev4 = dict(dev, B=dev["B"].unsqueeze(1).contiguous(), C=dev["C"].unsqueeze(1).contiguous())
    o4 = api.selective_scan_fn(**dev4, delta_softplus=True)
    assert torch.equal(o3, o4)


def test_host_entry_point_matches_device():
    w = workloads.Workload("host", 2, 48, 300, 16, groups=2, bc_4d=True, dtype="bf16",
                           return_last_state=True, seed=21)
    x = workloads.make_inputs(w)
    out, last = _run(x)
    hx = {k: (None if x[k] is None else x[k].pin_memory()) for k in NAMES}
    r = api.HostRunner(**hx, delta_softplus=True, return_last_state=True)
    for _ in range(2):
        ho, hl = r.run(**hx)
        assert torch.equal(ho, out.cpu()) and torch.equal(hl, last.cpu())


@pytest.mark.parametrize("w", [
    # about 100 MB of inputs: three blocks of whole batch rows
    workloads.Workload("host_batches", 4, 1024, 4096, 16, dtype="bf16", return_last_state=True, seed=22),
    # one batch row: four blocks of 512 channels (fixed B/C, one lane per channel, segments per block)
    workloads.Workload("host_channels", 1, 2048, 8192, 16, bc="fixed", dtype="fp32", has_z=False,
                       bc_std=1.0 / 16, dt_range=(0.001, 0.01), return_last_state=True, seed=23),
    # two batch rows of four groups: channel blocks that keep groups whole
    workloads.Workload("host_groups", 2, 1024, 8192, 16, groups=4, bc_4d=True, dtype="bf16",
                       return_last_state=True, seed=24),
], ids=lambda w: w.name)
def test_host_entry_point_overlapped_blocks(w, monkeypatch):
    """ss_fwd_host cuts large problems into row blocks whose copies overlap the
    kernels of their neighbours; the result matches the device path (and the
    serial single-block schedule) within the tolerance, start state included."""
    x = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 9)
    x0 = torch.randn(w.batch, w.dim, w.dstate, generator=g)
    dev = _to_dev(x)
    ref_out, ref_last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True,
                                              initial_state=x0.cuda())
    torch.cuda.synchronize()
    hx = {k: (None if x[k] is None else x[k].pin_memory()) for k in NAMES}
    tol = TOL[w.dtype]
    for serial in (False, True):
        if serial:
            monkeypatch.setenv("SSFWD_HOST_SERIAL", "1")
        r = api.HostRunner(**hx, delta_softplus=True, return_last_state=True, initial_state=x0.cuda())
        for _ in range(2):
            ho, hl = r.run(**hx)
            assert api.device_error() == 0
            assert float((ho.float() - ref_out.cpu().float()).abs().max()) <= tol * float(ref_out.float().abs().max())
            assert float((hl - ref_last.cpu()).abs().max()) <= tol * float(ref_last.abs().max())


def test_seqlen_zero_and_empty():
    w = workloads.Workload("e", 2, 8, 5, 4, dtype="fp32", return_last_state=True, seed=2)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    for k in ("u", "delta", "z"):
        if dev[k] is not None:
            dev[k] = dev[k][:, :, :0]
    dev["B"] = dev["B"][..., :0]
    dev["C"] = dev["C"][..., :0]
    out, last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True)
    torch.cuda.synchronize()
    assert out.shape == (2, 8, 0) and torch.equal(last, torch.zeros_like(last))
    dev = _to_dev(x)
    for k in ("u", "delta", "z"):
        if dev[k] is not None:
            dev[k] = dev[k][:0]
    dev["B"], dev["C"] = dev["B"][:0], dev["C"][:0]
    out = api.selective_scan_fn(**dev, delta_softplus=True)
    assert out.shape == (0, 8, 5)


def test_errors_raise_and_launch_nothing():
    w = workloads.Workload("err", 1, 12, 16, 4, groups=1, bc_4d=True, dtype="bf16", seed=3)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    bad = dict(dev, B=dev["B"].expand(1, 5, 4, 16).contiguous(), C=dev["C"].expand(1, 5, 4, 16).contiguous())
    with pytest.raises(api.SSError) as ei:
        api.selective_scan_fn(**bad, delta_softplus=True)  # 12 % 5 != 0
    assert ei.value.status == 2
    A65 = torch.zeros(12, 65, device="cuda")
    B65 = torch.zeros(1, 1, 65, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.SSError) as ei:
        api.selective_scan_fn(dev["u"], dev["delta"], A65, B65, B65, delta_softplus=True)
    assert ei.value.status == 7


def test_host_fault_injection(monkeypatch):
    """A failing launch (injected on the host) is reported as SS_ERR_CUDA with
    nothing enqueued; the next call works."""
    w = workloads.Workload("f", 1, 8, 32, 4, dtype="fp32", seed=4)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    monkeypatch.setenv("SSFWD_FAULT", "launch")
    with pytest.raises(api.SSError) as ei:
        api.selective_scan_fn(**dev, delta_softplus=True)
    assert ei.value.status == 8
    monkeypatch.delenv("SSFWD_FAULT")
    api.selective_scan_fn(**dev, delta_softplus=True)
    torch.cuda.synchronize()
    assert api.device_error() == 0


def test_repeatable_bitwise():
    w = workloads.Workload("rep", 2, 64, 512, 16, dtype="bf16", seed=9)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    a = api.selective_scan_fn(**dev, delta_softplus=True)
    b = api.selective_scan_fn(**dev, delta_softplus=True)
    assert torch.equal(a, b)


SEGMENTED = [
    # few channels and long sequences: the sequence is split across CTAs
    (1, 64, 8192, 16, 1, "variable", "bf16", True, True),
    (1, 40, 8000, 16, 1, "fixed", "fp32", False, True),
    (2, 32, 12345, 16, 2, "variable", "fp16", True, True),
    (1, 48, 9000, 5, 1, "variable", "fp32", False, True),
    (1, 24, 8193, 16, 1, "fixed", "bf16", True, False),
]


@pytest.mark.parametrize("case", SEGMENTED, ids=[f"{c[6]}-{c[5]}-b{c[0]}d{c[1]}l{c[2]}n{c[3]}" for c in SEGMENTED])
def test_segmented_sequence(case, monkeypatch):
    """Few (batch, channel) rows and a long sequence: the forward cuts the
    sequence into segments joined through per-segment state summaries. It must
    match the oracle, and the single-pass schedule up to rounding."""
    b, d, l, n, g, bc, dt, z, last = case
    w = workloads.Workload("seg", b, d, l, n, groups=g, bc=bc, dtype=dt, has_z=z, return_last_state=last,
                           bc_4d=g > 1, seed=77 + l, dt_range=(0.001, 0.01) if bc == "fixed" else (0.001, 0.1),
                           bc_std=1.0 / 16 if bc == "fixed" else 1.0)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    nu = api.normalise(*(dev[k] for k in NAMES))
    out = torch.empty(nu[0].shape, dtype=nu[0].dtype, device="cuda")
    lst = torch.empty(b, d, n, device="cuda") if last else None
    p = api.make_params(*nu, True, out, lst)
    ws = api.attach_workspace(p, out.device)
    assert ws is not None and p.workspace_bytes > 0, "expected a segmented schedule"
    import ctypes
    assert api.load_library().ss_fwd(ctypes.byref(p), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert api.device_error() == 0
    _check_full(w, x, out, lst)
    monkeypatch.setenv("SSFWD_NO_SEGMENTS", "1")
    o1, l1 = _run(x, dev)
    scale = float(o1.float().abs().max())
    assert float((out.float() - o1.float()).abs().max()) <= TOL[dt] * scale
    if last:
        assert float((lst - l1).abs().max()) <= TOL[dt] * float(l1.abs().max())


LANE = [
    # fixed B/C, dstate <= 16, TMA-legal rows: the one-lane-per-channel kernel.
    # (batch, dim, seqlen, dstate, dtype, z, D, bias, softplus, last, init, segmented)
    (2, 37, 264, 16, "bf16", True, True, True, True, True, False, False),
    (1, 40, 1000, 13, "fp16", True, False, True, True, True, False, False),
    (3, 32, 96, 4, "fp32", False, True, False, False, True, False, False),
    (1, 64, 8, 8, "bf16", True, True, True, True, True, False, False),
    (2, 33, 4000, 1, "fp32", True, True, True, True, True, False, True),
    (2, 37, 512, 16, "fp32", False, True, True, True, True, True, False),
    (1, 48, 16384, 16, "bf16", True, True, True, True, True, False, True),
    (1, 40, 8000, 13, "bf16", True, True, True, True, True, True, True),
    (1, 32, 10000, 16, "fp16", True, True, True, True, False, False, True),
    (1, 64, 9000, 8, "fp32", False, True, True, True, True, True, True),
]


@pytest.mark.parametrize("case", LANE, ids=[f"{c[4]}-b{c[0]}d{c[1]}l{c[2]}n{c[3]}{'-init' if c[10] else ''}"
                                            f"{'-seg' if c[11] else ''}" for c in LANE])
def test_fixed_bc_one_lane_per_channel(case, capfd, monkeypatch):
    """Fixed B/C with up to 16 states on TMA-legal rows runs the kernel that
    gives each lane a whole channel (the launch report says so); with few
    rows and a long sequence it splits the sequence into segments. Checked
    element by element against the oracle, start states included."""
    b, d, l, n, dt, z, D, bias, sp, last, init, seg = case
    w = workloads.Workload("lane", b, d, l, n, bc="fixed", dtype=dt, has_z=z, D_mode="normal" if D else "none",
                           has_bias=bias, delta_softplus=sp, return_last_state=last, bc_std=0.25,
                           dt_range=(0.001, 0.01) if seg else (0.001, 0.1), seed=2000 + l + n)
    x = workloads.make_inputs(w)
    if not sp:  # the raw sum is the step: keep delta + delta_bias a positive step size
        x["delta"] = (x["delta"].float().abs() * 0.05 + 0.01).to(x["delta"].dtype)
    x0 = None
    if init:
        g = torch.Generator().manual_seed(w.seed + 3)
        x0 = torch.randn(b, d, n, generator=g)
    monkeypatch.setenv("SSFWD_DEBUG", "1")
    dev = _to_dev(x)
    res = api.selective_scan_fn(**dev, delta_softplus=sp, return_last_state=last,
                                initial_state=None if x0 is None else x0.cuda())
    torch.cuda.synchronize()
    assert api.device_error() == 0
    report = capfd.readouterr().err
    assert "ssfwd: lane" in report, report
    nseg = int(report.split("ssfwd: lane")[1].split("grid=")[1].split()[0].split("x")[1])
    assert (nseg > 1) == seg, report
    out, lst = res if last else (res, None)
    ref = oracle.selective_scan_ref(**{k: x[k] for k in NAMES}, delta_softplus=sp, return_last_state=last,
                                    initial_state=x0, threads=8)
    ref_out, ref_last = ref if last else (ref, None)
    o = out.double().cpu().numpy()
    assert np.isfinite(o).all()
    assert _rel(o, ref_out) <= TOL[dt]
    if last:
        assert _rel(lst.double().cpu().numpy(), ref_last) <= TOL[dt]


# (ch, sub, ysum) of the launch report
VARIANT_OF = {("32", "16", "0"): 0, ("32", "8", "0"): 1, ("16", "16", "0"): 2, ("32", "16", "1"): 3}
VARIANT_CASES = [
    # 16 states (all four forward variants exist), ragged channel tiles and
    # steps, two groups; one 16-bit and one fp32 case
    workloads.Workload("variants_bf16", 2, 2 * 80, 296, 16, groups=2, bc_4d=True, dtype="bf16",
                       return_last_state=True, seed=31),
    workloads.Workload("variants_fp32", 1, 48, 200, 13, dtype="fp32", return_last_state=True, seed=33),
]


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("w", VARIANT_CASES, ids=lambda w: w.name)
def test_each_forward_variant(w, variant, monkeypatch, capfd):
    """Every forward variant (0: 32-channel CTAs, 16-step hand-offs; 1: 8-step
    hand-offs; 2: 16-channel CTAs; 3: as 0 with y summed over each channel's
    lanes by the scan warps), forced one at a time, matches the oracle.
    Rows are 16-byte aligned so that the TMA path (which has the variants)
    runs."""
    monkeypatch.setenv("SSFWD_VARIANT", str(variant))
    monkeypatch.setenv("SSFWD_DEBUG", "1")
    x = workloads.make_inputs(w)
    capfd.readouterr()
    out, last = _run(x)
    line = [ln for ln in capfd.readouterr().err.splitlines() if ln.startswith("ssfwd:")][-1]
    f = dict(kv.split("=") for kv in line.split()[2:] if "=" in kv)
    assert line.split()[1] == "tma" and VARIANT_OF[(f["ch"], f["sub"], f["ysum"])] == variant, line
    _check_full(w, x, out, last)


def _picked(capfd, w):
    """Variant the launch picks for workload w (from the SSFWD_DEBUG report)."""
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    capfd.readouterr()
    _run(x, dev)
    err = capfd.readouterr().err
    line = [ln for ln in err.splitlines() if ln.startswith("ssfwd:")][-1]
    f = dict(kv.split("=") for kv in line.split()[2:] if "=" in kv)
    return VARIANT_OF[(f["ch"], f["sub"], f["ysum"])]


def test_variant_choice_follows_waves(capfd, monkeypatch):
    """With 152 SMs: a grid that fits the resident 32-channel CTAs runs variant
    0; one that needs a second wave of them but fits with the smaller y
    hand-off (a fourth CTA per SM) runs variant 3, or variant 1 when variant 3
    is turned off; one that leaves every SM at most two 32-channel CTAs runs
    16-channel CTAs. Sizes are small in seqlen; the choice depends only on the
    grid."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are stated for 152 SMs")
    monkeypatch.setenv("SSFWD_DEBUG", "1")
    mk = lambda b, d, g: workloads.Workload("pick", b, d, 96, 16, groups=g, bc_4d=g > 1, dtype="bf16", seed=5)
    assert _picked(capfd, mk(8, 1536, 1)) == 0   # 384 CTAs <= 3 per SM
    assert _picked(capfd, mk(4, 4096, 4)) == 3   # 512 CTAs: 4 per SM fit with the smaller y hand-off
    assert _picked(capfd, mk(4, 1536, 1)) == 2   # 192 CTAs: at most 2 per SM
    monkeypatch.setenv("SSFWD_NO_YSUM", "1")
    assert _picked(capfd, mk(4, 4096, 4)) == 1   # ... or with 8-step hand-offs
