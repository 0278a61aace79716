"""ss_fwd_noalloc, the allocation-free entry point (collected last on purpose).

Callers that cannot allocate device memory (a runtime that owns every device
allocation and passes in only input and output buffers, or a plugin living
under another framework's allocator) use ss_fwd_noalloc: the same forward,
whose split-sequence scratch comes from a static device buffer inside the
library instead of a caller workspace. These tests call it through the C ABI
on a problem whose schedule does use that scratch, twice in a row, and check
it against ss_fwd with a caller workspace.
"""
import ctypes

import pytest
import torch

from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
TOL = {"fp32": 1e-5, "fp16": 1e-2, "bf16": 1e-2}
MAX_SCRATCH = 2 * 1024 * 1024  # SS_NOALLOC_MAX_SCRATCH


def _problem(w):
    x = workloads.make_inputs(w)
    dev = {k: (None if x[k] is None else x[k].to("cuda")) for k in NAMES}
    nu = api.normalise(*(dev[k] for k in NAMES))
    return x, nu


def _params(nu, w):
    out = torch.full(nu[0].shape, float("nan"), dtype=nu[0].dtype, device="cuda")
    last = torch.full((w.batch, w.dim, w.dstate), float("nan"), device="cuda") if w.return_last_state else None
    return api.make_params(*nu, w.delta_softplus, out, last), out, last


@pytest.mark.parametrize("w", [
    workloads.Workload("na_bf16", 1, 64, 8192, 16, dtype="bf16", return_last_state=True, seed=91),
    workloads.Workload("na_fixed", 1, 40, 8000, 16, bc="fixed", dtype="fp32", has_z=False, bc_std=1.0 / 16,
                       dt_range=(0.001, 0.01), return_last_state=True, seed=92),
], ids=lambda w: w.name)
def test_noalloc_matches_ss_fwd_on_two_calls(w):
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    _, nu = _problem(w)
    p_ref, out_ref, last_ref = _params(nu, w)
    ws = api.attach_workspace(p_ref, out_ref.device)
    assert ws is not None and 0 < p_ref.workspace_bytes <= MAX_SCRATCH  # the schedule uses scratch
    assert lib.ss_fwd(ctypes.byref(p_ref), stream) == 0
    torch.cuda.synchronize()
    tol = TOL[w.dtype]
    for _ in range(2):
        p, out, last = _params(nu, w)  # fresh outputs, no workspace attached
        assert lib.ss_fwd_noalloc(ctypes.byref(p), stream) == 0
        torch.cuda.synchronize()
        assert api.device_error() == 0
        assert torch.isfinite(out.float()).all()
        scale = float(out_ref.float().abs().max())
        assert float((out.float() - out_ref.float()).abs().max()) <= tol * scale
        if last is not None:
            assert float((last - last_ref).abs().max()) <= tol * float(last_ref.abs().max())


def _ref_with_workspace(lib, nu, w, init=None):
    out = torch.empty(nu[0].shape, dtype=nu[0].dtype, device="cuda")
    last = torch.empty((w.batch, w.dim, w.dstate), device="cuda")
    p = api.make_params(*nu, w.delta_softplus, out, last, init)
    ws = api.attach_workspace(p, out.device)
    assert ws is not None and 0 < p.workspace_bytes <= MAX_SCRATCH  # the schedule uses scratch
    assert lib.ss_fwd(ctypes.byref(p), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    return out, last


def test_noalloc_after_a_larger_call_with_padded_states_and_a_start_state():
    """The static buffer keeps the previous call's contents. A larger
    segmented problem fills it first; then a smaller one whose dstate (12, 13)
    is padded to 16 state slots, and a fixed-B/C problem with a start state
    (whose lanes switch from the x / B form to the general update), must each
    match ss_fwd with a caller workspace. The params also carry a stale
    workspace pointer that aliases an input, which ss_fwd_noalloc ignores."""
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    big = workloads.Workload("na_prefill", 1, 128, 16384, 16, dtype="bf16", return_last_state=True, seed=94)
    pad = workloads.Workload("na_pad12", 2, 48, 8192, 12, dtype="fp16", return_last_state=True, seed=95)
    fix = workloads.Workload("na_fixed_init", 1, 40, 8000, 13, bc="fixed", dtype="fp32", has_z=False,
                             bc_std=1.0 / 16, dt_range=(0.001, 0.01), return_last_state=True, seed=96)
    for w in (big, pad, fix):
        _, nu = _problem(w)
        init = None
        if w is fix:
            g = torch.Generator().manual_seed(w.seed + 7)
            init = torch.randn(w.batch, w.dim, w.dstate, generator=g).to("cuda")
        out_ref, last_ref = _ref_with_workspace(lib, nu, w, init)
        out = torch.full(nu[0].shape, float("nan"), dtype=nu[0].dtype, device="cuda")
        last = torch.full((w.batch, w.dim, w.dstate), float("nan"), device="cuda")
        p = api.make_params(*nu, w.delta_softplus, out, last, init)
        p.workspace, p.workspace_bytes = p.u, 64  # stale, aliasing u: ignored
        assert lib.ss_fwd_noalloc(ctypes.byref(p), stream) == 0
        torch.cuda.synchronize()
        assert api.device_error() == 0
        tol = TOL[w.dtype]
        assert float((out.float() - out_ref.float()).abs().max()) <= tol * float(out_ref.float().abs().max())
        assert float((last - last_ref).abs().max()) <= tol * float(last_ref.abs().max())


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A problem whose split-sequence schedule needs more than the static
    buffer is refused with SS_ERR_SCRATCH and nothing is written."""
    lib = api.load_library()
    w = workloads.Workload("na_big", 1, 8192, 4096, 64, dtype="bf16", has_z=False, seed=93)
    _, nu = _problem(w)
    p, out, _ = _params(nu, w)
    need = ctypes.c_int64(0)
    assert lib.ss_fwd_workspace_size(ctypes.byref(p), ctypes.byref(need)) == 0
    assert need.value > MAX_SCRATCH
    assert lib.ss_fwd_noalloc(ctypes.byref(p), torch.cuda.current_stream().cuda_stream) == 11
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
