"""Guard regions around every output of every entry point (the stand-in for a
memory checker on this pool).

Each output tensor is carved out of a larger byte buffer filled with a poison
pattern: a margin before and after it, and (for row-strided outputs) padding
after every row, so the tensor is a strided view with gaps. After the call,
every byte outside the view must still hold the poison, and the view itself
must equal the output of the same call on plainly allocated tensors. The
shapes are ragged on purpose: dim 37 (a partial channel tile), seqlen 1, 7 and
257 (partial chunks and sub-chunks), dstate 3 and 13 (padded state slots),
the TMA producer and the one without tensor maps (odd row lengths: out rows
stored as aligned blocks formed across each row's lanes, clipped at the
segment's ends), out views at odd offsets on every forward variant, the
one-lane-per-channel kernel (whole-row output stores, partial last chunks),
and the split-sequence schedule with its workspace guarded too.
"""
import ctypes

import pytest
import torch

from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

POISON = 0xA5
MARGIN = 4096  # bytes before and after each guarded tensor
NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")


class Guarded:
    """A tensor of `shape` and `dtype` inside a poisoned byte buffer: MARGIN
    bytes on each side and `row_pad` elements after every row of the last
    dimension."""

    def __init__(self, shape, dtype, row_pad=0):
        es = torch.empty((), dtype=dtype).element_size()
        padded = list(shape)
        if padded:
            padded[-1] += row_pad
        n = 1
        for s in padded:
            n *= s
        strides, acc = [], 1
        for s in reversed(padded):
            strides.append(acc)
            acc *= s
        strides = strides[::-1]
        total = 2 * MARGIN + n * es
        total = (total + 15) // 16 * 16
        self.raw = torch.full((total,), POISON, dtype=torch.uint8, device="cuda")
        typed = self.raw.view(dtype)
        self.view = typed.as_strided(shape, strides, MARGIN // es)
        # bytes that belong to the view
        idx = torch.arange(typed.numel(), device="cuda").as_strided(shape, strides, MARGIN // es).reshape(-1)
        self.mask = torch.zeros(total, dtype=torch.bool, device="cuda")
        for k in range(es):
            self.mask[idx * es + k] = True

    def untouched(self) -> bool:
        return bool((self.raw[~self.mask] == POISON).all())


def _inputs(w):
    x = workloads.make_inputs(w)
    dev = {k: (None if x[k] is None else x[k].to("cuda")) for k in NAMES}
    return api.normalise(*(dev[k] for k in NAMES))


def _close(a, b, tol):
    a, b = a.float(), b.float()
    den = float(b.abs().max()) if b.numel() else 0.0
    return float((a - b).abs().max()) <= tol * max(den, 1e-30) if b.numel() else True


W = workloads.Workload
FWD_CASES = [
    # (workload, out row pad, last_state row pad); pads that keep 16-byte rows exercise vector stores
    (W("g_bf16_d37_l257_n13", 2, 37, 257, 13, dtype="bf16", return_last_state=True, seed=301), 3, 2),
    (W("g_bf16_d37_l264_tma", 2, 37, 264, 13, groups=1, bc_4d=True, dtype="bf16", return_last_state=True,
       seed=302), 8, 1),
    (W("g_fp32_l1_n3", 3, 37, 1, 3, dtype="fp32", return_last_state=True, seed=303), 1, 5),
    (W("g_fp16_l7_n13", 2, 37, 7, 13, dtype="fp16", return_last_state=True, seed=304), 0, 0),
    (W("g_fp32_fixed_l257", 2, 37, 257, 13, bc="fixed", dtype="fp32", has_z=False, bc_std=0.25,
       return_last_state=True, seed=305), 4, 3),
    (W("g_grouped_bf16", 2, 74, 200, 16, groups=2, bc_4d=True, dtype="bf16", return_last_state=True,
       seed=306), 8, 0),
    # fixed B/C on TMA-legal rows: the one-lane-per-channel kernel, whose outputs leave as whole rows
    # of a chunk; a partial last chunk (264 = 4 x 64 + 8, 260 = 8 x 32 + 4) and a partial channel tile
    (W("g_lane_bf16_l264", 2, 37, 264, 13, bc="fixed", dtype="bf16", bc_std=0.25, return_last_state=True,
       seed=309), 8, 2),
    (W("g_lane_fp32_l260", 2, 37, 260, 13, bc="fixed", dtype="fp32", has_z=False, bc_std=0.25,
       return_last_state=True, seed=310), 4, 3),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: c[0].name)
def test_forward_writes_nothing_outside_its_outputs(case):
    w, opad, lpad = case
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    nu = _inputs(w)
    u = nu[0]
    ref_out = torch.empty(u.shape, dtype=u.dtype, device="cuda")
    ref_last = torch.empty((w.batch, w.dim, w.dstate), device="cuda")
    p = api.make_params(*nu, w.delta_softplus, ref_out, ref_last)
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0
    go = Guarded(tuple(u.shape), u.dtype, opad)
    gl = Guarded((w.batch, w.dim, w.dstate), torch.float32, lpad)
    p = api.make_params(*nu, w.delta_softplus, go.view, gl.view)
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    assert api.device_error() == 0
    assert go.untouched() and gl.untouched()
    assert torch.equal(go.view, ref_out) and torch.equal(gl.view, ref_last)


def _guarded_matches_plain(w, opad, lpad, segmented=False):
    """Run w into plainly allocated outputs and into guarded ones (out rows
    padded by opad elements, last_state rows by lpad): margins untouched, the
    same bits."""
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    nu = _inputs(w)
    u = nu[0]
    ref_out = torch.empty(u.shape, dtype=u.dtype, device="cuda")
    ref_last = torch.empty((w.batch, w.dim, w.dstate), device="cuda")
    p = api.make_params(*nu, w.delta_softplus, ref_out, ref_last)
    ws = api.attach_workspace(p, u.device)
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0
    go = Guarded(tuple(u.shape), u.dtype, opad)
    gl = Guarded((w.batch, w.dim, w.dstate), torch.float32, lpad)
    p = api.make_params(*nu, w.delta_softplus, go.view, gl.view)
    ws2 = api.attach_workspace(p, u.device)
    assert (ws2 is not None) or not segmented  # the schedule is split when asked
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    del ws, ws2
    assert api.device_error() == 0
    assert go.untouched() and gl.untouched()
    assert torch.equal(go.view, ref_out) and torch.equal(gl.view, ref_last)


@pytest.mark.parametrize("opad", [1, 3])
@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_unaligned_out_rows_on_every_forward_variant(variant, opad, monkeypatch):
    """Inputs TMA can describe, out rows that are not 16-byte aligned (296 + 1
    or + 3 elements a row; ragged channel tiles, two groups): every forced
    variant writes exactly out's bytes (element by element)."""
    monkeypatch.setenv("SSFWD_VARIANT", str(variant))
    _guarded_matches_plain(W("g_uout_bf16", 2, 2 * 40, 296, 16, groups=2, bc_4d=True, dtype="bf16",
                             return_last_state=True, seed=313), opad, 1)


@pytest.mark.parametrize("w", [
    W("g_uout_seg_bf16", 1, 37, 8192, 16, dtype="bf16", return_last_state=True, seed=314),
    W("g_uout_seg_fp32", 1, 40, 6000, 16, dtype="fp32", has_z=False, return_last_state=True, seed=315),
    W("g_uout_seg_bf16_odd", 1, 37, 8191, 16, dtype="bf16", return_last_state=True, seed=316),
    W("g_uout_seg_fp32_odd", 1, 40, 6001, 16, dtype="fp32", has_z=False, return_last_state=True, seed=317),
], ids=lambda w: w.name)
def test_unaligned_out_rows_on_the_split_sequence_schedule(w):
    """Segments that start and end inside out's 16-byte blocks: each CTA
    writes only its own steps, so neighbouring segments do not overwrite each
    other's bytes (the instance without tensor maps, whose aligned blocks are
    clipped at the segment's ends, runs the odd-length case below)."""
    _guarded_matches_plain(w, 3, 2, segmented=True)


@pytest.mark.parametrize("w", [
    W("g_seg_fixed", 1, 40, 8000, 13, bc="fixed", dtype="fp32", has_z=False, bc_std=1.0 / 16,
      dt_range=(0.001, 0.01), return_last_state=True, seed=307),
    W("g_seg_bf16", 1, 37, 8192, 16, dtype="bf16", return_last_state=True, seed=308),
], ids=lambda w: w.name)
def test_split_sequence_schedule_stays_inside_its_workspace(w):
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    nu = _inputs(w)
    u = nu[0]
    go = Guarded(tuple(u.shape), u.dtype, 8)
    gl = Guarded((w.batch, w.dim, w.dstate), torch.float32, 3)
    p = api.make_params(*nu, w.delta_softplus, go.view, gl.view)
    need = ctypes.c_int64(0)
    assert lib.ss_fwd_workspace_size(ctypes.byref(p), ctypes.byref(need)) == 0
    assert need.value > 0  # the schedule is segmented
    gw = Guarded((need.value,), torch.uint8)
    p.workspace, p.workspace_bytes = gw.view.data_ptr(), need.value
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    assert api.device_error() == 0
    assert go.untouched() and gl.untouched() and gw.untouched()
    ref_out, ref_last = api.selective_scan_fn(*nu[:5], D=nu[5], z=nu[6], delta_bias=nu[7],
                                              delta_softplus=w.delta_softplus, return_last_state=True)
    tol = 1e-5 if w.dtype == "fp32" else 1e-2
    assert _close(go.view, ref_out, tol) and _close(gl.view, ref_last, tol)


@pytest.mark.parametrize("w", [
    W("gb_bf16_d37_l257_n13", 2, 37, 257, 13, dtype="bf16", seed=311),
    W("gb_fp32_fixed_l7_n3", 2, 37, 7, 3, bc="fixed", dtype="fp32", bc_std=0.25, seed=312),
], ids=lambda w: w.name)
def test_backward_writes_nothing_outside_its_outputs(w):
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    u, delta, A, B, C, D, z, bias = _inputs(w)
    dout = workloads.make_dout(w).to("cuda")
    g = torch.Generator().manual_seed(w.seed + 5)
    init = torch.randn(w.batch, w.dim, w.dstate, generator=g).to("cuda")
    shape3 = tuple(u.shape)
    gdu, gdd = Guarded(shape3, u.dtype, 3), Guarded(shape3, u.dtype, 1)
    gdz = Guarded(shape3, u.dtype, 5) if z is not None else None
    gA = Guarded((w.dim, w.dstate), torch.float32)
    gB, gC = Guarded(tuple(B.shape), torch.float32), Guarded(tuple(C.shape), torch.float32)
    gD, gbias = Guarded((w.dim,), torch.float32), Guarded((w.dim,), torch.float32)
    ginit = Guarded((w.batch, w.dim, w.dstate), torch.float32)
    p = api.make_bwd_params(dout, u, delta, A, B, C, D, z, bias, w.delta_softplus, init,
                            gdu.view, gdd.view, None if gdz is None else gdz.view, gA.view, gB.view, gC.view,
                            gD.view, gbias.view, ginit.view)
    need = ctypes.c_int64(0)
    assert lib.ss_bwd_workspace_size(ctypes.byref(p), ctypes.byref(need)) == 0
    gw = Guarded((max(need.value, 16),), torch.uint8)
    p.workspace, p.workspace_bytes = gw.view.data_ptr(), need.value
    assert lib.ss_bwd(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    guards = [gdu, gdd, gA, gB, gC, gD, gbias, ginit, gw] + ([gdz] if gdz is not None else [])
    assert all(gg.untouched() for gg in guards)
    ref = api.selective_scan_bwd(dout, u, delta, A, B, C, D=D, z=z, delta_bias=bias,
                                 delta_softplus=w.delta_softplus, initial_state=init,
                                 want_dD=True, want_ddelta_bias=True, want_dinitial_state=True)
    tol = 1e-5 if w.dtype == "fp32" else 1e-2
    pairs = [(gdu, "du"), (gdd, "ddelta"), (gA, "dA"), (gD, "dD"), (gbias, "ddelta_bias"),
             (ginit, "dinitial_state")] + ([(gdz, "dz")] if gdz is not None else [])
    for gg, k in pairs:
        assert _close(gg.view, ref[k], tol), k
    assert _close(gB.view, ref["dB"].reshape(gB.view.shape), tol)
    assert _close(gC.view, ref["dC"].reshape(gC.view.shape), tol)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step_writes_nothing_outside_its_outputs(dtype):
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    g = torch.Generator().manual_seed(321)
    batch, dim, n = 3, 37, 13
    u = torch.randn(batch, dim, generator=g).to(dtype).cuda()
    delta = torch.randn(batch, dim, generator=g).to(dtype).cuda()
    z = torch.randn(batch, dim, generator=g).to(dtype).cuda()
    A = -(torch.rand(dim, n, generator=g) + 0.5).cuda()
    B = torch.randn(batch, n, generator=g).to(dtype).cuda()
    C = torch.randn(batch, n, generator=g).to(dtype).cuda()
    D = torch.randn(dim, generator=g).cuda()
    bias = torch.randn(dim, generator=g).cuda()
    s0 = torch.randn(batch, dim, n, generator=g).cuda()
    gs = Guarded((batch, dim, n), torch.float32, 3)
    gs.view.copy_(s0)
    go = Guarded((batch, dim), dtype, 5)
    p = api.make_state_update_params(gs.view, u, delta, A, B, C, D, z, bias, True, go.view)
    assert lib.ss_state_update(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    assert gs.untouched() and go.untouched()
    ref_state = s0.clone()
    ref_out = api.selective_state_update(ref_state, u, delta, A, B, C, D=D, z=z, delta_bias=bias,
                                         delta_softplus=True)
    assert torch.equal(gs.view, ref_state) and torch.equal(go.view, ref_out)


@pytest.mark.parametrize("seqlen", [1, 7, 257])
def test_conv1d_writes_nothing_outside_its_outputs(seqlen):
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    g = torch.Generator().manual_seed(331 + seqlen)
    batch, dim, width = 2, 37, 4
    x = torch.randn(batch, dim, seqlen, generator=g).to(torch.bfloat16).cuda()
    weight = torch.randn(dim, width, generator=g).cuda()
    bias = torch.randn(dim, generator=g).cuda()
    init = torch.randn(batch, dim, width - 1, generator=g).to(torch.bfloat16).cuda()
    go = Guarded((batch, dim, seqlen), torch.bfloat16, 3)
    gf = Guarded((batch, dim, width - 1), torch.bfloat16, 2)
    p = api.make_conv1d_params(x, weight, bias, None, init, gf.view, go.view, "silu")
    assert lib.ss_causal_conv1d(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    assert go.untouched() and gf.untouched()
    ref_out, ref_fin = api.causal_conv1d_fn(x, weight, bias, initial_states=init, return_final_states=True,
                                            activation="silu")
    assert torch.equal(go.view, ref_out) and torch.equal(gf.view, ref_fin)
    # the one-step update: its state is updated in place inside the guarded buffer
    xs = torch.randn(batch, dim, generator=g).to(torch.bfloat16).cuda()
    gs = Guarded((batch, dim, width - 1), torch.bfloat16, 1)
    gs.view.copy_(init)
    ref_state = init.clone()
    ref_step = api.causal_conv1d_update(xs, ref_state, weight, bias, activation="silu")
    step = api.causal_conv1d_update(xs, gs.view, weight, bias, activation="silu")
    torch.cuda.synchronize()
    assert gs.untouched()
    assert torch.equal(gs.view, ref_state) and torch.equal(step, ref_step)


def test_complex_forward_writes_nothing_outside_its_outputs():
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    w = W("g_cx_d37_l257_n13", 2, 37, 257, 13, dtype="bf16", return_last_state=True, seed=341)
    x = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed)
    x["A"] = torch.complex(-(torch.rand(w.dim, w.dstate, generator=g) + 0.2),
                           torch.rand(w.dim, w.dstate, generator=g) * 6 - 3)
    dev = {k: (None if x[k] is None else x[k].to("cuda")) for k in NAMES}
    nu = api.normalise(*(dev[k] for k in NAMES))
    ref_out, ref_last = api.selective_scan_fn(*nu[:5], D=nu[5], z=nu[6], delta_bias=nu[7],
                                              delta_softplus=True, return_last_state=True)
    go = Guarded(tuple(nu[0].shape), nu[0].dtype, 3)
    gl = Guarded((w.batch, w.dim, w.dstate), torch.complex64, 2)
    p = api.make_complex_params(*nu, True, go.view, gl.view)
    assert lib.ss_fwd_complex(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    assert go.untouched() and gl.untouched()
    assert torch.equal(go.view, ref_out) and torch.equal(gl.view, ref_last)
