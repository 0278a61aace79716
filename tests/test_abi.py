"""C ABI checks that need no GPU: the library loads, exports every function
include/ssfwd.h declares, and its validation returns the documented status
for each malformed call without launching anything (ss_fwd_validate makes no
CUDA call, and ss_fwd returns before its first CUDA call on these inputs)."""
import ctypes
import os
import re

import pytest

from state_space_model_03_gb300 import api
from state_space_model_03_gb300 import build as ssbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssfwd.h")


@pytest.fixture(scope="module")
def lib():
    ssbuild.build()
    return api.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) == {"ss_abi_version", "ss_status_string", "ss_fwd_validate", "ss_fwd",
                          "ss_fwd_host", "ss_device_error", "ss_fwd_workspace_size", "ss_fwd_noalloc",
                          "ss_state_update_validate", "ss_state_update", "ss_causal_conv1d_validate",
                          "ss_causal_conv1d", "ss_causal_conv1d_update_validate", "ss_causal_conv1d_update",
                          "ss_bwd_validate", "ss_bwd_workspace_size", "ss_bwd",
                          "ss_fwd_complex_validate", "ss_fwd_complex"}
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_strings(lib):
    assert lib.ss_abi_version() == api.SS_ABI_VERSION
    for s in range(0, 12):
        assert api.status_string(s) and api.status_string(s) != "unknown status"
    assert api.status_string(99) == "unknown status"


def _good():
    """A valid variable-B/C bf16 problem with fake (never dereferenced) device
    addresses, laid out contiguously and 16-byte aligned."""
    b, d, l, n, g = 2, 64, 128, 16, 2
    p = api.SSFwdParams()
    p.abi_version = api.SS_ABI_VERSION
    p.in_dtype = p.bc_dtype = api.SS_BF16
    p.bc_mode = api.SS_BC_VARIABLE
    p.delta_softplus = 1
    p.batch, p.dim, p.seqlen, p.dstate, p.ngroups = b, d, l, n, g
    base = 1 << 40
    sz3 = b * d * l * 2
    addrs = {}
    cur = base
    for k, nbytes in (("u", sz3), ("delta", sz3), ("z", sz3), ("B", b * g * n * l * 2), ("C", b * g * n * l * 2),
                      ("A", d * n * 4), ("D", d * 4), ("delta_bias", d * 4), ("out", sz3), ("last_state", b * d * n * 4)):
        addrs[k] = cur
        cur += (nbytes + 255) // 256 * 256
    for k, v in addrs.items():
        setattr(p, k, v)
    for k in ("u_stride", "delta_stride", "z_stride", "out_stride"):
        getattr(p, k)[:] = [d * l, l, 1]
    p.B_stride[:] = [g * n * l, n * l, l, 1]
    p.C_stride[:] = [g * n * l, n * l, l, 1]
    p.A_stride[:] = [n, 1]
    p.last_state_stride[:] = [d * n, n, 1]
    return p


def _val(lib, p):
    return lib.ss_fwd_validate(ctypes.byref(p)) if p is not None else lib.ss_fwd_validate(None)


def test_valid_params_pass(lib):
    assert _val(lib, _good()) == 0


@pytest.mark.parametrize("mutate,status", [
    (lambda p: setattr(p, "abi_version", 0), 10),
    (lambda p: setattr(p, "u", None), 1),
    (lambda p: setattr(p, "out", None), 1),
    (lambda p: setattr(p, "B", None), 1),
    (lambda p: setattr(p, "in_dtype", 7), 3),
    (lambda p: setattr(p, "bc_dtype", api.SS_F16), 3),        # bf16 inputs, fp16 B/C
    (lambda p: setattr(p, "ngroups", 3), 2),                  # 64 % 3 != 0
    (lambda p: setattr(p, "ngroups", 0), 2),
    (lambda p: setattr(p, "dstate", 0), 2),
    (lambda p: setattr(p, "dstate", 65), 7),
    (lambda p: setattr(p, "seqlen", -1), 2),
    (lambda p: setattr(p, "batch", 70000), 7),
    (lambda p: p.u_stride.__setitem__(2, 2), 4),
    (lambda p: p.out_stride.__setitem__(2, 2), 4),
    (lambda p: p.B_stride.__setitem__(3, 2), 4),
    (lambda p: p.A_stride.__setitem__(1, 2), 4),
    (lambda p: p.delta_stride.__setitem__(0, -5), 4),
    (lambda p: p.last_state_stride.__setitem__(2, 3), 4),
    (lambda p: setattr(p, "u", p.u + 1), 5),                  # bf16 needs 2-byte alignment
    (lambda p: setattr(p, "A", p.A + 2), 5),
    (lambda p: setattr(p, "out", p.u), 6),                    # out aliases u
    (lambda p: setattr(p, "out", p.z + 64), 6),               # partial overlap with z
    (lambda p: setattr(p, "last_state", p.A), 6),
    (lambda p: setattr(p, "last_state", p.out + 128), 6),
    (lambda p: setattr(p, "workspace_bytes", -1), 2),
    (lambda p: (setattr(p, "workspace", p.u + 64), setattr(p, "workspace_bytes", 256)), 6),
    (lambda p: setattr(p, "error_word", p.u + 2), 5),         # the error word needs 4-byte alignment
    (lambda p: setattr(p, "error_word", p.out + 64), 6),      # ... and must not alias an output
    (lambda p: setattr(p, "error_word", p.A), 6),             # ... or an input
    (lambda p: (setattr(p, "workspace", p.last_state + (1 << 20)), setattr(p, "workspace_bytes", 256),
                setattr(p, "error_word", p.last_state + (1 << 20) + 16)), 6),  # ... or the workspace
])
def test_invalid_params_rejected(lib, mutate, status):
    p = _good()
    mutate(p)
    assert _val(lib, p) == status
    # ss_fwd validates first and returns the same status with nothing launched
    assert lib.ss_fwd(ctypes.byref(p), None) == status


def test_caller_error_word_accepted(lib):
    p = _good()
    p.error_word = p.last_state + (1 << 20)  # a word of its own, clear of every tensor
    assert _val(lib, p) == 0


def test_noalloc_ignores_the_workspace_fields(lib, monkeypatch):
    """ss_fwd_noalloc neither uses nor validates p->workspace: a stale pointer
    that would alias an input under ss_fwd is no error there. The addresses
    are fake, so the host fault hook stops the call before any launch (on a
    machine with or without a GPU); the status is then SS_ERR_CUDA, not the
    alias or shape error a checked workspace would give."""
    monkeypatch.setenv("SSFWD_FAULT", "launch")
    p = _good()
    p.workspace, p.workspace_bytes = p.u + 64, 256
    assert _val(lib, p) == 6
    assert lib.ss_fwd_noalloc(ctypes.byref(p), None) == 8
    p.workspace_bytes = -1
    assert lib.ss_fwd_noalloc(ctypes.byref(p), None) == 8
    p.abi_version = 0
    assert lib.ss_fwd_noalloc(ctypes.byref(p), None) == 10
    assert lib.ss_fwd_noalloc(None, None) == 1


def test_null_params(lib):
    assert _val(lib, None) == 1
    assert lib.ss_fwd(None, None) == 1


def test_fixed_bc_rules(lib):
    p = _good()
    p.bc_mode = api.SS_BC_FIXED
    p.bc_dtype = api.SS_F32
    p.B_stride[:] = [16, 1, 0, 0]
    p.C_stride[:] = [16, 1, 0, 0]
    p.ngroups = 3  # ignored for fixed B/C
    assert _val(lib, p) == 0
    p.bc_dtype = api.SS_BF16
    assert _val(lib, p) == 3
    p.bc_dtype = api.SS_F32
    p.B_stride[1] = 2
    assert _val(lib, p) == 4


def test_empty_problems_validate(lib):
    p = _good()
    p.batch = 0
    assert _val(lib, p) == 0
    p = _good()
    p.seqlen = 0
    p.u = p.delta = p.out = None  # nothing is read or written but last_state
    assert _val(lib, p) == 0


def test_python_wrapper_refuses_cpu_tensors():
    import torch
    u = torch.zeros(1, 4, 8)
    with pytest.raises(RuntimeError):
        api.selective_scan_fn(u, u, torch.zeros(4, 4), torch.zeros(1, 4, 8), torch.zeros(1, 4, 8))


def test_python_entry_points_refuse_cpu_tensors():
    """The backward and the complex-A forward have no CPU path either."""
    import torch
    u = torch.zeros(1, 4, 8)
    bc = torch.zeros(1, 4, 8)
    with pytest.raises(RuntimeError):
        api.selective_scan_bwd(u, u, u, torch.zeros(4, 4), bc, bc)
    with pytest.raises(RuntimeError):
        api.selective_scan_fn(u, u, torch.zeros(4, 4, dtype=torch.complex64), bc, bc)


def test_bwd_and_complex_param_fillers_check_operands():
    """make_bwd_params / make_complex_params read shapes, dtypes and strides
    only (no device access), and reject mismatched operands."""
    import torch
    b, d, l, n = 2, 8, 16, 4
    u = torch.zeros(b, d, l)
    A = torch.zeros(d, n)
    B = torch.zeros(b, 1, n, l)
    f32 = lambda *s: torch.zeros(*s)
    args = dict(dout=u, u=u, delta=u, A=A, B=B, C=B, D=None, z=None, delta_bias=None, delta_softplus=True,
                initial_state=None, du=torch.zeros_like(u), ddelta=torch.zeros_like(u), dz=None, dA=f32(d, n),
                dB=f32(b, 1, n, l), dC=f32(b, 1, n, l), dD=None, ddelta_bias=None, dinitial_state=None)
    p = api.make_bwd_params(**args)
    assert (p.batch, p.dim, p.seqlen, p.dstate, p.ngroups) == (b, d, l, n, 1)
    assert list(p.dout_stride) == [d * l, l, 1] and p.in_dtype == api.SS_F32
    with pytest.raises(TypeError):
        api.make_bwd_params(**dict(args, dout=u.half()))
    with pytest.raises(TypeError):
        api.make_bwd_params(**dict(args, du=torch.zeros(b, d, l + 1)))
    Ac = torch.zeros(d, n, dtype=torch.complex64)
    out = torch.zeros_like(u)
    last = torch.zeros(b, d, n, dtype=torch.complex64)
    q = api.make_complex_params(u, u, Ac, B, B, None, None, None, True, out, last)
    assert list(q.A_stride) == [n, 1] and list(q.last_state_stride) == [d * n, n, 1]
    with pytest.raises(TypeError):
        api.make_complex_params(u, u, A, B, B, None, None, None, True, out, None)          # real A
    with pytest.raises(TypeError):
        api.make_complex_params(u, u, Ac, B, B, None, None, None, True, out, last.real)    # real state


def test_complex_A_normalised_to_complex64():
    import torch
    u = torch.zeros(1, 4, 8)
    A = api.normalise(u, u, torch.zeros(4, 4, dtype=torch.complex128), torch.zeros(1, 4, 8), torch.zeros(1, 4, 8))[2]
    assert A.dtype == torch.complex64


def test_initial_state_rules(lib):
    """The forward's optional start state: state stride 1, 4-byte alignment, and
    no overlap with out or (unless it is the very same buffer) last_state."""
    p = _good()
    base = p.out + (1 << 20)
    p.initial_state = base
    p.initial_state_stride[:] = [64 * 16, 16, 1]
    assert _val(lib, p) == 0
    p.initial_state_stride[2] = 2
    assert _val(lib, p) == 4
    p.initial_state_stride[:] = [64 * 16, 16, 1]
    p.initial_state = base + 2
    assert _val(lib, p) == 5
    p.initial_state = p.out
    assert _val(lib, p) == 6                                  # overlaps out
    p.initial_state = p.last_state                            # in place: allowed
    p.initial_state_stride[:] = list(p.last_state_stride)
    assert _val(lib, p) == 0
    p.initial_state = p.last_state + 64                       # partial overlap with last_state
    assert _val(lib, p) == 6


def _good_su():
    """A valid decode-step problem with fake (never dereferenced) addresses."""
    b, d, n, g = 4, 64, 16, 2
    p = api.SSStateUpdateParams()
    p.abi_version = api.SS_ABI_VERSION
    p.in_dtype = p.bc_dtype = api.SS_BF16
    p.bc_mode = api.SS_BC_VARIABLE
    p.delta_softplus = 1
    p.batch, p.dim, p.dstate, p.ngroups = b, d, n, g
    cur = 1 << 40
    addrs = {}
    for k, nbytes in (("state", b * d * n * 4), ("u", b * d * 2), ("delta", b * d * 2), ("z", b * d * 2),
                      ("B", b * g * n * 2), ("C", b * g * n * 2), ("A", d * n * 4), ("D", d * 4),
                      ("delta_bias", d * 4), ("out", b * d * 2)):
        addrs[k] = cur
        cur += (nbytes + 255) // 256 * 256
    for k, v in addrs.items():
        setattr(p, k, v)
    p.state_stride[:] = [d * n, n, 1]
    for k in ("u_stride", "delta_stride", "z_stride", "out_stride"):
        getattr(p, k)[:] = [d, 1]
    p.B_stride[:] = [g * n, n, 1]
    p.C_stride[:] = [g * n, n, 1]
    p.A_stride[:] = [n, 1]
    return p


@pytest.mark.parametrize("mutate,status", [
    (lambda p: None, 0),
    (lambda p: setattr(p, "abi_version", 2), 10),
    (lambda p: setattr(p, "state", None), 1),
    (lambda p: setattr(p, "out", None), 1),
    (lambda p: setattr(p, "in_dtype", 5), 3),
    (lambda p: setattr(p, "bc_dtype", api.SS_F16), 3),
    (lambda p: setattr(p, "ngroups", 3), 2),
    (lambda p: setattr(p, "dstate", 0), 2),
    (lambda p: setattr(p, "dstate", 65), 7),
    (lambda p: p.state_stride.__setitem__(2, 2), 4),
    (lambda p: p.B_stride.__setitem__(2, 2), 4),
    (lambda p: p.u_stride.__setitem__(0, -1), 4),
    (lambda p: setattr(p, "state", p.state + 2), 5),
    (lambda p: setattr(p, "out", p.u), 6),                    # out aliases an input
    (lambda p: setattr(p, "out", p.state + 64), 6),           # out inside the state
    (lambda p: setattr(p, "state", p.A), 6),                  # state aliases an input
    (lambda p: setattr(p, "batch", 0), 0),                    # empty: no-op
])
def test_state_update_validation(lib, mutate, status):
    p = _good_su()
    mutate(p)
    assert lib.ss_state_update_validate(ctypes.byref(p)) == status
    if status != 0:
        assert lib.ss_state_update(ctypes.byref(p), None) == status


def test_state_update_fixed_bc_rules(lib):
    p = _good_su()
    p.bc_mode = api.SS_BC_FIXED
    p.bc_dtype = api.SS_F32
    p.B_stride[:] = [16, 1, 0]
    p.C_stride[:] = [16, 1, 0]
    assert lib.ss_state_update_validate(ctypes.byref(p)) == 0
    p.bc_dtype = api.SS_BF16
    assert lib.ss_state_update_validate(ctypes.byref(p)) == 3


def _good_conv():
    b, d, l, w = 2, 64, 128, 4
    p = api.SSConv1dParams()
    p.abi_version = api.SS_ABI_VERSION
    p.dtype = api.SS_BF16
    p.activation = api.SS_ACT_SILU
    p.batch, p.dim, p.seqlen, p.width = b, d, l, w
    cur = 1 << 40
    for k, nbytes in (("x", b * d * l * 2), ("weight", d * w * 4), ("bias", d * 4), ("out", b * d * l * 2)):
        setattr(p, k, cur)
        cur += (nbytes + 255) // 256 * 256
    p.x_stride[:] = [d * l, l, 1]
    p.out_stride[:] = [d * l, l, 1]
    p.weight_stride[:] = [w, 1]
    return p, cur


@pytest.mark.parametrize("mutate,status", [
    (lambda p, c: None, 0),
    (lambda p, c: setattr(p, "width", 5), 7),
    (lambda p, c: setattr(p, "width", 1), 7),
    (lambda p, c: setattr(p, "activation", 2), 7),
    (lambda p, c: setattr(p, "dtype", 9), 3),
    (lambda p, c: setattr(p, "x", None), 1),
    (lambda p, c: p.x_stride.__setitem__(2, 2), 4),
    (lambda p, c: setattr(p, "out", p.x), 6),
    (lambda p, c: setattr(p, "out", p.x + 2), 6),
    (lambda p, c: setattr(p, "x", p.x + 1), 5),
    (lambda p, c: (setattr(p, "seq_idx", c), setattr(p, "final_states", c + 4096),
                   p.seq_idx_stride.__setitem__(slice(0, 2), [128, 1]),
                   p.final_states_stride.__setitem__(slice(0, 3), [192, 3, 1])), 7),
    (lambda p, c: (setattr(p, "final_states", p.weight),
                   p.final_states_stride.__setitem__(slice(0, 3), [192, 3, 1])), 6),
    (lambda p, c: setattr(p, "seqlen", -1), 2),
])
def test_conv1d_validation(lib, mutate, status):
    p, cur = _good_conv()
    mutate(p, cur)
    assert lib.ss_causal_conv1d_validate(ctypes.byref(p)) == status
    if status != 0:
        assert lib.ss_causal_conv1d(ctypes.byref(p), None) == status


def test_conv1d_update_validation(lib):
    p = api.SSConv1dUpdateParams()
    p.abi_version = api.SS_ABI_VERSION
    p.dtype = api.SS_F32
    p.batch, p.dim, p.width = 2, 16, 3
    base = 1 << 40
    p.x, p.conv_state, p.weight, p.out = base, base + 4096, base + 8192, base + 12288
    p.x_stride[:] = [16, 1]
    p.conv_state_stride[:] = [32, 2, 1]
    p.weight_stride[:] = [3, 1]
    p.out_stride[:] = [16, 1]
    assert lib.ss_causal_conv1d_update_validate(ctypes.byref(p)) == 0
    p.out = p.conv_state
    assert lib.ss_causal_conv1d_update_validate(ctypes.byref(p)) == 6
    p.out = base + 12288
    p.width = 6
    assert lib.ss_causal_conv1d_update_validate(ctypes.byref(p)) == 7


# ---------------------------------------------------------------------------
# backward (ss_bwd): validation only (no launch on the CPU)
# ---------------------------------------------------------------------------
def _good_bwd(with_ws=True):
    """A valid variable-B/C bf16 backward with fake (never dereferenced)
    device addresses, contiguous and 256-byte aligned."""
    b, d, l, n, g = 2, 64, 300, 16, 2
    p = api.SSBwdParams()
    p.abi_version = api.SS_ABI_VERSION
    p.in_dtype = p.bc_dtype = api.SS_BF16
    p.bc_mode = api.SS_BC_VARIABLE
    p.delta_softplus = 1
    p.batch, p.dim, p.seqlen, p.dstate, p.ngroups = b, d, l, n, g
    sz3, szb = b * d * l * 2, b * g * n * l
    cur = 1 << 40
    for k, nbytes in (("u", sz3), ("delta", sz3), ("z", sz3), ("dout", sz3), ("B", szb * 2), ("C", szb * 2),
                      ("A", d * n * 4), ("D", d * 4), ("delta_bias", d * 4), ("initial_state", b * d * n * 4),
                      ("du", sz3), ("ddelta", sz3), ("dz", sz3), ("dA", d * n * 4), ("dB", szb * 4),
                      ("dC", szb * 4), ("dD", d * 4), ("ddelta_bias", d * 4), ("dinitial_state", b * d * n * 4)):
        setattr(p, k, cur)
        cur += (nbytes + 255) // 256 * 256
    for k in ("u_stride", "delta_stride", "z_stride", "dout_stride", "du_stride", "ddelta_stride", "dz_stride"):
        getattr(p, k)[:] = [d * l, l, 1]
    p.B_stride[:] = [g * n * l, n * l, l, 1]
    p.C_stride[:] = [g * n * l, n * l, l, 1]
    p.A_stride[:] = [n, 1]
    p.initial_state_stride[:] = [d * n, n, 1]
    if with_ws:
        need = ctypes.c_int64(0)
        assert api.load_library().ss_bwd_workspace_size(ctypes.byref(p), ctypes.byref(need)) == 0
        p.workspace, p.workspace_bytes = cur, need.value
    return p


def test_bwd_workspace_size(lib):
    p = _good_bwd(with_ws=False)
    n = ctypes.c_int64(-1)
    assert lib.ss_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    # one fp32 state per (batch, channel, state) and checkpoint interval of the row
    assert n.value > 0 and n.value % (2 * 64 * 16 * 4) == 0
    assert lib.ss_bwd_workspace_size(ctypes.byref(p), None) == 1
    assert lib.ss_bwd_validate(ctypes.byref(p)) == 11  # no workspace: SS_ERR_SCRATCH
    assert lib.ss_bwd(ctypes.byref(p), None) == 11
    assert lib.ss_bwd_validate(ctypes.byref(_good_bwd())) == 0


@pytest.mark.parametrize("mutate,status", [
    (lambda p: setattr(p, "abi_version", 3), 10),
    (lambda p: setattr(p, "dout", None), 1),
    (lambda p: setattr(p, "du", None), 1),
    (lambda p: setattr(p, "dA", None), 1),
    (lambda p: setattr(p, "dB", None), 1),
    (lambda p: setattr(p, "dz", None), 1),                    # z given, dz missing
    (lambda p: setattr(p, "dstate", 65), 7),
    (lambda p: setattr(p, "ngroups", 3), 2),
    (lambda p: setattr(p, "bc_dtype", api.SS_F16), 3),
    (lambda p: p.dout_stride.__setitem__(2, 2), 4),
    (lambda p: p.du_stride.__setitem__(2, 2), 4),
    (lambda p: p.dz_stride.__setitem__(1, -1), 4),
    (lambda p: setattr(p, "du", p.du + 1), 5),
    (lambda p: setattr(p, "dB", p.dB + 2), 5),
    (lambda p: setattr(p, "workspace", p.workspace + 8), 5),  # not 16-byte aligned
    (lambda p: setattr(p, "du", p.u), 6),                     # gradient written over an input
    (lambda p: setattr(p, "dA", p.A), 6),
    (lambda p: setattr(p, "dC", p.dB + 64), 6),               # two outputs overlap
    (lambda p: setattr(p, "dinitial_state", p.initial_state), 6),
    (lambda p: setattr(p, "workspace", p.dA), 6),
    (lambda p: setattr(p, "workspace_bytes", 100), 11),
    (lambda p: setattr(p, "workspace_bytes", -1), 2),
])
def test_bwd_invalid_params_rejected(lib, mutate, status):
    p = _good_bwd()
    mutate(p)
    assert lib.ss_bwd_validate(ctypes.byref(p)) == status
    assert lib.ss_bwd(ctypes.byref(p), None) == status


def test_bwd_optional_outputs_and_empty(lib):
    p = _good_bwd()
    for k in ("dD", "ddelta_bias", "dinitial_state", "D", "delta_bias", "initial_state"):
        setattr(p, k, None)
    assert lib.ss_bwd_validate(ctypes.byref(p)) == 0
    p.z = None
    p.dz = None
    assert lib.ss_bwd_validate(ctypes.byref(p)) == 0
    q = _good_bwd(with_ws=False)
    q.seqlen = 0  # zero gradients, no workspace needed
    assert lib.ss_bwd_validate(ctypes.byref(q)) == 0
    q = _good_bwd(with_ws=False)
    q.batch = 0
    assert lib.ss_bwd_validate(ctypes.byref(q)) == 0


# ---------------------------------------------------------------------------
# complex-A forward (ss_fwd_complex): validation only
# ---------------------------------------------------------------------------
def _good_cx():
    f = _good()
    p = api.SSFwdComplexParams()
    for k in ("abi_version", "in_dtype", "bc_dtype", "bc_mode", "delta_softplus", "batch", "dim", "seqlen",
              "dstate", "ngroups", "u", "delta", "z", "B", "C", "D", "delta_bias", "out"):
        setattr(p, k, getattr(f, k))
    for k in ("u_stride", "delta_stride", "z_stride", "out_stride", "B_stride", "C_stride", "A_stride"):
        getattr(p, k)[:] = list(getattr(f, k))
    cur = 1 << 44  # complex A and states: a region of their own
    p.A = cur
    p.last_state = cur + 64 * 16 * 8
    p.last_state_stride[:] = [64 * 16, 16, 1]
    p.initial_state_stride[:] = [0, 0, 1]
    return p


@pytest.mark.parametrize("mutate,status", [
    (lambda p: None, 0),
    (lambda p: setattr(p, "abi_version", 2), 10),
    (lambda p: setattr(p, "A", None), 1),
    (lambda p: setattr(p, "A", p.A + 4), 5),                  # complex64 needs 8-byte alignment
    (lambda p: setattr(p, "last_state", p.last_state + 4), 5),
    (lambda p: p.A_stride.__setitem__(1, 2), 4),
    (lambda p: setattr(p, "dstate", 65), 7),
    (lambda p: setattr(p, "out", p.u), 6),
    (lambda p: setattr(p, "last_state", p.A + 8), 6),         # overlaps A (16-byte elements span)
    (lambda p: (setattr(p, "initial_state", p.last_state), p.initial_state_stride.__setitem__(0, 64 * 16),
                p.initial_state_stride.__setitem__(1, 16)), 0),  # in place: allowed
])
def test_complex_validation(lib, mutate, status):
    p = _good_cx()
    mutate(p)
    assert lib.ss_fwd_complex_validate(ctypes.byref(p)) == status
    if status:
        assert lib.ss_fwd_complex(ctypes.byref(p), None) == status
