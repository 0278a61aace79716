"""Python binding of libssfwd.so (C ABI in include/ssfwd.h).

Argument marshalling only: shapes, strides, dtypes and device pointers are
read from torch tensors and handed to ``ss_fwd``; every step of the
selective scan runs in the library's CUDA kernels. torch supplies device
memory and the current stream. There is no CPU fallback: without the built
library or a CUDA device the calls raise.

``selective_scan_fn`` mirrors the signature and layout handling of the page
"PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南",
section 4.1: tensors whose last stride is not 1 are made contiguous, a 3-D
(batch, dstate, seqlen) B/C is treated as 4-D with one group, and the result
is ``out`` or ``(out, last_state)``. When an input requires a gradient the
call goes through ``SelectiveScanFn``, whose backward runs ``ss_bwd``
(last_state carries no gradient, as on the page).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

# SSFWD_LIBRARY may point at another build of the same library (e.g. one built
# with different compile-time knobs); default: the in-tree build.
_LIB_PATH = os.environ.get("SSFWD_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "_build", "libssfwd.so")
_lock = threading.Lock()
_lib = None

SS_F32, SS_F16, SS_BF16 = 0, 1, 2
SS_BC_FIXED, SS_BC_VARIABLE = 0, 1
SS_ABI_VERSION = 5
_DT = {torch.float32: SS_F32, torch.float16: SS_F16, torch.bfloat16: SS_BF16}

_i64x2, _i64x3, _i64x4 = ctypes.c_int64 * 2, ctypes.c_int64 * 3, ctypes.c_int64 * 4


class SSFwdParams(ctypes.Structure):
    """Mirror of ``ss_fwd_params``."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("bc_dtype", ctypes.c_int32),
        ("bc_mode", ctypes.c_int32), ("delta_softplus", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
        ("u", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("delta_bias", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("last_state", ctypes.c_void_p),
        ("u_stride", _i64x3), ("delta_stride", _i64x3), ("z_stride", _i64x3), ("out_stride", _i64x3),
        ("B_stride", _i64x4), ("C_stride", _i64x4), ("A_stride", _i64x2), ("last_state_stride", _i64x3),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64),
        ("initial_state", ctypes.c_void_p), ("initial_state_stride", _i64x3),
        ("error_word", ctypes.c_void_p),
    ]


class SSStateUpdateParams(ctypes.Structure):
    """Mirror of ``ss_state_update_params``."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("bc_dtype", ctypes.c_int32),
        ("bc_mode", ctypes.c_int32), ("delta_softplus", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
        ("state", ctypes.c_void_p),
        ("u", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("delta_bias", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("state_stride", _i64x3),
        ("u_stride", _i64x2), ("delta_stride", _i64x2), ("z_stride", _i64x2), ("out_stride", _i64x2),
        ("B_stride", _i64x3), ("C_stride", _i64x3), ("A_stride", _i64x2),
    ]


class SSConv1dParams(ctypes.Structure):
    """Mirror of ``ss_conv1d_params``."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("dtype", ctypes.c_int32), ("activation", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("width", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("seq_idx", ctypes.c_void_p), ("initial_states", ctypes.c_void_p), ("final_states", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("x_stride", _i64x3), ("out_stride", _i64x3), ("weight_stride", _i64x2), ("seq_idx_stride", _i64x2),
        ("initial_states_stride", _i64x3), ("final_states_stride", _i64x3),
    ]


class SSConv1dUpdateParams(ctypes.Structure):
    """Mirror of ``ss_conv1d_update_params``."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("dtype", ctypes.c_int32), ("activation", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("width", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("conv_state", ctypes.c_void_p), ("weight", ctypes.c_void_p),
        ("bias", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("x_stride", _i64x2), ("conv_state_stride", _i64x3), ("weight_stride", _i64x2), ("out_stride", _i64x2),
    ]


class SSFwdComplexParams(ctypes.Structure):
    """Mirror of ``ss_fwd_complex_params``."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("bc_dtype", ctypes.c_int32),
        ("bc_mode", ctypes.c_int32), ("delta_softplus", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
        ("u", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("delta_bias", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("last_state", ctypes.c_void_p), ("initial_state", ctypes.c_void_p),
        ("u_stride", _i64x3), ("delta_stride", _i64x3), ("z_stride", _i64x3), ("out_stride", _i64x3),
        ("B_stride", _i64x4), ("C_stride", _i64x4), ("A_stride", _i64x2),
        ("last_state_stride", _i64x3), ("initial_state_stride", _i64x3),
    ]


class SSBwdParams(ctypes.Structure):
    """Mirror of ``ss_bwd_params``."""
    _fields_ = [
        ("abi_version", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("bc_dtype", ctypes.c_int32),
        ("bc_mode", ctypes.c_int32), ("delta_softplus", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("seqlen", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
        ("u", ctypes.c_void_p), ("delta", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("B", ctypes.c_void_p), ("C", ctypes.c_void_p), ("dout", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("delta_bias", ctypes.c_void_p),
        ("initial_state", ctypes.c_void_p),
        ("du", ctypes.c_void_p), ("ddelta", ctypes.c_void_p), ("dz", ctypes.c_void_p),
        ("dA", ctypes.c_void_p), ("dB", ctypes.c_void_p), ("dC", ctypes.c_void_p),
        ("dD", ctypes.c_void_p), ("ddelta_bias", ctypes.c_void_p), ("dinitial_state", ctypes.c_void_p),
        ("u_stride", _i64x3), ("delta_stride", _i64x3), ("z_stride", _i64x3), ("dout_stride", _i64x3),
        ("du_stride", _i64x3), ("ddelta_stride", _i64x3), ("dz_stride", _i64x3),
        ("B_stride", _i64x4), ("C_stride", _i64x4), ("A_stride", _i64x2),
        ("initial_state_stride", _i64x3),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64),
    ]


SS_ACT_NONE, SS_ACT_SILU = 0, 1


class SSError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libssfwd call failed: status {status} ({msg})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libssfwd.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"libssfwd.so is not built ({_LIB_PATH}); build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER(SSFwdParams)
            vp = ctypes.c_void_p
            lib.ss_abi_version.restype = ctypes.c_int
            lib.ss_status_string.argtypes = [ctypes.c_int]
            lib.ss_status_string.restype = ctypes.c_char_p
            lib.ss_fwd_validate.argtypes = [P]
            lib.ss_fwd_validate.restype = ctypes.c_int
            lib.ss_fwd.argtypes = [P, vp]
            lib.ss_fwd.restype = ctypes.c_int
            lib.ss_fwd_noalloc.argtypes = [P, vp]
            lib.ss_fwd_noalloc.restype = ctypes.c_int
            lib.ss_fwd_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
            lib.ss_fwd_workspace_size.restype = ctypes.c_int
            lib.ss_fwd_host.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.ss_fwd_host.restype = ctypes.c_int
            PS = ctypes.POINTER(SSStateUpdateParams)
            lib.ss_state_update_validate.argtypes = [PS]
            lib.ss_state_update_validate.restype = ctypes.c_int
            lib.ss_state_update.argtypes = [PS, vp]
            lib.ss_state_update.restype = ctypes.c_int
            PC, PU = ctypes.POINTER(SSConv1dParams), ctypes.POINTER(SSConv1dUpdateParams)
            lib.ss_causal_conv1d_validate.argtypes = [PC]
            lib.ss_causal_conv1d_validate.restype = ctypes.c_int
            lib.ss_causal_conv1d.argtypes = [PC, vp]
            lib.ss_causal_conv1d.restype = ctypes.c_int
            lib.ss_causal_conv1d_update_validate.argtypes = [PU]
            lib.ss_causal_conv1d_update_validate.restype = ctypes.c_int
            lib.ss_causal_conv1d_update.argtypes = [PU, vp]
            lib.ss_causal_conv1d_update.restype = ctypes.c_int
            PX = ctypes.POINTER(SSFwdComplexParams)
            lib.ss_fwd_complex_validate.argtypes = [PX]
            lib.ss_fwd_complex_validate.restype = ctypes.c_int
            lib.ss_fwd_complex.argtypes = [PX, vp]
            lib.ss_fwd_complex.restype = ctypes.c_int
            PB = ctypes.POINTER(SSBwdParams)
            lib.ss_bwd_validate.argtypes = [PB]
            lib.ss_bwd_validate.restype = ctypes.c_int
            lib.ss_bwd_workspace_size.argtypes = [PB, ctypes.POINTER(ctypes.c_int64)]
            lib.ss_bwd_workspace_size.restype = ctypes.c_int
            lib.ss_bwd.argtypes = [PB, vp]
            lib.ss_bwd.restype = ctypes.c_int
            lib.ss_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
            lib.ss_device_error.restype = ctypes.c_int
            if lib.ss_abi_version() != SS_ABI_VERSION:
                raise RuntimeError("libssfwd.so ABI version mismatch")
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().ss_status_string(status).decode()


def _check(status: int):
    if status != 0:
        raise SSError(status, status_string(status))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _unit_last(t):
    if t is not None and t.dim() > 0 and t.stride(-1) != 1:
        return t.contiguous()
    return t


def normalise(u, delta, A, B, C, D=None, z=None, delta_bias=None):
    """Layout handling of the page's selective_scan_fn: unit last stride (else
    .contiguous()), 3-D B/C -> 4-D with one group. Returns the tensors. A
    complex A becomes complex64 (the complex-A variant, ss_fwd_complex)."""
    if A.is_complex() and A.dtype != torch.complex64:
        A = A.to(torch.complex64)
    u, delta, z, B, C, A = (_unit_last(t) for t in (u, delta, z, B, C, A))
    if B.dim() == 3:
        B = B.unsqueeze(1)
    if C.dim() == 3:
        C = C.unsqueeze(1)
    if D is not None:
        D = D.contiguous()
    if delta_bias is not None:
        delta_bias = delta_bias.contiguous()
    return u, delta, A, B, C, D, z, delta_bias


def make_params(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, last_state,
                initial_state=None) -> SSFwdParams:
    """Fill an ss_fwd_params from already-normalised tensors (see normalise)."""
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    if u.dtype not in _DT:
        raise TypeError(f"unsupported dtype {u.dtype}")
    for name, t in (("delta", delta), ("z", z)):
        if t is not None and (t.dtype != u.dtype or t.shape != u.shape):
            raise TypeError(f"{name} must match u in shape and dtype")
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    batch, dim, seqlen = u.shape
    if A.dim() != 2 or A.shape[0] != dim:
        raise ValueError("A must be (dim, dstate)")
    dstate = A.shape[1]
    p = SSFwdParams()
    p.abi_version = SS_ABI_VERSION
    p.in_dtype = _DT[u.dtype]
    if B.dim() == 2:
        p.bc_mode, p.ngroups = SS_BC_FIXED, 1
        if B.dtype != torch.float32 or C.dtype != torch.float32:
            raise TypeError("fixed (dim, dstate) B/C must be float32")
        if tuple(B.shape) != (dim, dstate) or tuple(C.shape) != (dim, dstate):
            raise ValueError("fixed B/C must be (dim, dstate)")
        p.B_stride[:] = [B.stride(0), B.stride(1), 0, 0]
        p.C_stride[:] = [C.stride(0), C.stride(1), 0, 0]
    elif B.dim() == 4:
        p.bc_mode, p.ngroups = SS_BC_VARIABLE, B.shape[1]
        if B.dtype not in (u.dtype, torch.float32) or C.dtype != B.dtype:
            raise TypeError("variable B/C must share a dtype, equal to u's or float32")
        want = (batch, B.shape[1], dstate, seqlen)
        if tuple(B.shape) != want or tuple(C.shape) != want:
            raise ValueError(f"variable B/C must be {want}")
        p.B_stride[:] = list(B.stride())
        p.C_stride[:] = list(C.stride())
    else:
        raise ValueError("B/C must be (dim, dstate), (batch, dstate, seqlen) or (batch, groups, dstate, seqlen)")
    p.bc_dtype = _DT[B.dtype]
    p.delta_softplus = int(bool(delta_softplus))
    p.batch, p.dim, p.seqlen, p.dstate = batch, dim, seqlen, dstate
    p.u, p.delta, p.z, p.B, p.C = _ptr(u), _ptr(delta), _ptr(z), _ptr(B), _ptr(C)
    p.A, p.D, p.delta_bias = _ptr(A), _ptr(D), _ptr(delta_bias)
    p.out, p.last_state = _ptr(out), _ptr(last_state)
    p.u_stride[:] = list(u.stride())
    p.delta_stride[:] = list(delta.stride())
    p.z_stride[:] = list(z.stride()) if z is not None else [0, 0, 1]
    p.out_stride[:] = list(out.stride())
    p.A_stride[:] = list(A.stride())
    p.last_state_stride[:] = list(last_state.stride()) if last_state is not None else [0, 0, 1]
    if initial_state is not None:
        if initial_state.dtype != torch.float32 or tuple(initial_state.shape) != (batch, dim, dstate):
            raise TypeError("initial_state must be float32 (batch, dim, dstate)")
        p.initial_state = _ptr(initial_state)
        p.initial_state_stride[:] = list(initial_state.stride())
    else:
        p.initial_state_stride[:] = [0, 0, 1]
    return p


def attach_workspace(p: SSFwdParams, device) -> "torch.Tensor | None":
    """Allocate (torch, on `device`) and attach the workspace the fastest
    schedule of p asks for; returns the tensor to keep alive, or None."""
    lib = load_library()
    n = ctypes.c_int64(0)
    with torch.cuda.device(device):
        _check(lib.ss_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    if n.value <= 0:
        return None
    ws = torch.empty(int(n.value), dtype=torch.uint8, device=device)
    p.workspace, p.workspace_bytes = ws.data_ptr(), int(n.value)
    return ws


def _forward(u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state, initial_state):
    """ss_fwd on normalised CUDA tensors; returns (out, last_state or None)."""
    lib = load_library()
    out = torch.empty(u.shape, dtype=u.dtype, device=u.device)
    last = (torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.float32, device=u.device)
            if return_last_state else None)
    p = make_params(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, last, initial_state)
    ws = attach_workspace(p, u.device)
    stream = torch.cuda.current_stream(u.device)
    with torch.cuda.device(u.device):
        _check(lib.ss_fwd(ctypes.byref(p), stream.cuda_stream))
    if ws is not None:
        ws.record_stream(stream)
    return out, last


def make_complex_params(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, last_state,
                        initial_state=None) -> SSFwdComplexParams:
    """Fill an ss_fwd_complex_params from normalised tensors; A, last_state and
    initial_state are complex64 (interleaved (re, im) in memory)."""
    if A.dtype != torch.complex64 or A.dim() != 2:
        raise TypeError("complex A must be complex64 (dim, dstate)")
    # the real-A filler checks every other operand; A's real view stands in for it
    f = make_params(u, delta, torch.view_as_real(A)[..., 0], B, C, D, z, delta_bias, delta_softplus, out, None)
    p = SSFwdComplexParams()
    for k in ("abi_version", "in_dtype", "bc_dtype", "bc_mode", "delta_softplus", "batch", "dim", "seqlen",
              "dstate", "ngroups", "u", "delta", "z", "B", "C", "D", "delta_bias", "out"):
        setattr(p, k, getattr(f, k))
    for k in ("u_stride", "delta_stride", "z_stride", "out_stride", "B_stride", "C_stride"):
        getattr(p, k)[:] = list(getattr(f, k))
    p.A = A.data_ptr()
    p.A_stride[:] = list(A.stride())
    shape = (f.batch, f.dim, f.dstate)
    for name, t in (("last_state", last_state), ("initial_state", initial_state)):
        if t is not None:
            if t.dtype != torch.complex64 or tuple(t.shape) != shape:
                raise TypeError(f"{name} must be complex64 (batch, dim, dstate)")
            setattr(p, name, t.data_ptr())
            getattr(p, name + "_stride")[:] = list(t.stride())
        else:
            getattr(p, name + "_stride")[:] = [0, 0, 1]
    return p


def _forward_complex(u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state, initial_state):
    out = torch.empty(u.shape, dtype=u.dtype, device=u.device)
    last = (torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.complex64, device=u.device)
            if return_last_state else None)
    p = make_complex_params(u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, last, initial_state)
    with torch.cuda.device(u.device):
        _check(load_library().ss_fwd_complex(ctypes.byref(p), torch.cuda.current_stream(u.device).cuda_stream))
    return out, last


def selective_scan_fn(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                      delta_softplus=False, return_last_state=False, initial_state=None):
    """Selective-scan forward on CUDA tensors; runs on the current stream.

    u, delta, z: (batch, dim, seqlen), fp32/fp16/bf16, one dtype.
    A: (dim, dstate) fp32 (real). B, C: (dim, dstate) fp32 fixed, or
    (batch, dstate, seqlen) / (batch, groups, dstate, seqlen) in u's dtype or
    fp32. D, delta_bias: (dim,) fp32. initial_state: optional (batch, dim,
    dstate) fp32 start state (zero if None). Returns out (u's dtype), or
    (out, last_state) with last_state (batch, dim, dstate) fp32. Differentiable
    (through ss_bwd) in every input but last_state. A complex A (complex64,
    real B/C) runs the complex-A variant (ss_fwd_complex; forward only): the
    state and last_state are complex, out takes the real part of the
    contraction.
    """
    if not u.is_cuda:
        raise RuntimeError("selective_scan_fn needs CUDA tensors (there is no CPU path)")
    ins = (u, delta, A, B, C, D, z, delta_bias, initial_state)
    if A.is_complex():
        if torch.is_grad_enabled() and any(t is not None and t.requires_grad for t in ins):
            raise NotImplementedError("the complex-A variant is forward only")
        u, delta, A, B, C, D, z, delta_bias = normalise(u, delta, A, B, C, D, z, delta_bias)
        if initial_state is not None:
            initial_state = _unit_last(initial_state.to(torch.complex64))
        out, last = _forward_complex(u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state,
                                     initial_state)
        return (out, last) if return_last_state else out
    if torch.is_grad_enabled() and any(t is not None and t.requires_grad for t in ins):
        out, last = SelectiveScanFn.apply(u, delta, A, B, C, D, z, delta_bias, bool(delta_softplus),
                                          bool(return_last_state), initial_state)
        return (out, last) if return_last_state else out
    u, delta, A, B, C, D, z, delta_bias = normalise(u, delta, A, B, C, D, z, delta_bias)
    if initial_state is not None:
        initial_state = _unit_last(initial_state)
    out, last = _forward(u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state, initial_state)
    return (out, last) if return_last_state else out


def make_bwd_params(dout, u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state,
                    du, ddelta, dz, dA, dB, dC, dD, ddelta_bias, dinitial_state) -> SSBwdParams:
    """Fill an ss_bwd_params from normalised CUDA tensors (B/C 2-D or 4-D);
    the workspace is attached separately (attach_bwd_workspace)."""
    f = make_params(u, delta, A, B, C, D, z, delta_bias, delta_softplus, du, None, initial_state)
    for name, t in (("dout", dout), ("du", du), ("ddelta", ddelta), ("dz", dz)):
        if t is not None and (t.dtype != u.dtype or t.shape != u.shape):
            raise TypeError(f"{name} must match u in shape and dtype")
    p = SSBwdParams()
    for k in ("abi_version", "in_dtype", "bc_dtype", "bc_mode", "delta_softplus", "batch", "dim", "seqlen",
              "dstate", "ngroups", "u", "delta", "z", "B", "C", "A", "D", "delta_bias", "initial_state"):
        setattr(p, k, getattr(f, k))
    for k in ("u_stride", "delta_stride", "z_stride", "B_stride", "C_stride", "A_stride", "initial_state_stride"):
        getattr(p, k)[:] = list(getattr(f, k))
    p.dout = _ptr(dout)
    p.du, p.ddelta, p.dz = _ptr(du), _ptr(ddelta), _ptr(dz)
    p.dA, p.dB, p.dC = _ptr(dA), _ptr(dB), _ptr(dC)
    p.dD, p.ddelta_bias, p.dinitial_state = _ptr(dD), _ptr(ddelta_bias), _ptr(dinitial_state)
    p.dout_stride[:] = list(dout.stride())
    p.du_stride[:] = list(du.stride())
    p.ddelta_stride[:] = list(ddelta.stride())
    p.dz_stride[:] = list(dz.stride()) if dz is not None else [0, 0, 1]
    return p


def attach_bwd_workspace(p: SSBwdParams, device) -> "torch.Tensor | None":
    """Allocate (torch) and attach the checkpoint workspace ss_bwd needs."""
    n = ctypes.c_int64(0)
    _check(load_library().ss_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    if n.value <= 0:
        return None
    ws = torch.empty(int(n.value), dtype=torch.uint8, device=device)
    p.workspace, p.workspace_bytes = ws.data_ptr(), int(n.value)
    return ws


def selective_scan_bwd(dout, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                       initial_state=None, want_dD=None, want_ddelta_bias=None, want_dinitial_state=None):
    """Gradients of sum(dout * out) for selective_scan_fn (through ss_bwd), on
    the current stream. Returns a dict: du, ddelta, dz (u's dtype), dA (fp32),
    dB, dC (B/C's dtype and shape), dD, ddelta_bias, dinitial_state (fp32;
    None when not wanted, by default when the input is absent)."""
    if not u.is_cuda:
        raise RuntimeError("selective_scan_bwd needs CUDA tensors (there is no CPU path)")
    B_in = B
    u, delta, A, B, C, D, z, delta_bias = normalise(u, delta, A, B, C, D, z, delta_bias)
    dout = _unit_last(dout)
    if initial_state is not None:
        initial_state = _unit_last(initial_state)
    want_dD = D is not None if want_dD is None else want_dD
    want_ddelta_bias = delta_bias is not None if want_ddelta_bias is None else want_ddelta_bias
    want_dinitial_state = initial_state is not None if want_dinitial_state is None else want_dinitial_state
    dev = u.device
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    f32 = dict(dtype=torch.float32, device=dev)
    du, ddelta = torch.empty_like(u), torch.empty_like(u)
    dz = torch.empty_like(u) if z is not None else None
    dA = torch.empty((dim, dstate), **f32)
    dB, dC = torch.empty(B.shape, **f32), torch.empty(C.shape, **f32)
    dD = torch.empty(dim, **f32) if want_dD else None
    ddb = torch.empty(dim, **f32) if want_ddelta_bias else None
    dx0 = torch.empty((batch, dim, dstate), **f32) if want_dinitial_state else None
    p = make_bwd_params(dout, u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state,
                        du, ddelta, dz, dA, dB, dC, dD, ddb, dx0)
    ws = attach_bwd_workspace(p, dev)
    stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        _check(load_library().ss_bwd(ctypes.byref(p), stream.cuda_stream))
    if ws is not None:
        ws.record_stream(stream)
    if B_in.dim() == 3:
        dB, dC = dB[:, 0], dC[:, 0]
    return dict(du=du, ddelta=ddelta, dz=dz, dA=dA, dB=dB.to(B_in.dtype), dC=dC.to(B_in.dtype),
                dD=dD, ddelta_bias=ddb, dinitial_state=dx0)


class SelectiveScanFn(torch.autograd.Function):
    """selective_scan_fn with its backward (the page's SelectiveScanFn layer):
    forward through ss_fwd, backward through ss_bwd; last_state has no
    gradient."""

    @staticmethod
    def forward(ctx, u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state, initial_state):
        B3 = B.dim() == 3
        nu, nd, nA, nB, nC, nD, nz, nb = normalise(u, delta, A, B, C, D, z, delta_bias)
        x0 = _unit_last(initial_state) if initial_state is not None else None
        out, last = _forward(nu, nd, nA, nB, nC, nD, nz, nb, delta_softplus, return_last_state, x0)
        ctx.save_for_backward(nu, nd, nA, nB, nC, nD, nz, nb, x0)
        ctx.delta_softplus, ctx.B3 = delta_softplus, B3
        ctx.dtypes = (B.dtype, C.dtype)
        if last is not None:
            ctx.mark_non_differentiable(last)
        return out, last

    @staticmethod
    def backward(ctx, dout, dlast):
        u, delta, A, B, C, D, z, bias, x0 = ctx.saved_tensors
        need = ctx.needs_input_grad
        g = selective_scan_bwd(dout, u, delta, A, B, C, D, z, bias, ctx.delta_softplus, x0,
                               want_dD=D is not None and need[5],
                               want_ddelta_bias=bias is not None and need[7],
                               want_dinitial_state=x0 is not None and need[10])
        dB, dC = g["dB"].to(ctx.dtypes[0]), g["dC"].to(ctx.dtypes[1])
        if ctx.B3:
            dB, dC = dB[:, 0], dC[:, 0]
        return (g["du"], g["ddelta"], g["dA"], dB, dC, g["dD"], g["dz"], g["ddelta_bias"], None, None,
                g["dinitial_state"])


class HostRunner:
    """End-to-end runner for HOST tensors through ``ss_fwd_host``: each call
    copies the (pinned) host inputs into device buffers owned by this object,
    runs the kernel and copies ``out`` (and ``last_state``) back, all on one
    stream; ``run`` returns once the stream has completed.

    The device buffers are allocated once (torch) for the given shapes/dtypes;
    host tensors passed to ``run`` must have exactly those shapes and dtypes
    and be contiguous.
    """

    def __init__(self, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                 delta_softplus=False, return_last_state=False, device="cuda", initial_state=None):
        lib = load_library()
        self._lib = lib
        # an optional start state stays on the device (float32 (batch, dim, dstate))
        self.initial_state = None if initial_state is None else _unit_last(initial_state)
        host = normalise(u, delta, A, B, C, D, z, delta_bias)
        self._host_shapes = [None if t is None else (tuple(t.shape), t.dtype) for t in host]
        dev = [None if t is None else torch.empty(t.shape, dtype=t.dtype, device=device) for t in host]
        self.dev = dev
        du = dev[0]
        self.out = torch.empty(du.shape, dtype=du.dtype, device=device)
        self.last = (torch.empty((du.shape[0], du.shape[1], dev[2].shape[1]), dtype=torch.float32, device=device)
                     if return_last_state else None)
        self.params = make_params(*dev, delta_softplus, self.out, self.last, self.initial_state)
        self.workspace = attach_workspace(self.params, self.out.device)
        self.h_out = torch.empty(du.shape, dtype=du.dtype, pin_memory=True)
        self.h_last = (torch.empty(self.last.shape, dtype=torch.float32, pin_memory=True)
                       if return_last_state else None)
        self.stream = torch.cuda.Stream(device=device)

    @property
    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.dev if t is not None)

    @property
    def d2h_bytes(self) -> int:
        return self.h_out.numel() * self.h_out.element_size() + (
            0 if self.h_last is None else self.h_last.numel() * 4)

    def enqueue(self, u, delta, A, B, C, D=None, z=None, delta_bias=None):
        host = normalise(u, delta, A, B, C, D, z, delta_bias)
        for t, want in zip(host, self._host_shapes):
            if (t is None) != (want is None) or (t is not None and (tuple(t.shape), t.dtype) != want):
                raise ValueError("host tensors do not match the runner's shapes/dtypes")
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("host tensors must be contiguous CPU tensors")
        hp = [None if t is None else t.data_ptr() for t in host]
        # order of ss_fwd_host: u, delta, z, B, C, A, D, delta_bias
        _check(self._lib.ss_fwd_host(
            ctypes.byref(self.params), hp[0], hp[1], hp[6], hp[3], hp[4], hp[2], hp[5], hp[7],
            self.h_out.data_ptr(), None if self.h_last is None else self.h_last.data_ptr(),
            self.stream.cuda_stream))

    def run(self, *args, **kwargs):
        self.enqueue(*args, **kwargs)
        self.stream.synchronize()
        return (self.h_out, self.h_last) if self.h_last is not None else self.h_out


def selective_scan_fn_host(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                           delta_softplus=False, return_last_state=False):
    """selective_scan_fn for CPU tensors: copies in, runs on the GPU, copies
    out (through ss_fwd_host). Returns CPU tensors."""
    r = HostRunner(u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state)
    res = r.run(u.contiguous(), delta.contiguous(), A, B.contiguous(), C.contiguous(), D,
                None if z is None else z.contiguous(), delta_bias)
    if return_last_state:
        return res[0].clone(), res[1].clone()
    return res.clone()


def make_state_update_params(state, u, delta, A, B, C, D, z, delta_bias, delta_softplus, out,
                             bc_fixed=False) -> SSStateUpdateParams:
    """Fill an ss_state_update_params from CUDA tensors (no copies made)."""
    if u.dim() != 2 or u.dtype not in _DT:
        raise TypeError("u must be (batch, dim) fp32/fp16/bf16")
    batch, dim = u.shape
    for name, t in (("delta", delta), ("z", z), ("out", out)):
        if t is not None and (t.dtype != u.dtype or tuple(t.shape) != (batch, dim)):
            raise TypeError(f"{name} must match u in shape and dtype")
    if A.dim() != 2 or A.shape[0] != dim or A.dtype != torch.float32:
        raise TypeError("A must be float32 (dim, dstate)")
    dstate = A.shape[1]
    if state.dtype != torch.float32 or tuple(state.shape) != (batch, dim, dstate):
        raise TypeError("state must be float32 (batch, dim, dstate)")
    for name, t in (("D", D), ("delta_bias", delta_bias)):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (dim,)):
            raise TypeError(f"{name} must be float32 (dim,)")
    p = SSStateUpdateParams()
    p.abi_version = SS_ABI_VERSION
    p.in_dtype = _DT[u.dtype]
    if bc_fixed:
        if B.dtype != torch.float32 or C.dtype != torch.float32 or tuple(B.shape) != (dim, dstate) \
                or tuple(C.shape) != (dim, dstate):
            raise TypeError("fixed B/C must be float32 (dim, dstate)")
        p.bc_mode, p.ngroups = SS_BC_FIXED, 1
        p.B_stride[:] = [B.stride(0), B.stride(1), 0]
        p.C_stride[:] = [C.stride(0), C.stride(1), 0]
    else:
        if B.dim() == 2:
            B, C = B.unsqueeze(1), C.unsqueeze(1)
        if B.dim() != 3 or B.shape[0] != batch or B.shape[2] != dstate or tuple(C.shape) != tuple(B.shape):
            raise ValueError("B/C must be (batch, dstate) or (batch, groups, dstate)")
        if B.dtype not in (u.dtype, torch.float32) or C.dtype != B.dtype:
            raise TypeError("B/C must share a dtype, equal to u's or float32")
        p.bc_mode, p.ngroups = SS_BC_VARIABLE, B.shape[1]
        p.B_stride[:] = list(B.stride())
        p.C_stride[:] = list(C.stride())
    p.bc_dtype = _DT[B.dtype]
    p.delta_softplus = int(bool(delta_softplus))
    p.batch, p.dim, p.dstate = batch, dim, dstate
    p.state = _ptr(state)
    p.u, p.delta, p.z, p.B, p.C = _ptr(u), _ptr(delta), _ptr(z), _ptr(B), _ptr(C)
    p.A, p.D, p.delta_bias, p.out = _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(out)
    p.state_stride[:] = list(state.stride())
    p.u_stride[:] = list(u.stride())
    p.delta_stride[:] = list(delta.stride())
    p.z_stride[:] = list(z.stride()) if z is not None else [0, 0]
    p.out_stride[:] = list(out.stride())
    p.A_stride[:] = list(A.stride())
    return p


def selective_state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                           delta_softplus=False, bc_fixed=False):
    """One decode step on CUDA tensors (current stream): updates ``state``
    (batch, dim, dstate) fp32 in place and returns out (batch, dim).

    u, delta, z: (batch, dim) in one dtype; B, C: (batch, dstate) or
    (batch, groups, dstate) in u's dtype or fp32, or with bc_fixed (dim, dstate)
    fp32; A: (dim, dstate) fp32; D, delta_bias: (dim,) fp32.
    """
    if not u.is_cuda:
        raise RuntimeError("selective_state_update needs CUDA tensors (there is no CPU path)")
    lib = load_library()
    if state.stride(-1) != 1:
        raise ValueError("state must have a unit last stride (it is updated in place)")
    A = _unit_last(A)
    B, C = _unit_last(B), _unit_last(C)
    out = torch.empty(u.shape, dtype=u.dtype, device=u.device)
    p = make_state_update_params(state, u, delta, A, B, C, D, z, delta_bias, delta_softplus, out, bc_fixed)
    stream = torch.cuda.current_stream(u.device).cuda_stream
    with torch.cuda.device(u.device):
        _check(lib.ss_state_update(ctypes.byref(p), stream))
    return out


def _activation(activation) -> int:
    if activation is None:
        return SS_ACT_NONE
    if activation in ("silu", "swish"):
        return SS_ACT_SILU
    raise NotImplementedError("activation must be None, 'silu' or 'swish'")


def make_conv1d_params(x, weight, bias, seq_idx, initial_states, final_states, out, activation) -> SSConv1dParams:
    """Fill an ss_conv1d_params from CUDA tensors (no copies made)."""
    if x.dim() != 3 or x.dtype not in _DT:
        raise TypeError("x must be (batch, dim, seqlen) fp32/fp16/bf16")
    batch, dim, seqlen = x.shape
    if weight.dim() != 2 or weight.shape[0] != dim or weight.dtype != torch.float32:
        raise TypeError("weight must be float32 (dim, width)")
    width = weight.shape[1]
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (dim,)):
        raise TypeError("bias must be float32 (dim,)")
    for name, t in (("initial_states", initial_states), ("final_states", final_states)):
        if t is not None and (t.dtype != x.dtype or tuple(t.shape) != (batch, dim, width - 1)):
            raise TypeError(f"{name} must be x's dtype (batch, dim, width - 1)")
    if seq_idx is not None and (seq_idx.dtype != torch.int32 or tuple(seq_idx.shape) != (batch, seqlen)):
        raise TypeError("seq_idx must be int32 (batch, seqlen)")
    p = SSConv1dParams()
    p.abi_version = SS_ABI_VERSION
    p.dtype = _DT[x.dtype]
    p.activation = _activation(activation)
    p.batch, p.dim, p.seqlen, p.width = batch, dim, seqlen, width
    p.x, p.weight, p.bias, p.seq_idx = _ptr(x), _ptr(weight), _ptr(bias), _ptr(seq_idx)
    p.initial_states, p.final_states, p.out = _ptr(initial_states), _ptr(final_states), _ptr(out)
    p.x_stride[:] = list(x.stride())
    p.out_stride[:] = list(out.stride())
    p.weight_stride[:] = list(weight.stride())
    p.seq_idx_stride[:] = list(seq_idx.stride()) if seq_idx is not None else [0, 1]
    p.initial_states_stride[:] = list(initial_states.stride()) if initial_states is not None else [0, 0, 1]
    p.final_states_stride[:] = list(final_states.stride()) if final_states is not None else [0, 0, 1]
    return p


def causal_conv1d_fn(x, weight, bias=None, seq_idx=None, initial_states=None, return_final_states=False,
                     final_states_out=None, activation=None):
    """Causal depthwise conv1d on CUDA tensors (current stream), with the
    signature of the page's causal_conv1d_fn: x (batch, dim, seqlen); weight
    (dim, width) fp32, 2 <= width <= 4; bias (dim,) fp32; seq_idx (batch,
    seqlen) int32; initial_states / final_states_out (batch, dim, width - 1) in
    x's dtype; activation None, 'silu' or 'swish'. Returns out, or
    (out, final_states) when return_final_states."""
    if not x.is_cuda:
        raise RuntimeError("causal_conv1d_fn needs CUDA tensors (there is no CPU path)")
    lib = load_library()
    _activation(activation)
    if seq_idx is not None and (initial_states is not None or return_final_states):
        raise ValueError("seq_idx cannot be combined with initial_states or return_final_states")
    x = _unit_last(x)
    weight = _unit_last(weight)
    out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    fin = None
    if return_final_states:
        fin = final_states_out if final_states_out is not None else torch.empty(
            (x.shape[0], x.shape[1], weight.shape[1] - 1), dtype=x.dtype, device=x.device)
    p = make_conv1d_params(x, weight, bias, seq_idx, initial_states, fin, out, activation)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        _check(lib.ss_causal_conv1d(ctypes.byref(p), stream))
    return (out, fin) if return_final_states else out


def causal_conv1d_update(x, conv_state, weight, bias=None, activation=None):
    """One decode step of the convolution on CUDA tensors: x (batch, dim) new
    input, conv_state (batch, dim, width - 1) updated in place (oldest first).
    Returns out (batch, dim)."""
    if not x.is_cuda:
        raise RuntimeError("causal_conv1d_update needs CUDA tensors (there is no CPU path)")
    lib = load_library()
    if x.dim() != 2 or x.dtype not in _DT:
        raise TypeError("x must be (batch, dim) fp32/fp16/bf16")
    batch, dim = x.shape
    if weight.dim() != 2 or weight.shape[0] != dim or weight.dtype != torch.float32:
        raise TypeError("weight must be float32 (dim, width)")
    width = weight.shape[1]
    if conv_state.dtype != x.dtype or tuple(conv_state.shape) != (batch, dim, width - 1):
        raise TypeError("conv_state must be x's dtype (batch, dim, width - 1)")
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (dim,)):
        raise TypeError("bias must be float32 (dim,)")
    out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    p = SSConv1dUpdateParams()
    p.abi_version = SS_ABI_VERSION
    p.dtype = _DT[x.dtype]
    p.activation = _activation(activation)
    p.batch, p.dim, p.width = batch, dim, width
    p.x, p.conv_state, p.weight, p.bias, p.out = _ptr(x), _ptr(conv_state), _ptr(weight), _ptr(bias), _ptr(out)
    p.x_stride[:] = list(x.stride())
    p.conv_state_stride[:] = list(conv_state.stride())
    p.weight_stride[:] = list(weight.stride())
    p.out_stride[:] = list(out.stride())
    stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        _check(lib.ss_causal_conv1d_update(ctypes.byref(p), stream))
    return out


def device_error(clear: bool = False) -> int:
    """The library's device error word on the current device (0 = none)."""
    w = ctypes.c_int32(0)
    _check(load_library().ss_device_error(ctypes.byref(w), int(bool(clear))))
    return int(w.value)
