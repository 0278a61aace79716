"""fp64 CPU oracle for the selective-scan forward.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg may import this module; the product path never does. It shares
no code with the CUDA library and imports nothing from the product package.

The arithmetic lives in ``ss_oracle.c`` (plain sequential fp64, one
(batch, channel) row at a time; see that file's header for the definition it
follows: operands of the page "PaddleNLP Kernel 算子库：CUDA 与 Triton 双实现的
高性能 NLP GPU 算子实战指南", section 4.1). This module only compiles it with gcc,
widens the stored inputs exactly to fp64 and hands rows to it, optionally on
several host threads (rows are independent, so the result does not depend on
the thread count).

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(brute-force unrolling, closed-form geometric sum, LTI convolution against
numpy.convolve, B = 0, linearity, causality, last_state, B/C-mode
equivalences, softplus/silu against torch) and, for the start state and the
one-step update, by ``tests/test_oracle_state.py``.

The other operators have oracles of their own, each pinned by its test file:
``oracle.backward`` (the gradients; ``tests/test_oracle_bwd.py``),
``oracle.complex_a`` (complex A; ``tests/test_oracle_complex.py``) and
``oracle.conv1d`` (the causal conv1d; ``tests/test_oracle_conv.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libssoracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so the x86 and Arm
# builds round identically.
_CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c99", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ss_oracle.c into oracle/_build/libssoracle.so (gcc)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.ss_oracle_fwd
            i64, dp = ctypes.c_int64, ctypes.c_void_p
            f.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                          dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                          dp, dp, dp, i64, i64, dp]
            f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    """Exact widening of a stored tensor/array to a contiguous fp64 numpy array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (bf16 has no numpy dtype)
        import torch
        return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _normalise_bc(B, C, dim):
    """B/C forms: 2-D (dim, dstate) fixed; 3-D (batch, dstate, seqlen) = 4-D with
    one group; 4-D (batch, groups, dstate, seqlen)."""
    if B.ndim == 2:
        return B, C, True, 1
    if B.ndim == 3:
        B, C = B[:, None], C[:, None]
    return np.ascontiguousarray(B), np.ascontiguousarray(C), False, B.shape[1]


def selective_scan_ref(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=False, return_last_state=False, threads=1,
                       initial_state=None):
    """Whole-problem fp64 reference. Returns out (b, d, l) fp64 numpy, and
    last_state (b, d, n) fp64 when return_last_state. initial_state (b, d, n),
    if given, is the state before the first step (else zero)."""
    u, delta, A, B, C = (_f64(t) for t in (u, delta, A, B, C))
    D, z, delta_bias = _f64(D), _f64(z), _f64(delta_bias)
    x0 = _f64(initial_state)
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    B, C, fixed, ngroups = _normalise_bc(B, C, dim)
    out = np.empty((batch, dim, seqlen), np.float64)
    last = np.empty((batch, dim, dstate), np.float64) if return_last_state else None
    lib = _load()
    nrows = batch * dim

    def run(r0, r1):
        scratch = np.empty(dstate, np.float64)
        rc = lib.ss_oracle_fwd(batch, dim, seqlen, dstate, ngroups, int(fixed),
                               _ptr(u), _ptr(delta), _ptr(z), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(delta_bias), int(bool(delta_softplus)),
                               _ptr(x0), _ptr(out), _ptr(last), r0, r1, _ptr(scratch))
        if rc != 0:
            raise ValueError("oracle: bad shape")

    threads = max(1, min(int(threads), nrows)) if nrows else 1
    if threads == 1 or nrows == 0:
        run(0, nrows)
    else:
        bounds = np.linspace(0, nrows, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as ex:  # ctypes releases the GIL
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return (out, last) if return_last_state else out


def selective_scan_rows(rows, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                        delta_softplus=False, threads=1):
    """fp64 reference for selected (b, d) rows only, each solved as its own
    one-row problem. Returns (out_rows (R, l), last_rows (R, n)) fp64."""
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    fixed = B.ndim == 2
    ngroups = 1 if B.ndim <= 3 else B.shape[1]
    dpg = dim // ngroups
    R = len(rows)
    out = np.empty((R, seqlen), np.float64)
    last = np.empty((R, dstate), np.float64)

    def one(i):
        b, d = rows[i]
        if fixed:
            Bi, Ci = B[d:d + 1], C[d:d + 1]
        elif B.ndim == 3:
            Bi, Ci = B[b:b + 1, None], C[b:b + 1, None]
        else:
            g = d // dpg
            Bi, Ci = B[b:b + 1, g:g + 1], C[b:b + 1, g:g + 1]
        o, s = selective_scan_ref(
            u[b:b + 1, d:d + 1], delta[b:b + 1, d:d + 1], A[d:d + 1], Bi, Ci,
            None if D is None else D[d:d + 1], None if z is None else z[b:b + 1, d:d + 1],
            None if delta_bias is None else delta_bias[d:d + 1],
            delta_softplus, True, threads=1)
        out[i] = o[0, 0]
        last[i] = s[0, 0]

    if threads <= 1:
        for i in range(R):
            one(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(R)))
    return out, last


def selective_state_update_ref(state, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                               delta_softplus=False, bc_fixed=False):
    """One step of the same recurrence for every (batch, channel), in plain
    numpy fp64, written independently of ``ss_oracle.c`` (the decode step the
    page lists as "selective_state_update"; it prints no signature, so the
    operands are the scan's at a single time step):

      state (b, d, n), u, delta, z (b, d), A (d, n), D, delta_bias (d,),
      B, C per token (b, n) or grouped (b, g, n); with bc_fixed, (d, n).
      dt = softplus(delta + delta_bias) (or the sum itself),
      state' = exp(dt A) state + dt B u,  y = sum_n C state' + D u,
      out = y silu(z) when z is given.

    Returns (out (b, d), new state (b, d, n)) as fp64 arrays; the input state
    is not modified."""
    x = _f64(state)
    u, delta, A, B, C = (_f64(t) for t in (u, delta, A, B, C))
    D, z, delta_bias = _f64(D), _f64(z), _f64(delta_bias)
    batch, dim = u.shape
    v = delta + (delta_bias[None, :] if delta_bias is not None else 0.0)
    if delta_softplus:
        dt = np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v)))
    else:
        dt = v
    if bc_fixed:
        Bd, Cd = B[None, :, :], C[None, :, :]          # per channel
    else:
        if B.ndim == 2:                                 # (b, n): one group
            B, C = B[:, None, :], C[:, None, :]
        g = B.shape[1]
        grp = np.arange(dim) // (dim // g)
        Bd, Cd = B[:, grp, :], C[:, grp, :]             # (b, d, n)
    x = np.exp(dt[:, :, None] * A[None, :, :]) * x + (dt * u)[:, :, None] * Bd
    y = np.sum(Cd * x, axis=2)
    if D is not None:
        y = y + D[None, :] * u
    if z is not None:
        y = y * (z / (1.0 + np.exp(-z)))
    return y, x
