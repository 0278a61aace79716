"""Seeded synthetic inputs for the selective-scan forward.

This module only draws numbers; it holds none of the scan's arithmetic. Both
the CUDA path's tests/bench and the fp64 oracle consume what it produces, so it
imports nothing from either.

Draws use numpy's PCG64 generator (``numpy.random.default_rng(seed)``), whose
stream is fixed by numpy's stability policy, in float32, in the fixed order
B, C, u, delta, z, D, dt0; A is deterministic. Values are then cast once
(round-to-nearest-even) to the stored dtype; both sides read the stored values.

Readings of the workload recipes:
  * N(mu, s): s is the standard deviation.
  * "delta_bias = inverse-softplus of U(a, b)": dt0 ~ U(a, b) per channel
    (uniform), bias = log(expm1(dt0)), so softplus(bias) = dt0.
  * A[d, n] = -(n + 1) for every channel (real S4D initialisation).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

_TORCH_DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    dim: int
    seqlen: int
    dstate: int
    groups: int = 1            # variable B/C: number of groups (4-D form); 1 = 3-D form
    bc: str = "variable"       # "variable" | "fixed"
    dtype: str = "fp32"        # u, delta, z, out
    bc_dtype: Optional[str] = None  # variable B/C dtype (default: dtype); fixed is fp32
    bc_std: float = 1.0
    delta_std: float = 1.0
    has_z: bool = True
    D_mode: str = "normal"     # "normal" N(1, 0.1) | "ones" | "none"
    dt_range: tuple = (0.001, 0.1)
    has_bias: bool = True
    delta_softplus: bool = True
    return_last_state: bool = False
    bc_4d: bool = False        # store variable B/C as (b, g, n, l) even when g == 1
    seed: int = 0

    @property
    def elems(self) -> int:
        return self.batch * self.dim * self.seqlen

    def bc_stored_dtype(self) -> str:
        return "fp32" if self.bc == "fixed" else (self.bc_dtype or self.dtype)


# The five workloads the measurements are quoted on (Mamba-layer shapes).
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 16, 64, 4, dtype="fp32", delta_std=0.5,
                          has_z=False, return_last_state=True, seed=0),
    "mamba130m_bf16": Workload("mamba130m_bf16", 8, 1536, 2048, 16, dtype="bf16", seed=1),
    "grouped_bf16": Workload("grouped_bf16", 4, 4096, 4096, 16, groups=4, bc_4d=True,
                             dtype="bf16", return_last_state=True, seed=2),
    "mamba2p8b_fp16": Workload("mamba2p8b_fp16", 2, 5120, 8192, 16, dtype="fp16", seed=3),
    "long_fixed_fp32": Workload("long_fixed_fp32", 1, 2048, 65536, 16, bc="fixed", dtype="fp32",
                                bc_std=1.0 / 16, delta_std=0.5, has_z=False, D_mode="ones",
                                dt_range=(0.001, 0.01), return_last_state=True, seed=4),
    # the 130M-shaped layer on a sequence length with no 16-byte row stride (a
    # typical prompt length): the rows cannot be described to TMA, so the
    # forward streams them with plain loads
    "mamba130m_bf16_l2047": Workload("mamba130m_bf16_l2047", 8, 1536, 2047, 16, dtype="bf16", seed=5),
}


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(_TORCH_DTYPES[dtype])


def make_inputs(w: Workload) -> dict:
    """CPU tensors in their stored dtypes: u, delta, A, B, C, D, z, delta_bias
    (absent operands are None) plus the flags."""
    rng = np.random.default_rng(w.seed)
    f32 = np.float32
    b, d, l, n, g = w.batch, w.dim, w.seqlen, w.dstate, w.groups
    if w.bc == "fixed":
        bc_shape = (d, n)
    elif g == 1 and not w.bc_4d:
        bc_shape = (b, n, l)
    else:
        bc_shape = (b, g, n, l)
    Bf = rng.standard_normal(bc_shape, dtype=f32) * f32(w.bc_std)
    Cf = rng.standard_normal(bc_shape, dtype=f32) * f32(w.bc_std)
    uf = rng.standard_normal((b, d, l), dtype=f32)
    deltaf = rng.standard_normal((b, d, l), dtype=f32) * f32(w.delta_std)
    zf = rng.standard_normal((b, d, l), dtype=f32) if w.has_z else None
    if w.D_mode == "normal":
        Df = rng.standard_normal(d, dtype=f32) * f32(0.1) + f32(1.0)
    elif w.D_mode == "ones":
        Df = np.ones(d, f32)
    else:
        Df = None
    if w.has_bias:
        dt0 = rng.uniform(w.dt_range[0], w.dt_range[1], size=d)  # float64
        biasf = np.log(np.expm1(dt0)).astype(f32)
    else:
        biasf = None
    Af = -np.tile(np.arange(1, n + 1, dtype=f32), (d, 1))
    bcdt = w.bc_stored_dtype()
    return dict(
        u=_cast(uf, w.dtype), delta=_cast(deltaf, w.dtype),
        A=torch.from_numpy(Af), B=_cast(Bf, bcdt), C=_cast(Cf, bcdt),
        D=None if Df is None else torch.from_numpy(Df),
        z=None if zf is None else _cast(zf, w.dtype),
        delta_bias=None if biasf is None else torch.from_numpy(biasf),
        delta_softplus=w.delta_softplus, return_last_state=w.return_last_state,
    )


def compulsory_bytes(w: Workload) -> int:
    """Bytes the operation must move at least once: u, delta, (z), out at the
    stored dtype; B/C once per (batch, group) or once if fixed; A, D, bias;
    last_state in fp32."""
    s = torch.tensor([], dtype=_TORCH_DTYPES[w.dtype]).element_size()
    sbc = torch.tensor([], dtype=_TORCH_DTYPES[w.bc_stored_dtype()]).element_size()
    per_elem = s * (3 + (1 if w.has_z else 0))
    total = per_elem * w.elems
    if w.bc == "fixed":
        total += 2 * w.dim * w.dstate * sbc
    else:
        total += 2 * w.batch * w.groups * w.dstate * w.seqlen * sbc
    total += w.dim * w.dstate * 4
    total += w.dim * 4 * ((1 if w.D_mode != "none" else 0) + (1 if w.has_bias else 0))
    if w.return_last_state:
        total += 4 * w.batch * w.dim * w.dstate
    return total


def make_dout(w: Workload, seed: Optional[int] = None) -> torch.Tensor:
    """The upstream gradient for the backward: dout ~ N(0, 1) of u's shape,
    drawn with PCG64 from seed (default w.seed + 1000), stored in w.dtype."""
    rng = np.random.default_rng(w.seed + 1000 if seed is None else seed)
    return _cast(rng.standard_normal((w.batch, w.dim, w.seqlen), dtype=np.float32), w.dtype)


def backward_compulsory_bytes(w: Workload) -> int:
    """Bytes the backward must move at least once: u, delta, (z), dout read and
    du, ddelta, (dz) written at the stored dtype; B/C read once and dB/dC
    written once in fp32 (per (batch, group), or per channel if fixed); A, D,
    bias read and dA, dD, ddelta_bias written in fp32."""
    s = torch.tensor([], dtype=_TORCH_DTYPES[w.dtype]).element_size()
    sbc = torch.tensor([], dtype=_TORCH_DTYPES[w.bc_stored_dtype()]).element_size()
    total = s * (5 + (2 if w.has_z else 0)) * w.elems
    nbc = w.dim * w.dstate if w.bc == "fixed" else w.batch * w.groups * w.dstate * w.seqlen
    total += 2 * nbc * (sbc + 4)
    total += 2 * w.dim * w.dstate * 4
    total += 2 * w.dim * 4 * ((1 if w.D_mode != "none" else 0) + (1 if w.has_bias else 0))
    return total


# ---------------------------------------------------------------------------
# Decode step (one token per sequence against a resident state)
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    groups: int = 1            # B/C (batch, groups, dstate); 1 = (batch, dstate)
    dtype: str = "bf16"        # u, delta, z, out and B/C
    seed: int = 0

    @property
    def channels(self) -> int:
        return self.batch * self.dim


# Decode shapes of the same two Mamba layers (dim 1536 and 5120, dstate 16),
# with batches large enough that one step streams tens of MB of state.
DECODE_WORKLOADS = {
    "decode130m_bf16": DecodeWorkload("decode130m_bf16", 256, 1536, 16, dtype="bf16", seed=11),
    "decode2p8b_fp16": DecodeWorkload("decode2p8b_fp16", 64, 5120, 16, dtype="fp16", seed=12),
}


def make_decode_inputs(w: DecodeWorkload) -> dict:
    """CPU tensors for one decode step, drawn in the order state, B, C, u,
    delta, z, D, dt0 (same recipes as the forward workloads; the state is
    N(0, 1)): state fp32 (b, d, n); u, delta, z (b, d) and B, C (b, [g,] n)
    in the stored dtype; A, D, delta_bias fp32."""
    rng = np.random.default_rng(w.seed)
    f32 = np.float32
    b, d, n, g = w.batch, w.dim, w.dstate, w.groups
    st = rng.standard_normal((b, d, n), dtype=f32)
    bc_shape = (b, n) if g == 1 else (b, g, n)
    Bf = rng.standard_normal(bc_shape, dtype=f32)
    Cf = rng.standard_normal(bc_shape, dtype=f32)
    uf = rng.standard_normal((b, d), dtype=f32)
    deltaf = rng.standard_normal((b, d), dtype=f32)
    zf = rng.standard_normal((b, d), dtype=f32)
    Df = rng.standard_normal(d, dtype=f32) * f32(0.1) + f32(1.0)
    dt0 = rng.uniform(0.001, 0.1, size=d)
    biasf = np.log(np.expm1(dt0)).astype(f32)
    Af = -np.tile(np.arange(1, n + 1, dtype=f32), (d, 1))
    return dict(state=torch.from_numpy(st), u=_cast(uf, w.dtype), delta=_cast(deltaf, w.dtype),
                A=torch.from_numpy(Af), B=_cast(Bf, w.dtype), C=_cast(Cf, w.dtype),
                D=torch.from_numpy(Df), z=_cast(zf, w.dtype), delta_bias=torch.from_numpy(biasf))


def decode_compulsory_bytes(w: DecodeWorkload) -> int:
    """Bytes one decode step must move: the fp32 state read and written,
    u, delta, z and out, B/C once per (batch, group), A, D and delta_bias."""
    s = torch.tensor([], dtype=_TORCH_DTYPES[w.dtype]).element_size()
    return (8 * w.batch * w.dim * w.dstate + 4 * s * w.batch * w.dim
            + 2 * s * w.batch * w.groups * w.dstate + 4 * w.dim * w.dstate + 8 * w.dim)


# ---------------------------------------------------------------------------
# Causal depthwise conv1d (the convolution in front of the scan)
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ConvWorkload:
    name: str
    batch: int
    dim: int
    seqlen: int
    width: int = 4
    dtype: str = "bf16"
    seed: int = 0

    @property
    def elems(self) -> int:
        return self.batch * self.dim * self.seqlen


# The two Mamba layers' convolutions (same batch, channels and length as the
# forward workloads), width 4, silu activation, with bias.
CONV_WORKLOADS = {
    "conv130m_bf16": ConvWorkload("conv130m_bf16", 8, 1536, 2048, 4, "bf16", seed=21),
    "conv2p8b_fp16": ConvWorkload("conv2p8b_fp16", 2, 5120, 8192, 4, "fp16", seed=22),
}


def make_conv_inputs(w: ConvWorkload) -> dict:
    """x (b, d, l) in the stored dtype ~ N(0, 1); weight (d, width) fp32 ~
    N(0, 1) / sqrt(width); bias (d,) fp32 ~ N(0, 0.1); drawn in that order."""
    rng = np.random.default_rng(w.seed)
    f32 = np.float32
    xf = rng.standard_normal((w.batch, w.dim, w.seqlen), dtype=f32)
    wf = rng.standard_normal((w.dim, w.width), dtype=f32) * f32(1.0 / np.sqrt(w.width))
    bf = rng.standard_normal(w.dim, dtype=f32) * f32(0.1)
    return dict(x=_cast(xf, w.dtype), weight=torch.from_numpy(wf), bias=torch.from_numpy(bf))


def conv_compulsory_bytes(w: ConvWorkload) -> int:
    """x read and out written once, plus weight and bias."""
    s = torch.tensor([], dtype=_TORCH_DTYPES[w.dtype]).element_size()
    return 2 * s * w.elems + 4 * w.dim * w.width + 4 * w.dim
