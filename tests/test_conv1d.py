"""GPU parity of the causal depthwise conv1d (page "PaddleNLP Kernel 算子库：CUDA 与
Triton 双实现的高性能 NLP GPU 算子实战指南", section 4.2, causal_conv1d_fn) and its
one-step update against the fp64 oracle, on seeded inputs.

Tolerance: max|gpu - oracle| / max|oracle| <= 1e-5 for fp32, <= 1e-2 for
fp16/bf16 (outputs are rounded once to the input dtype); states are copies of
inputs and must match exactly.
"""
import numpy as np
import pytest
import torch

from oracle import conv1d as ref
from state_space_model_03_gb300 import api

pytestmark = pytest.mark.gpu

TDT = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}
TOL = {"fp32": 1e-5, "fp16": 1e-2, "bf16": 1e-2}


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _inputs(b, d, l, w, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(b, d, l, generator=g).to(TDT[dtype])
    weight = torch.randn(d, w, generator=g) * 0.5
    bias = torch.randn(d, generator=g)
    return x, weight, bias


CASES = [
    # (batch, dim, seqlen, width, dtype)
    (2, 64, 2048, 4, "bf16"),
    (3, 40, 1000, 4, "fp16"),
    (1, 33, 4099, 3, "fp32"),
    (2, 16, 8200, 2, "bf16"),
    (1, 8, 5, 4, "fp32"),         # shorter than a thread's steps
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[4]}_b{c[0]}d{c[1]}l{c[2]}w{c[3]}")
@pytest.mark.parametrize("act", [None, "silu"])
def test_conv1d_matches_oracle(case, act):
    b, d, l, w, dtype = case
    x, weight, bias = _inputs(b, d, l, w, dtype, 11 + l + w)
    out = api.causal_conv1d_fn(x.cuda(), weight.cuda(), bias.cuda(), activation=act)
    torch.cuda.synchronize()
    assert _rel(_np(out), ref.causal_conv1d_ref(x, weight, bias, activation=act)) <= TOL[dtype]


def test_conv1d_views_without_bias():
    """Rows of a strided view (no 16-byte vector path) and no bias."""
    x, weight, _ = _inputs(2, 24, 333, 4, "bf16", 3)
    big = torch.zeros(2, 24, 340, dtype=torch.bfloat16)
    big[:, :, 3:336] = x
    xv = big.cuda()[:, :, 3:336]
    out = api.causal_conv1d_fn(xv, weight.cuda(), activation="swish")
    torch.cuda.synchronize()
    assert _rel(_np(out), ref.causal_conv1d_ref(x, weight, activation="swish")) <= 1e-2


@pytest.mark.parametrize("l", [1, 2, 3, 700])
def test_conv1d_initial_and_final_states(l):
    b, d, w = 2, 48, 4
    x, weight, bias = _inputs(b, d, l, w, "fp32", 21 + l)
    init = torch.randn(b, d, w - 1, generator=torch.Generator().manual_seed(l))
    out, fin = api.causal_conv1d_fn(x.cuda(), weight.cuda(), bias.cuda(), initial_states=init.cuda(),
                                    return_final_states=True, activation="silu")
    torch.cuda.synchronize()
    ro, rf = ref.causal_conv1d_ref(x, weight, bias, initial_states=init, return_final_states=True, activation="silu")
    assert _rel(_np(out), ro) <= 1e-5
    assert np.array_equal(_np(fin), rf)


def test_conv1d_empty_sequence_final_states():
    x = torch.empty(2, 8, 0, device="cuda")
    weight = torch.randn(8, 4, device="cuda")
    init = torch.randn(2, 8, 3, device="cuda")
    out, fin = api.causal_conv1d_fn(x, weight, initial_states=init, return_final_states=True)
    torch.cuda.synchronize()
    assert out.shape == (2, 8, 0) and torch.equal(fin, init)


def test_conv1d_packed_sequences():
    b, d, l, w = 2, 32, 3000, 4
    x, weight, bias = _inputs(b, d, l, w, "bf16", 31)
    seq = torch.zeros(b, l, dtype=torch.int32)
    seq[0, 1000:] = 1
    seq[0, 1001:] = 2
    seq[0, 2047:] = 3
    seq[1, 5:] = 1
    out = api.causal_conv1d_fn(x.cuda(), weight.cuda(), bias.cuda(), seq_idx=seq.cuda(), activation="silu")
    torch.cuda.synchronize()
    assert _rel(_np(out), ref.causal_conv1d_ref(x, weight, bias, seq_idx=seq.numpy(), activation="silu")) <= 1e-2
    with pytest.raises((api.SSError, ValueError)):
        api.causal_conv1d_fn(x.cuda(), weight.cuda(), seq_idx=seq.cuda(), return_final_states=True)


def test_conv1d_activation_rules():
    x, weight, _ = _inputs(1, 8, 16, 4, "fp32", 41)
    with pytest.raises(NotImplementedError):
        api.causal_conv1d_fn(x.cuda(), weight.cuda(), activation="relu")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("w", [2, 4])
def test_conv1d_update_chains_to_the_sequence(dtype, w):
    """l decode steps from a zero state reproduce the sequence and end in its
    final states."""
    b, d, l = 3, 100, 9
    x, weight, bias = _inputs(b, d, l, w, dtype, 51 + w)
    ro, rf = ref.causal_conv1d_ref(x, weight, bias, return_final_states=True, activation="silu")
    st = torch.zeros(b, d, w - 1, dtype=TDT[dtype], device="cuda")
    xc, wc, bc = x.cuda(), weight.cuda(), bias.cuda()
    outs = [api.causal_conv1d_update(xc[:, :, t], st, wc, bc, activation="silu") for t in range(l)]
    torch.cuda.synchronize()
    assert _rel(_np(torch.stack(outs, dim=2)), ro) <= TOL[dtype]
    assert np.array_equal(_np(st), rf)
