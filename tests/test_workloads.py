"""The seeded generator and the stored oracle fixture (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from state_space_model_03_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_fp32_oracle.json")


def test_golden_tiny_oracle():
    """Oracle output on the tiny workload equals the committed fixture (written
    by tests/golden/make_golden.py, which calls only the oracle). libm's exp
    and log1p may differ by an ulp between hosts, hence 1e-12 and not equality."""
    with open(GOLDEN) as f:
        doc = json.load(f)
    w = workloads.WORKLOADS["tiny_fp32"]
    x = workloads.make_inputs(w)
    for k, head in doc["inputs_head"].items():
        assert x[k].reshape(-1)[:6].tolist() == head, k
    out, last = oracle.selective_scan_ref(
        x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
        delta_bias=x["delta_bias"], delta_softplus=True, return_last_state=True)
    g_out = np.array([float(v) for v in doc["out"]])
    g_last = np.array([float(v) for v in doc["last_state"]])
    assert np.max(np.abs(out.reshape(-1) - g_out)) <= 1e-12 * np.max(np.abs(g_out))
    assert np.max(np.abs(last.reshape(-1) - g_last)) <= 1e-12 * np.max(np.abs(g_last))


@pytest.mark.parametrize("name", ["tiny_fp32"])
def test_shapes_dtypes_small(name):
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    assert x["u"].shape == (w.batch, w.dim, w.seqlen) and x["u"].dtype == torch.float32
    assert x["B"].shape == (w.batch, w.dstate, w.seqlen)
    assert x["z"] is None and x["return_last_state"]


def test_recipe_readings():
    """delta_bias is the inverse softplus of U(a, b); A = -(n + 1); draws are
    repeatable for a seed and differ across seeds."""
    w = workloads.Workload("t", 2, 64, 32, 8, dtype="bf16", seed=5)
    x = workloads.make_inputs(w)
    dt0 = torch.nn.functional.softplus(x["delta_bias"].double(), threshold=1e4)
    assert float(dt0.min()) >= 0.001 * (1 - 1e-5) and float(dt0.max()) <= 0.1 * (1 + 1e-5)
    assert torch.equal(x["A"][3], -torch.arange(1, 9, dtype=torch.float32))
    assert x["u"].dtype == torch.bfloat16 and x["B"].dtype == torch.bfloat16
    y = workloads.make_inputs(w)
    assert torch.equal(x["u"], y["u"]) and torch.equal(x["B"], y["B"])
    z = workloads.make_inputs(workloads.Workload("t", 2, 64, 32, 8, dtype="bf16", seed=6))
    assert not torch.equal(x["u"], z["u"])
    assert abs(float(x["D"].mean()) - 1.0) < 0.1


def test_compulsory_bytes_table():
    """Compulsory bytes of the five workloads (u, delta, z, out at the stored
    dtype; B/C once per (batch, group); A, D, bias; fp32 last_state)."""
    expect = {
        "tiny_fp32": 14976,
        "mamba130m_bf16": 202485760,
        "grouped_bf16": 542408704,
        "mamba2p8b_fp16": 672505856,
        "long_fixed_fp32": 1611153408,
    }
    for k, v in expect.items():
        assert workloads.compulsory_bytes(workloads.WORKLOADS[k]) == v, k


def test_dout_and_backward_bytes():
    """The backward's upstream gradient is seeded and shaped like u; the
    backward's compulsory bytes follow the formula in its docstring."""
    w = workloads.WORKLOADS["mamba130m_bf16"]
    small = workloads.Workload("s", 2, 8, 40, 16, dtype="bf16", seed=5)
    a, b = workloads.make_dout(small), workloads.make_dout(small)
    assert a.shape == (2, 8, 40) and a.dtype == torch.bfloat16 and torch.equal(a, b)
    assert not torch.equal(a, workloads.make_dout(small, seed=6))
    # u, delta, z, dout read and du, ddelta, dz written (2 bytes); B, C read (2) and dB, dC written (4);
    # A read and dA written; D, bias read and their gradients written
    want = (2 * 7 * 8 * 1536 * 2048 + 2 * 8 * 16 * 2048 * (2 + 4) + 2 * 1536 * 16 * 4 + 2 * 1536 * 4 * 2)
    assert workloads.backward_compulsory_bytes(w) == want
