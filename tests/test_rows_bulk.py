"""Rows that TMA cannot describe (sequence lengths whose rows are not 16-byte
multiples, views at odd offsets): the forward's producer copies the 16-byte
blocks that cover each row (reading only inside the tensor, loading the ends of
a tensor's first and last rows itself), the element warps read the rows at
their byte offset, B/C rows are shifted into their tiles, and out rows that
are not 16-byte aligned are stored as aligned 16-byte blocks, each lane forming
its blocks from its own piece and the 16 bytes before it. The plain-load
producer (SSFWD_NO_BULK) builds the same tiles, so the two give identical
results, and both match the oracle."""
import ctypes

import pytest
import torch

from state_space_model_03_gb300 import api, workloads

from test_parity import NAMES, _check_full, _to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # (batch, dim, seqlen, dstate, groups, bc, dtype, bc_dtype, z)
    (2, 37, 2047, 16, 1, "variable", "bf16", None, True),    # 130M-like rows, ragged channel tile
    (1, 40, 1001, 16, 2, "variable", "fp16", None, True),    # fp32 B/C hand-off, two groups
    (1, 33, 999, 16, 1, "variable", "fp32", None, False),
    (2, 48, 191, 16, 1, "variable", "bf16", "fp32", True),   # fp32 B/C rows of 256 bytes (two pieces)
    (1, 36, 201, 32, 2, "variable", "fp16", "fp32", True),   # 64 B/C pieces per tensor: two batches
    (1, 20, 131, 64, 1, "variable", "bf16", None, True),     # 64 B/C rows: two batches
    (1, 40, 333, 3, 1, "fixed", "fp16", None, True),
    (1, 40, 501, 16, 1, "fixed", "fp32", None, False),
    (2, 40, 9, 16, 1, "variable", "bf16", None, True),       # pieces of 18 bytes: some without an interior
    (1, 24, 1, 16, 1, "variable", "bf16", None, True),
    (1, 64, 20001, 16, 1, "variable", "bf16", None, True),   # few CTAs: split sequence (summary pass too)
    (2, 40, 1001, 16, 2, "variable", "bf16", None, True),    # odd out rows: a CTA's rows cross a group end
    (3, 72, 517, 16, 3, "variable", "bf16", None, False),    # the same, three groups, no gate
]


def _launch(dev, x, capfd):
    capfd.readouterr()
    res = api.selective_scan_fn(**dev, delta_softplus=x["delta_softplus"], return_last_state=x["return_last_state"])
    torch.cuda.synchronize()
    lines = [ln for ln in capfd.readouterr().err.splitlines() if ln.startswith("ssfwd:")]
    out, last = res if isinstance(res, tuple) else (res, None)
    return out, last, lines


@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}-{c[5]}-b{c[0]}d{c[1]}l{c[2]}n{c[3]}g{c[4]}" for c in CASES])
def test_bulk_rows_match_plain_loads_and_oracle(case, capfd, monkeypatch):
    b, d, l, n, g, bc, dt, bcdt, z = case
    w = workloads.Workload("bulk", b, d, l, n, groups=g, bc=bc, dtype=dt, bc_dtype=bcdt, has_z=z,
                           return_last_state=True, bc_4d=g > 1, seed=3000 + l + n)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    monkeypatch.setenv("SSFWD_DEBUG", "1")
    out, last, rep = _launch(dev, x, capfd)
    assert rep and all(r.split()[1] == "generic-bulk" for r in rep), rep
    assert api.device_error() == 0
    monkeypatch.setenv("SSFWD_NO_BULK", "1")
    out_p, last_p, rep_p = _launch(dev, x, capfd)
    assert rep_p and all(r.split()[1] == "generic" for r in rep_p), rep_p
    assert torch.equal(out, out_p) and torch.equal(last, last_p)
    _check_full(w, x, out, last)


@pytest.mark.parametrize("offset", [1, 3, 5, 8])
def test_views_at_every_alignment(offset, capfd, monkeypatch):
    """u / delta / z as views starting `offset` elements into wider rows (every
    row start alignment modulo 16 bytes occurs): same bits as the contiguous
    inputs on the TMA path."""
    w = workloads.Workload("views", 2, 24, 250, 16, dtype="bf16", return_last_state=True, seed=40 + offset)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    ref_out, ref_last = api.selective_scan_fn(**dev, delta_softplus=True, return_last_state=True)
    wide = 250 + 13
    v = dict(dev)
    for k in ("u", "delta", "z"):
        t = torch.full((2, 24, wide), float("nan"), dtype=dev[k].dtype, device="cuda")
        t[:, :, offset:offset + 250] = dev[k]
        v[k] = t[:, :, offset:offset + 250]
    monkeypatch.setenv("SSFWD_DEBUG", "1")
    out, last, rep = _launch(v, x, capfd)
    assert rep and rep[-1].split()[1] == "generic-bulk", rep
    assert torch.equal(out, ref_out) and torch.equal(last, ref_last)


@pytest.mark.parametrize("pitch", [2048, 2047 + 9])
def test_odd_rows_into_other_out_pitches(pitch):
    """Rows TMA cannot describe written into an out tensor whose rows have
    another pitch (16-byte aligned: vector stores; not: aligned blocks formed
    across each row's lanes): the same bits as a contiguous out."""
    w = workloads.Workload("pitch", 2, 48, 2047, 16, dtype="bf16", return_last_state=True, seed=77)
    x = workloads.make_inputs(w)
    dev = _to_dev(x)
    nu = api.normalise(*(dev[k] for k in NAMES))
    lib = api.load_library()
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for pt in (2047, pitch):
        big = torch.full((2, 48, pt), float("nan"), dtype=torch.bfloat16, device="cuda")
        out = big[:, :, :2047]
        last = torch.empty(2, 48, 16, device="cuda")
        prm = api.make_params(*nu, True, out, last)
        ws = api.attach_workspace(prm, out.device)
        assert lib.ss_fwd(ctypes.byref(prm), s) == 0
        torch.cuda.synchronize()
        assert api.device_error() == 0
        if pt > 2047:
            assert torch.isnan(big[:, :, 2047:].float()).all()  # the padding is never written
        outs.append((out.clone(), last.clone()))
        del ws
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
