"""Writes the stored oracle fixtures of tests/golden/:

- tiny_fp32_oracle.json: the fp64 forward oracle's output on the seeded tiny
  fp32 workload (batch 1, dim 16, seqlen 64, dstate 4), plus the first input
  draws so that a change of the generator's stream is caught;
- tiny_fp32_bwd_oracle.json: the fp64 backward oracle's gradients on the same
  workload with the seeded upstream gradient dout.

It calls only the oracles and the seeded input generator, never the CUDA
library. Regenerate with:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import backward as bwd_oracle  # noqa: E402
from state_space_model_03_gb300 import workloads  # noqa: E402


def main():
    w = workloads.WORKLOADS["tiny_fp32"]
    x = workloads.make_inputs(w)
    out, last = oracle.selective_scan_ref(
        x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
        delta_bias=x["delta_bias"], delta_softplus=True, return_last_state=True)
    doc = {
        "what": "fp64 oracle output on the seeded tiny fp32 workload",
        "workload": w.name, "seed": w.seed,
        "shape": [w.batch, w.dim, w.seqlen, w.dstate],
        "inputs_head": {k: [float(v) for v in x[k].reshape(-1)[:6].tolist()]
                        for k in ("u", "delta", "B", "C", "D", "delta_bias")},
        "out": [repr(float(v)) for v in out.reshape(-1)],
        "last_state": [repr(float(v)) for v in last.reshape(-1)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", path)

    dout = workloads.make_dout(w)
    g = bwd_oracle.selective_scan_bwd_ref(dout, x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                          delta_bias=x["delta_bias"], delta_softplus=True)
    doc = {
        "what": "fp64 backward oracle gradients of sum(dout * out) on the seeded tiny fp32 workload",
        "workload": w.name, "seed": w.seed, "dout_seed": w.seed + 1000,
        "dout_head": [float(v) for v in dout.reshape(-1)[:6].tolist()],
        "grads": {k: [repr(float(v)) for v in g[k].reshape(-1)] for k in sorted(g) if g[k] is not None},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_bwd_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
