"""Write ``oracle_small.json``: small problems with the oracle's outputs.

Calls only the CPU oracle (``oracle/``) and the seeded input generator.  The
file stores inputs and outputs as storage bits, so a check needs neither the
generator nor a particular platform's maths library: it pins the oracle built
on one machine (x86-64) against the same source built on another (aarch64),
and gives the GPU tests fixed expected values.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from residual_add_rmsnorm_gb300 import workloads as W  # noqa: E402

CASES = [
    ("rms_norm", "f32", 3, 37, 0, 1e-6),
    ("rms_norm", "f16", 2, 72, 0, 1e-5),
    ("rms_norm", "bf16", 2, 129, 0, 1e-6),
    ("fused_add_rms_norm", "f32", 2, 40, 1, 1e-6),
    ("fused_add_rms_norm", "f16", 3, 33, 1, 1e-5),
    ("fused_add_rms_norm", "bf16", 2, 64, 1, 1e-6),
    ("reduce_add_rms_norm", "bf16", 2, 24, 8, 1e-6),
    ("reduce_add_rms_norm", "f16", 2, 17, 3, 1e-5),
    ("reduce_add_rms_norm", "f32", 1, 16, 2, 1e-6),
]


def hexbits(a, dtype):
    a = np.ascontiguousarray(a)
    u = a.view(np.uint32) if dtype == "f32" else a.view(np.uint16)
    width = 8 if dtype == "f32" else 4
    return " ".join(f"{int(v):0{width}x}" for v in u.ravel())


def main():
    out = []
    for op, dt, T, H, R, eps in CASES:
        w = W.workload(op, dt, T, H, R=R, eps=eps, seed=11)
        d = W.generate(w)
        if op == "rms_norm":
            r = oracle.rms_norm(d["x"], d["gamma"], eps, dt)
        elif op == "fused_add_rms_norm":
            r = oracle.fused_add_rms_norm(d["x"], d["residual"], d["gamma"], eps, dt)
        else:
            r = oracle.reduce_add_rms_norm(d["partials"], d["residual"], d["gamma"], eps, dt)
        case = {"op": op, "dtype": dt, "T": T, "H": H, "R": R, "eps": eps,
                "inputs": {k: hexbits(v, dt) for k, v in d.items()},
                "y": hexbits(r.y, dt),
                "residual_out": None if r.residual is None else hexbits(r.residual, dt)}
        out.append(case)
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump({"source": "tests/golden/make_golden.py (CPU oracle only)", "cases": out}, f,
                  indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
