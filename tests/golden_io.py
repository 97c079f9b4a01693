"""Reader for ``tests/golden/oracle_small.json`` (storage bits as hex)."""
import json
import os

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_small.json")


def unhex(s, dtype, shape):
    vals = [int(v, 16) for v in s.split()]
    if dtype == "f32":
        return np.array(vals, np.uint32).view(np.float32).reshape(shape)
    return np.array(vals, np.uint16).reshape(shape)


def cases():
    """Yield dicts with numpy inputs and expected outputs."""
    with open(PATH) as f:
        data = json.load(f)
    for c in data["cases"]:
        dt, T, H, R = c["dtype"], c["T"], c["H"], c["R"]
        shapes = {"x": (T, H), "residual": (T, H), "partials": (R, T, H), "gamma": (H,)}
        inp = {k: unhex(v, dt, shapes[k]) for k, v in c["inputs"].items()}
        out = {"y": unhex(c["y"], dt, (T, H))}
        if c["residual_out"] is not None:
            out["residual"] = unhex(c["residual_out"], dt, (T, H))
        yield dict(c, inputs=inp, expected=out)
