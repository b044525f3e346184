"""Reader for the hand-worked fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FMT = {"E4M3": 0, "E5M2": 1}


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def read_cast(name):
    out = {"x": [], "q": []}
    for tok in _lines(name):
        key, vals = tok[0], tok[1:]
        if key == "fmt":
            out["fmt"] = FMT[vals[0]]
        elif key in ("scale", "amax", "scale_inv"):
            out[key] = np.float32(float(vals[0]))
        elif key == "x":
            out["x"].append([float(v) for v in vals])
        elif key == "q":
            out["q"].append([int(v, 16) for v in vals])
    out["x"] = np.array(out["x"], dtype=np.float32)
    out["q"] = np.array(out["q"], dtype=np.uint8)
    return out


def read_update(name):
    out = {"steps": []}
    for tok in _lines(name):
        key, vals = tok[0], tok[1:]
        if key == "fmt":
            out["fmt"] = FMT[vals[0]]
        elif key in ("L", "margin"):
            out[key] = int(vals[0])
        elif key == "init_scale":
            out["init_scale"] = np.array([float(v) for v in vals], dtype=np.float32)
        elif key == "step":
            arrow = vals.index("->")
            amax = np.array([float(v) for v in vals[:arrow]], dtype=np.float32)
            scale = np.array([float(v) for v in vals[arrow + 1:]], dtype=np.float32)
            out["steps"].append((amax, scale))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns of fp32 values that must already be exact in bf16."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "fixture value not exact in bf16"
    return (bits >> 16).astype(np.uint16)
