"""Helpers of the GPU parity tests: run the CUDA path through the binding
(which calls the C ABI) with guard bytes around every output."""
import numpy as np
import torch

import cast_transpose_gb300 as ct

GUARD = 256          # bytes of canary on each side (keeps 16-byte alignment)
CANARY = 0xA5


class Guarded:
    """A device buffer of `n` bytes (or n fp32) between two canary zones."""

    def __init__(self, n, dtype=torch.uint8, offset=0, device="cuda"):
        esz = torch.empty(0, dtype=dtype).element_size()
        g = GUARD // esz
        self.g, self.n, self.off = g, n, offset
        self.buf = torch.empty(n + 2 * g + offset, dtype=dtype, device=device)
        self.buf.view(torch.uint8).fill_(CANARY)
        self.t = self.buf[g + offset: g + offset + n]

    def check(self):
        b = self.buf.view(torch.uint8).cpu().numpy()
        esz = self.buf.element_size()
        head = b[: (self.g + self.off) * esz]
        tail = b[(self.g + self.off + self.n) * esz:]
        assert np.all(head == CANARY) and np.all(tail == CANARY), "canary overwritten"

    def numpy(self):
        return self.t.cpu().numpy()


def scalar(v, device="cuda"):
    return torch.tensor([v], dtype=torch.float32, device=device)


def f32_bits(v) -> int:
    return int(np.array([v], dtype=np.float32).view(np.uint32)[0])


def cast_transpose_gpu(x: torch.Tensor, scale: float, fmt: int, amax_in: float = 0.0,
                       out_offset: int = 0, noop=None):
    rows, cols = x.shape
    n = rows * cols
    q = Guarded(n, offset=out_offset)
    qt = Guarded(n, offset=out_offset)
    s = scalar(scale)
    a = scalar(amax_in)
    si = scalar(-1.0)
    ct.fp8_cast_transpose(x, s, a, si, q.t, qt.t, fmt, noop_flag=noop)
    torch.cuda.synchronize()
    q.check()
    qt.check()
    return {"q": q.numpy().reshape(rows, cols), "qt": qt.numpy().reshape(cols, rows),
            "amax": a.item(), "scale_inv": si.item()}


def assert_same_cast(got: dict, ref: dict):
    assert got["q"].shape == ref["q"].shape
    bad = np.argwhere(got["q"] != ref["q"])
    assert bad.size == 0, f"{len(bad)} FP8 bytes differ, first at {bad[:4].tolist()}"
    assert np.array_equal(got["qt"], ref["qt"]), "transpose differs"
    assert f32_bits(got["amax"]) == f32_bits(ref["amax"]), (got["amax"], ref["amax"])
    assert f32_bits(got["scale_inv"]) == f32_bits(ref["scale_inv"])


def dbias_tolerance_ok(db: np.ndarray, ref: np.ndarray, x_cpu: torch.Tensor) -> bool:
    col_abs = x_cpu.double().abs().sum(dim=0).numpy()
    return bool(np.all(np.abs(db.astype(np.float64) - ref.astype(np.float64))
                       <= 1e-5 * col_abs + 1e-6))
