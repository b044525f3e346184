"""Plain CPU oracle for the FP8 cast-transpose path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never loads it, and it shares no code with the CUDA sources: the
arithmetic lives in ``ct_oracle.c`` (plain scalar C, one thread), and this
module only compiles it with gcc and marshals numpy arrays.

Every function here follows the passage cited in ``ct_oracle.c``:
``[PyTorch] cuda graph support`` (DbiasCastTranspose example: ``db =
dy.sum(dim=0)`` next to ``cast_transpose(dy)`` with a transpose cache) and
``[PyTorch] Refactor FP8 workspaces in linear modules`` (Motivations: private
scale-inverse, scale update kernel, infinite-scale case), with the FP8
formats of the OCP OFP8 specification.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ct_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ct_oracle.c into _build/liboracle.so (if missing or stale)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            c = ctypes
            L.oracle_fp8_encode.restype = c.c_uint8
            L.oracle_fp8_encode.argtypes = [c.c_float, c.c_int]
            L.oracle_fp8_decode.restype = c.c_float
            L.oracle_fp8_decode.argtypes = [c.c_uint8, c.c_int]
            L.oracle_fp8_encode_array.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p]
            L.oracle_fp8_decode_array.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p]
            L.oracle_cast_transpose.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_float,
                                                c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
                                                c.c_void_p]
            L.oracle_amax.argtypes = [c.c_void_p, c.c_int64, c.c_void_p]
            L.oracle_dbias.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_void_p]
            L.oracle_fp8_transpose.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_void_p]
            L.oracle_f32_to_bf16_array.argtypes = [c.c_void_p, c.c_int64, c.c_void_p]
            L.oracle_amax_and_scale_update.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p,
                                                       c.c_int, c.c_int, c.c_int, c.c_int]
            L.oracle_amax_and_scale_update_algo.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p,
                                                            c.c_int, c.c_int, c.c_int, c.c_int,
                                                            c.c_int]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits16(x) -> np.ndarray:
    """Accept a numpy uint16/int16 array of bf16 bit patterns, or a torch
    bfloat16 tensor on the CPU, and return a C-contiguous uint16 array."""
    if hasattr(x, "dtype") and not isinstance(x, np.ndarray):  # torch tensor
        import torch
        assert x.dtype == torch.bfloat16, x.dtype
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.int16:
        x = x.view(np.uint16)
    assert x.dtype == np.uint16, x.dtype
    return x


def fp8_encode(p, fmt: int) -> np.ndarray:
    p = np.ascontiguousarray(p, dtype=np.float32)
    out = np.empty(p.shape, dtype=np.uint8)
    lib().oracle_fp8_encode_array(_ptr(p), p.size, fmt, _ptr(out))
    return out


def fp8_decode(codes, fmt: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float32)
    lib().oracle_fp8_decode_array(_ptr(codes), codes.size, fmt, _ptr(out))
    return out


def cast_transpose(x, scale: float, fmt: int, amax_in: float = 0.0,
                   want_q: bool = True, want_qt: bool = True) -> dict:
    """q, qt, amax (max-merged with amax_in) and scale_inv of a bf16 matrix."""
    x = _bits16(x)
    assert x.ndim == 2
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8) if want_q else None
    qt = np.empty((cols, rows), dtype=np.uint8) if want_qt else None
    amax = np.array([amax_in], dtype=np.float32)
    sinv = np.zeros(1, dtype=np.float32)
    lib().oracle_cast_transpose(_ptr(x), rows, cols, float(np.float32(scale)), fmt,
                                _ptr(q) if q is not None else None,
                                _ptr(qt) if qt is not None else None,
                                _ptr(amax), _ptr(sinv))
    return {"q": q, "qt": qt, "amax": amax[0], "scale_inv": sinv[0]}


def amax(x, amax_in: float = 0.0) -> np.float32:
    """max(amax_in, max |x|) by IEEE magnitude bit pattern (NaN propagates)."""
    x = _bits16(x)
    out = np.array([amax_in], dtype=np.float32)
    lib().oracle_amax(_ptr(x), x.size, _ptr(out))
    return out[0]


def dbias(x) -> np.ndarray:
    x = _bits16(x)
    rows, cols = x.shape
    db = np.empty(cols, dtype=np.float32)
    lib().oracle_dbias(_ptr(x), rows, cols, _ptr(db))
    return db


def f32_to_bf16(f) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values, round to nearest even."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(f), f.size, _ptr(out))
    return out


def dbias_bf16(x) -> np.ndarray:
    """db as bf16 bit patterns: the fp32 column sum of dbias(), rounded to bf16."""
    return f32_to_bf16(dbias(x))


def fp8_transpose(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows, cols = q.shape
    out = np.empty((cols, rows), dtype=np.uint8)
    lib().oracle_fp8_transpose(_ptr(q), rows, cols, _ptr(out))
    return out


AMAX_MAX = 0
AMAX_MOST_RECENT = 1


def amax_and_scale_update(hist, scale, scale_inv, fmt: int, margin: int = 0,
                          algo: int = AMAX_MAX):
    """Return updated copies (hist [L, n], scale [n], scale_inv [n]).
    algo: AMAX_MAX (window maximum) or AMAX_MOST_RECENT (row 0 only)."""
    hist = np.array(hist, dtype=np.float32, copy=True, order="C")
    scale = np.array(scale, dtype=np.float32, copy=True)
    scale_inv = np.array(scale_inv, dtype=np.float32, copy=True)
    L, n = hist.shape
    assert scale.shape == (n,) and scale_inv.shape == (n,)
    if algo == AMAX_MAX:
        lib().oracle_amax_and_scale_update(_ptr(hist), _ptr(scale), _ptr(scale_inv),
                                           L, n, fmt, margin)
    else:
        lib().oracle_amax_and_scale_update_algo(_ptr(hist), _ptr(scale), _ptr(scale_inv),
                                                L, n, fmt, margin, 1)
    return hist, scale, scale_inv
