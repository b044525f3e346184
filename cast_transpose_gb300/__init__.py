"""GB300 (sm_103a) FP8 cast-transpose library: thin Python binding.

The compute lives in ``libct_gb300.so`` (hand-written CUDA for sm_103a)
behind the C ABI declared in ``include/cast_transpose.h``.  This module only
marshals arguments: it takes torch CUDA tensors (torch provides device
memory and streams), checks dtype/device/contiguity, and passes raw device
pointers and the current stream to the C entry points of the same names.
There is no CPU fallback: if the library is missing every call raises.

Operations (TransformerEngine pages "[PyTorch] cuda graph support" and
"[PyTorch] Refactor FP8 workspaces in linear modules"):
  fp8_cast_transpose        q = fp8(x*scale), qT, amax merge, scale_inv
  fp8_dbias_cast_transpose  the same plus db = x.sum(dim=0) (DbiasCastTranspose)
  fp8_multi_cast_transpose  a list of tensors in one launch
  fp8_amax_and_scale_update delayed-scaling update with the infinite-scale guard
  fp8_transpose             FP8 byte transpose (transpose-cache fill)
  fp8_cast                  cast without transpose
Every call accepts ``noop_flag``: a CUDA fp32 scalar tensor; when it holds a
nonzero value at run time the kernels write nothing.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

E4M3 = 0
E5M2 = 1
X_READY = 1          # fp8_cast_transpose_ex flag CT_X_READY
DBIAS_FP32, DBIAS_BF16 = 0, 1   # fp8_dbias_cast_transpose_ex db element types
DBIAS_X_READY = 0x100           # ... OR'd with the CT_X_READY promise for dy
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libct_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "cast_transpose.h")

_lock = threading.Lock()
_lib = None


class CTError(RuntimeError):
    """A C entry point returned a nonzero ct_status."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class _Desc(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("scale", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("scale_inv", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("out_t", ctypes.c_void_p)]


def lib() -> ctypes.CDLL:
    """Load libct_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            c = ctypes
            vp, i64, i32 = c.c_void_p, c.c_int64, c.c_int
            L.ct_status_string.restype = c.c_char_p
            L.ct_status_string.argtypes = [i32]
            L.fp8_cast_transpose.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, i32, vp, vp]
            L.fp8_cast_transpose_ex.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, i32, vp,
                                                c.c_uint, vp]
            L.fp8_cast.argtypes = [vp, i64, i64, vp, vp, vp, vp, i32, vp, vp]
            L.fp8_dbias_cast_transpose.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp,
                                                   c.c_size_t, i32, vp, vp]
            L.fp8_dbias_cast_transpose_ex.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, vp, i32,
                                                      vp, c.c_size_t, i32, vp, vp]
            L.fp8_dbias_cast_transpose_workspace_size.restype = c.c_size_t
            L.fp8_dbias_cast_transpose_workspace_size.argtypes = [i64, i64]
            L.fp8_multi_cast_transpose.argtypes = [vp, i32, i32, vp, vp]
            L.fp8_multi_cast_transpose_ex.argtypes = [vp, vp, i32, vp, vp]
            L.fp8_amax_and_scale_update.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
            L.fp8_amax_and_scale_update_ex.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                                       vp]
            L.fp8_cast_transpose_pending.argtypes = [vp, i64, i64, vp, vp, vp, i32, i32, i32,
                                                     i32, i32, i32, vp, vp, vp, i32, vp,
                                                     c.c_uint, vp]
            L.fp8_amax_and_scale_update_pending.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32,
                                                            i32, i32, vp, vp]
            L.fp8_transpose.argtypes = [vp, i64, i64, vp, vp, vp]
            L.ct_device_error.argtypes = [c.POINTER(c.c_uint), i32]
            L.ct_selftest_bounded_wait.argtypes = [c.c_uint, vp]
            L.ct_selftest_bounded_wait.restype = i32
            L.ct_fp8_convert_f32.argtypes = [vp, i64, i32, vp, vp]
            L.ct_fp8_convert_f32.restype = i32
            for name in ("fp8_cast_transpose", "fp8_cast_transpose_ex", "fp8_cast",
                         "fp8_dbias_cast_transpose", "fp8_dbias_cast_transpose_ex",
                         "fp8_multi_cast_transpose", "fp8_multi_cast_transpose_ex",
                         "fp8_amax_and_scale_update", "fp8_amax_and_scale_update_ex",
                         "fp8_cast_transpose_pending", "fp8_amax_and_scale_update_pending",
                         "fp8_transpose", "ct_device_error"):
                getattr(L, name).restype = i32
            _lib = L
    return _lib


def header_functions() -> list:
    """Names of the functions declared in include/cast_transpose.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def _check(status: int) -> None:
    if status != 0:
        raise CTError(status, lib().ct_status_string(status).decode())


def _dev(t: torch.Tensor, name: str, dtype=None, numel=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return t.data_ptr()


def _opt(t, name) -> int | None:
    return None if t is None else _dev(t, name, torch.float32, 1)


_U8 = (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _rc(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("expected a 2-D matrix")
    return x.shape[0], x.shape[1]


def fp8_cast_transpose(x, scale, amax, scale_inv, out, out_t, fmt=E4M3, noop_flag=None,
                       stream=None, x_ready=False) -> None:
    """x_ready=True calls fp8_cast_transpose_ex with CT_X_READY: the caller
    promises that no kernel still running when this call starts writes x."""
    rows, cols = _rc(x)
    n = rows * cols
    args = (_dev(x, "x", torch.bfloat16), rows, cols, _dev(scale, "scale", torch.float32, 1),
            _dev(amax, "amax", torch.float32, 1), _dev(scale_inv, "scale_inv", torch.float32, 1),
            _dev(out, "out", _U8, n), _dev(out_t, "out_t", _U8, n), fmt,
            _opt(noop_flag, "noop_flag"))
    if x_ready:
        _check(lib().fp8_cast_transpose_ex(*args, X_READY, _stream(stream)))
    else:
        _check(lib().fp8_cast_transpose(*args, _stream(stream)))


def fp8_cast(x, scale, amax, scale_inv, out, fmt=E4M3, noop_flag=None, stream=None) -> None:
    rows, cols = _rc(x)
    _check(lib().fp8_cast(
        _dev(x, "x", torch.bfloat16), rows, cols, _dev(scale, "scale", torch.float32, 1),
        _dev(amax, "amax", torch.float32, 1), _dev(scale_inv, "scale_inv", torch.float32, 1),
        _dev(out, "out", _U8, rows * cols), fmt, _opt(noop_flag, "noop_flag"), _stream(stream)))


def dbias_workspace_size(rows: int, cols: int) -> int:
    return int(lib().fp8_dbias_cast_transpose_workspace_size(rows, cols))


def fp8_dbias_cast_transpose(dy, scale, amax, scale_inv, out, out_t, dbias, workspace,
                             fmt=E5M2, noop_flag=None, stream=None, x_ready=False) -> None:
    """dbias: fp32 or bf16 [cols]; a bf16 dbias, or x_ready=True (the
    CT_X_READY promise for dy: no kernel still running when this call starts
    writes it), calls fp8_dbias_cast_transpose_ex."""
    rows, cols = _rc(dy)
    n = rows * cols
    ws = _dev(workspace, "workspace", torch.uint8)
    db = _dev(dbias, "dbias", (torch.float32, torch.bfloat16), cols)
    head = (_dev(dy, "dy", torch.bfloat16), rows, cols, _dev(scale, "scale", torch.float32, 1),
            _dev(amax, "amax", torch.float32, 1), _dev(scale_inv, "scale_inv", torch.float32, 1),
            _dev(out, "out", _U8, n), _dev(out_t, "out_t", _U8, n), db)
    tail = (ws, workspace.numel(), fmt, _opt(noop_flag, "noop_flag"), _stream(stream))
    if dbias.dtype == torch.bfloat16 or x_ready:
        kind = (DBIAS_BF16 if dbias.dtype == torch.bfloat16 else DBIAS_FP32) | \
               (DBIAS_X_READY if x_ready else 0)
        _check(lib().fp8_dbias_cast_transpose_ex(*head, kind, *tail))
    else:
        _check(lib().fp8_dbias_cast_transpose(*head, *tail))


def _descs(xs, scales, amaxes, scale_invs, outs, outs_t):
    n = len(xs)
    if not (len(scales) == len(amaxes) == len(scale_invs) == len(outs) == len(outs_t) == n):
        raise ValueError("all lists must have the same length")
    descs = (_Desc * max(n, 1))()
    for i in range(n):
        rows, cols = _rc(xs[i])
        m = rows * cols
        descs[i] = _Desc(_dev(xs[i], f"xs[{i}]", torch.bfloat16), rows, cols,
                         _dev(scales[i], f"scales[{i}]", torch.float32, 1),
                         _dev(amaxes[i], f"amaxes[{i}]", torch.float32, 1),
                         _dev(scale_invs[i], f"scale_invs[{i}]", torch.float32, 1),
                         _dev(outs[i], f"outs[{i}]", _U8, m), _dev(outs_t[i], f"outs_t[{i}]", _U8, m))
    return descs, n


def fp8_multi_cast_transpose(xs, scales, amaxes, scale_invs, outs, outs_t, fmt=E4M3,
                             noop_flag=None, stream=None) -> None:
    """Each of scales/amaxes/scale_invs is a list of 1-element fp32 tensors
    (views into one buffer are fine)."""
    descs, n = _descs(xs, scales, amaxes, scale_invs, outs, outs_t)
    _check(lib().fp8_multi_cast_transpose(descs, n, fmt, _opt(noop_flag, "noop_flag"),
                                          _stream(stream)))


def fp8_multi_cast_transpose_ex(xs, scales, amaxes, scale_invs, outs, outs_t, fmts,
                                noop_flag=None, stream=None) -> None:
    """As fp8_multi_cast_transpose with one FP8 format per tensor."""
    descs, n = _descs(xs, scales, amaxes, scale_invs, outs, outs_t)
    if len(fmts) != n:
        raise ValueError("one format per tensor")
    fmt_arr = (ctypes.c_int * max(n, 1))(*fmts)
    _check(lib().fp8_multi_cast_transpose_ex(descs, fmt_arr, n, _opt(noop_flag, "noop_flag"),
                                             _stream(stream)))


def fp8_amax_and_scale_update(amax_history, scale, scale_inv, fmt=E4M3, margin=0,
                              noop_flag=None, stream=None) -> None:
    if amax_history.dim() != 2:
        raise ValueError("amax_history must be [hist_len, n]")
    L, n = amax_history.shape
    _check(lib().fp8_amax_and_scale_update(
        _dev(amax_history, "amax_history", torch.float32), _dev(scale, "scale", torch.float32, n),
        _dev(scale_inv, "scale_inv", torch.float32, n), L, n, fmt, margin,
        _opt(noop_flag, "noop_flag"), _stream(stream)))


AMAX_MAX = 0
AMAX_MOST_RECENT = 1


def fp8_amax_and_scale_update_ex(amax_history, scale, scale_inv, fmt=E4M3, margin=0,
                                 amax_algo=AMAX_MAX, noop_flag=None, stream=None) -> None:
    if amax_history.dim() != 2:
        raise ValueError("amax_history must be [hist_len, n]")
    L, n = amax_history.shape
    _check(lib().fp8_amax_and_scale_update_ex(
        _dev(amax_history, "amax_history", torch.float32), _dev(scale, "scale", torch.float32, n),
        _dev(scale_inv, "scale_inv", torch.float32, n), L, n, fmt, margin, amax_algo,
        _opt(noop_flag, "noop_flag"), _stream(stream)))


def fp8_cast_transpose_pending(x, amax_history, scale, pending, col, k, scale_inv, out, out_t,
                               fmt=E4M3, margin=0, amax_algo=AMAX_MAX, noop_flag=None,
                               stream=None, x_ready=False) -> None:
    """Cast k of a run of casts on history column `col` whose scale updates
    are deferred: the scale is derived from amax_history [L, n] and scale [n]
    as they stood before the run and from pending rows 0 .. k-1 [K, n]; the
    amax goes to pending[k, col]."""
    rows, cols = _rc(x)
    if amax_history.dim() != 2 or pending.dim() != 2:
        raise ValueError("amax_history must be [hist_len, n] and pending [run, n]")
    L, n = amax_history.shape
    if pending.shape[1] != n or not 0 <= k < pending.shape[0]:
        raise ValueError("pending must be [run, n] with k < run")
    _check(lib().fp8_cast_transpose_pending(
        _dev(x, "x", torch.bfloat16), rows, cols, _dev(amax_history, "amax_history", torch.float32),
        _dev(scale, "scale", torch.float32, n), _dev(pending, "pending", torch.float32), L, n, col,
        k, margin, amax_algo, _dev(scale_inv, "scale_inv", torch.float32, 1),
        _dev(out, "out", _U8, rows * cols), _dev(out_t, "out_t", _U8, rows * cols), fmt,
        _opt(noop_flag, "noop_flag"), X_READY if x_ready else 0, _stream(stream)))


def fp8_amax_and_scale_update_pending(amax_history, scale, scale_inv, pending, fmt=E4M3,
                                      margin=0, amax_algo=AMAX_MAX, noop_flag=None,
                                      stream=None) -> None:
    """The updates deferred by a run of len(pending) fp8_cast_transpose_pending
    calls, applied at once; pending is zeroed."""
    if amax_history.dim() != 2 or pending.dim() != 2:
        raise ValueError("amax_history must be [hist_len, n] and pending [run, n]")
    L, n = amax_history.shape
    run = pending.shape[0]
    if pending.shape[1] != n:
        raise ValueError("pending must be [run, n]")
    _check(lib().fp8_amax_and_scale_update_pending(
        _dev(amax_history, "amax_history", torch.float32), _dev(scale, "scale", torch.float32, n),
        _dev(scale_inv, "scale_inv", torch.float32, n), _dev(pending, "pending", torch.float32),
        L, n, run, fmt, margin, amax_algo, _opt(noop_flag, "noop_flag"), _stream(stream)))


def fp8_transpose(q, out_t, noop_flag=None, stream=None) -> None:
    rows, cols = _rc(q)
    _check(lib().fp8_transpose(_dev(q, "q", _U8), rows, cols, _dev(out_t, "out_t", _U8, rows * cols),
                               _opt(noop_flag, "noop_flag"), _stream(stream)))


def fp8_convert_f32(x, out, fmt=E4M3, stream=None) -> None:
    """out[i] = FP8 code of the fp32 value x[i] (the cast kernels' conversion
    step without the scale); x fp32, out uint8, both contiguous, same size."""
    n = x.numel()
    _check(lib().ct_fp8_convert_f32(_dev(x, "x", torch.float32), n, fmt, _dev(out, "out", _U8, n),
                                    _stream(stream)))


def device_error(clear: bool = False) -> int:
    v = ctypes.c_uint(0)
    _check(lib().ct_device_error(ctypes.byref(v), 1 if clear else 0))
    return v.value


def selftest_bounded_wait(limit_us: int = 20000, stream=None) -> None:
    """Launch the bounded-wait self-test (its wait times out by design and
    sets bit 2 of the device diagnostic word)."""
    _check(lib().ct_selftest_bounded_wait(limit_us, _stream(stream)))


def empty_outputs(x: torch.Tensor):
    """Convenience allocation of (out, out_t) uint8 buffers for a 2-D x."""
    rows, cols = _rc(x)
    return (torch.empty(rows, cols, dtype=torch.uint8, device=x.device),
            torch.empty(cols, rows, dtype=torch.uint8, device=x.device))
