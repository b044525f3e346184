"""Host-side checks of the C ABI (no GPU needed).

The library must load without a GPU, export every function that
include/cast_transpose.h declares, and reject bad arguments on the host
with the documented status codes before anything is launched.  Only calls
that are rejected (or that have nothing to do) are made here: the pointers
passed are never dereferenced.
"""
import ctypes

import pytest

import cast_transpose_gb300 as ct

CT_OK, CT_ERR_NULL, CT_ERR_SHAPE, CT_ERR_ALIGN, CT_ERR_FORMAT, CT_ERR_ARG, CT_ERR_ALIAS, \
    CT_ERR_WORKSPACE, CT_ERR_CUDA = range(9)

# fake, well-separated, 256-byte aligned "device" addresses: never dereferenced
X, Q, QT, S, A, SI, DB, WS, NOOP = (0x10000000 * (i + 1) for i in range(9))


@pytest.fixture(scope="module")
def L():
    return ct.lib()


def test_exports_every_declared_function(L):
    names = ct.header_functions()
    expected = {"fp8_cast_transpose", "fp8_cast_transpose_ex", "fp8_dbias_cast_transpose",
                "fp8_dbias_cast_transpose_ex",
                "fp8_dbias_cast_transpose_workspace_size", "fp8_multi_cast_transpose",
                "fp8_amax_and_scale_update", "fp8_transpose", "fp8_cast", "ct_status_string",
                "ct_device_error"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for s in range(9):
        assert L.ct_status_string(s).decode().startswith("CT_")
    assert L.ct_status_string(99) == b"unknown status"


def _ct(L, x=X, rows=64, cols=64, scale=S, amax=A, sinv=SI, q=Q, qt=QT, fmt=0):
    return L.fp8_cast_transpose(x, rows, cols, scale, amax, sinv, q, qt, fmt, None, None)


def test_cast_transpose_rejects(L):
    assert _ct(L, x=None) == CT_ERR_NULL
    assert _ct(L, q=None) == CT_ERR_NULL
    assert _ct(L, qt=None) == CT_ERR_NULL
    assert _ct(L, scale=None) == CT_ERR_NULL
    assert _ct(L, fmt=2) == CT_ERR_FORMAT
    assert _ct(L, fmt=-1) == CT_ERR_FORMAT
    assert _ct(L, rows=-1) == CT_ERR_SHAPE
    assert _ct(L, cols=-5) == CT_ERR_SHAPE
    assert _ct(L, rows=1 << 40, cols=1 << 20) == CT_ERR_SHAPE
    assert _ct(L, x=X + 1) == CT_ERR_ALIGN
    assert _ct(L, amax=A + 2) == CT_ERR_ALIGN
    assert _ct(L, q=X) == CT_ERR_ALIAS                 # output over the input
    assert _ct(L, qt=Q + 100) == CT_ERR_ALIAS          # outputs overlap
    assert _ct(L, sinv=S) == CT_ERR_ALIAS              # scale_inv over scale
    assert _ct(L, amax=SI) == CT_ERR_ALIAS


def test_cast_transpose_ex_rejects(L):
    def ex(flags, **kw):
        a = dict(x=X, rows=64, cols=64, scale=S, amax=A, sinv=SI, q=Q, qt=QT, fmt=0)
        a.update(kw)
        return L.fp8_cast_transpose_ex(a["x"], a["rows"], a["cols"], a["scale"], a["amax"],
                                       a["sinv"], a["q"], a["qt"], a["fmt"], None, flags, None)
    assert ex(2) == CT_ERR_ARG                      # unknown flag bit
    assert ex(0x80000000) == CT_ERR_ARG
    assert ex(ct.X_READY, x=None) == CT_ERR_NULL    # the same checks as fp8_cast_transpose
    assert ex(ct.X_READY, fmt=3) == CT_ERR_FORMAT
    assert ex(ct.X_READY, q=X) == CT_ERR_ALIAS
    assert ex(ct.X_READY, rows=0) == CT_OK
    assert ex(0, cols=0) == CT_OK


def test_empty_shapes_are_ok_without_launch(L):
    assert _ct(L, rows=0) == CT_OK
    assert _ct(L, cols=0) == CT_OK
    assert L.fp8_cast(X, 0, 7, S, A, SI, Q, 0, None, None) == CT_OK
    assert L.fp8_transpose(X, 5, 0, Q, None, None) == CT_OK


def test_dbias_rejects(L):
    need = L.fp8_dbias_cast_transpose_workspace_size(300, 70)
    assert need == ((300 + 127) // 128) * 70 * 4 + 8   # rounded up to 16 bytes
    assert L.fp8_dbias_cast_transpose_workspace_size(0, 70) == 0
    assert L.fp8_dbias_cast_transpose_workspace_size(-3, 70) == 0

    def call(ws=WS, nbytes=need, db=DB, rows=300, cols=70):
        return L.fp8_dbias_cast_transpose(X, rows, cols, S, A, SI, Q, QT, db, ws, nbytes, 1,
                                          None, None)
    assert call(db=None) == CT_ERR_NULL
    assert call(ws=None) == CT_ERR_WORKSPACE
    assert call(nbytes=need - 1) == CT_ERR_WORKSPACE
    assert call(ws=WS + 4) == CT_ERR_ALIGN
    assert call(db=DB + 2) == CT_ERR_ALIGN
    assert call(db=X) == CT_ERR_ALIAS
    assert call(ws=Q) == CT_ERR_ALIAS
    assert call(rows=0) == CT_OK

    def ex(dtype, db=DB, ws=WS):
        return L.fp8_dbias_cast_transpose_ex(X, 300, 70, S, A, SI, Q, QT, db, dtype, ws, need, 1,
                                             None, None)
    assert ex(2) == CT_ERR_ARG                      # unknown db element type
    assert ex(-1) == CT_ERR_ARG
    assert ex(ct.DBIAS_BF16, db=DB + 1) == CT_ERR_ALIGN
    assert ex(ct.DBIAS_FP32, db=DB + 2) == CT_ERR_ALIGN
    assert ex(ct.DBIAS_BF16, db=None) == CT_ERR_NULL
    assert ex(ct.DBIAS_BF16, ws=None) == CT_ERR_WORKSPACE
    assert ex(ct.DBIAS_BF16, db=X + 2) == CT_ERR_ALIAS


def test_update_rejects(L):
    def call(h=X, s=S, si=SI, L_=16, n=4, fmt=0, margin=0):
        return L.fp8_amax_and_scale_update(h, s, si, L_, n, fmt, margin, None, None)
    assert call(L_=0) == CT_ERR_ARG
    assert call(n=-1) == CT_ERR_ARG
    assert call(margin=-1) == CT_ERR_ARG
    assert call(margin=127) == CT_ERR_ARG
    assert call(fmt=3) == CT_ERR_FORMAT
    assert call(h=None) == CT_ERR_NULL
    assert call(s=S + 1) == CT_ERR_ALIGN
    assert call(si=S) == CT_ERR_ALIAS
    assert call(s=X + 8) == CT_ERR_ALIAS               # scale inside the history
    assert call(n=0) == CT_OK


def test_transpose_and_cast_reject(L):
    assert L.fp8_transpose(None, 4, 4, Q, None, None) == CT_ERR_NULL
    assert L.fp8_transpose(X, -4, 4, Q, None, None) == CT_ERR_SHAPE
    assert L.fp8_transpose(X, 4, 4, X + 8, None, None) == CT_ERR_ALIAS
    assert L.fp8_cast(X, 4, 4, S, A, SI, None, 0, None, None) == CT_ERR_NULL
    assert L.fp8_cast(X, 4, 4, S, A, SI, X, 0, None, None) == CT_ERR_ALIAS


def _desc(x=X, rows=64, cols=64, scale=S, amax=A, sinv=SI, q=Q, qt=QT):
    return ct._Desc(x, rows, cols, scale, amax, sinv, q, qt)


def test_multi_rejects(L):
    arr = (ct._Desc * 2)
    assert L.fp8_multi_cast_transpose(None, 0, 0, None, None) == CT_OK
    assert L.fp8_multi_cast_transpose(None, 2, 0, None, None) == CT_ERR_NULL
    assert L.fp8_multi_cast_transpose(arr(), -1, 0, None, None) == CT_ERR_ARG
    good = _desc()
    other = _desc(x=X + 0x100000, q=Q + 0x100000, qt=QT + 0x100000, amax=A + 64, sinv=SI + 64,
                  scale=S + 64)
    assert L.fp8_multi_cast_transpose(arr(good, _desc(qt=None)), 2, 0, None, None) == CT_ERR_NULL
    assert L.fp8_multi_cast_transpose(arr(good, other), 2, 9, None, None) == CT_ERR_FORMAT
    # second entry writes its data over the first entry's transpose
    clash = _desc(x=X + 0x100000, q=QT, qt=QT + 0x100000, amax=A + 64, sinv=SI + 64)
    assert L.fp8_multi_cast_transpose(arr(good, clash), 2, 0, None, None) == CT_ERR_ALIAS
    # second entry's amax is the first entry's scale_inv
    clash = _desc(x=X + 0x100000, q=Q + 0x100000, qt=QT + 0x100000, amax=SI, sinv=SI + 64)
    assert L.fp8_multi_cast_transpose(arr(good, clash), 2, 0, None, None) == CT_ERR_ALIAS
    # empty entries are skipped: nothing to launch
    e1, e2 = _desc(rows=0), _desc(cols=0, x=X + 0x100000, q=Q + 0x100000, qt=QT + 0x100000,
                                  amax=A + 64, sinv=SI + 64)
    assert L.fp8_multi_cast_transpose(arr(e1, e2), 2, 0, None, None) == CT_OK


def test_device_error_needs_pointer(L):
    assert L.ct_device_error(None, 0) == CT_ERR_NULL


def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(4, 4, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ct.fp8_cast_transpose(x, torch.ones(1), torch.zeros(1), torch.zeros(1),
                              torch.empty(16, dtype=torch.uint8), torch.empty(16, dtype=torch.uint8))


def test_selftest_rejects_bad_limits(L):
    assert L.ct_selftest_bounded_wait(0, None) == CT_ERR_ARG
    assert L.ct_selftest_bounded_wait(2000000, None) == CT_ERR_ARG


def test_update_ex_rejects_unknown_algo(L):
    assert L.fp8_amax_and_scale_update_ex(X, S, SI, 16, 4, 0, 0, 2, None, None) == CT_ERR_ARG
    assert L.fp8_amax_and_scale_update_ex(X, S, SI, 16, 0, 0, 0, 1, None, None) == CT_OK


def test_multi_ex_rejects(L):
    arr = (ct._Desc * 1)(_desc())
    assert L.fp8_multi_cast_transpose_ex(arr, None, 1, None, None) == CT_ERR_NULL
    bad = (ctypes.c_int * 1)(7)
    assert L.fp8_multi_cast_transpose_ex(arr, bad, 1, None, None) == CT_ERR_FORMAT
    assert L.fp8_multi_cast_transpose_ex(None, None, 0, None, None) == CT_OK


def test_fp8_convert_f32_rejects(L):
    f = L.ct_fp8_convert_f32
    assert f(X, 100, 2, Q, None) == CT_ERR_FORMAT
    assert f(X, -1, 0, Q, None) == CT_ERR_SHAPE
    assert f(None, 100, 0, Q, None) == CT_ERR_NULL
    assert f(X, 100, 1, None, None) == CT_ERR_NULL
    assert f(X + 2, 100, 0, Q, None) == CT_ERR_ALIGN
    assert f(X, 100, 0, X + 399, None) == CT_ERR_ALIAS    # out starts inside the 400 input bytes
    assert f(None, 0, 0, None, None) == CT_OK              # nothing to do, nothing launched


def test_dbias_ex_x_ready_flag(L):
    def ex(kind, rows=300):
        return L.fp8_dbias_cast_transpose_ex(X, rows, 70, S, A, SI, Q, QT, DB, kind, WS, 1 << 20, 1,
                                             None, None)
    assert ex(0x200) == CT_ERR_ARG                 # unknown flag bit
    assert ex(0x100 | 2) == CT_ERR_ARG             # the flag does not make a bad dtype valid
    assert ex(0x100 | 1, rows=0) == CT_OK          # empty: nothing launched
    assert ex(0x100, rows=0) == CT_OK



def test_pending_cast_rejects(L):
    H, P = DB, WS          # history and pending rows (fake addresses)

    def cast(x=X, rows=64, cols=64, h=H, s=S, p=P, L_=16, n=2, col=1, k=3, margin=0, algo=0,
             sinv=SI, q=Q, qt=QT, fmt=0, flags=0):
        return L.fp8_cast_transpose_pending(x, rows, cols, h, s, p, L_, n, col, k, margin, algo,
                                            sinv, q, qt, fmt, None, flags, None)
    assert cast(flags=2) == CT_ERR_ARG
    assert cast(L_=0) == CT_ERR_ARG
    assert cast(L_=1025) == CT_ERR_ARG
    assert cast(n=0) == CT_ERR_ARG
    assert cast(col=2) == CT_ERR_ARG                   # col >= n
    assert cast(col=-1) == CT_ERR_ARG
    assert cast(k=-1) == CT_ERR_ARG
    assert cast(k=16) == CT_ERR_ARG                    # k >= hist_len
    assert cast(L_=64, k=32) == CT_ERR_ARG             # runs of at most 32 casts
    assert cast(margin=127) == CT_ERR_ARG
    assert cast(algo=2) == CT_ERR_ARG
    assert cast(h=None) == CT_ERR_NULL
    assert cast(p=None) == CT_ERR_NULL
    assert cast(s=None) == CT_ERR_NULL
    assert cast(x=None) == CT_ERR_NULL
    assert cast(h=H + 2) == CT_ERR_ALIGN
    assert cast(p=P + 2) == CT_ERR_ALIGN
    assert cast(fmt=3) == CT_ERR_FORMAT
    assert cast(sinv=H + 4) == CT_ERR_ALIAS            # scale_inv inside the history
    assert cast(sinv=P) == CT_ERR_ALIAS                # scale_inv over pending row 0 (read)
    assert cast(sinv=S + 4) == CT_ERR_ALIAS            # scale_inv over scale[1]
    assert cast(qt=H) == CT_ERR_ALIAS
    assert cast(rows=0) == CT_OK                       # empty: nothing launched


def test_pending_update_rejects(L):
    H, P = DB, WS

    def upd(h=H, s=S, si=SI, p=P, L_=16, n=2, run=4, fmt=0, margin=0, algo=0):
        return L.fp8_amax_and_scale_update_pending(h, s, si, p, L_, n, run, fmt, margin, algo,
                                                   None, None)
    assert upd(run=0) == CT_ERR_ARG
    assert upd(run=17) == CT_ERR_ARG                   # run > hist_len
    assert upd(L_=64, run=33) == CT_ERR_ARG
    assert upd(L_=1025) == CT_ERR_ARG
    assert upd(n=-1) == CT_ERR_ARG
    assert upd(margin=-1) == CT_ERR_ARG
    assert upd(algo=5) == CT_ERR_ARG
    assert upd(fmt=2) == CT_ERR_FORMAT
    assert upd(p=None) == CT_ERR_NULL
    assert upd(p=P + 1) == CT_ERR_ALIGN
    assert upd(si=S) == CT_ERR_ALIAS
    assert upd(p=H + 8) == CT_ERR_ALIAS                # pending inside the history
    assert upd(n=0) == CT_OK
