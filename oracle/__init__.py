"""CPU oracle for sparse 3-D convolution (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library path never calls it, and it
shares no code with the CUDA path: the C source ``spc_oracle.c`` beside this
file is compiled on its own with the host C compiler and loaded through ctypes.

Every floating-point result is computed in double precision from the exact
values of the inputs (fp32/fp16/bf16 tensors are widened exactly to float64).
See ``spc_oracle.c`` for the definition each function follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_spc.so")
_lock = threading.Lock()
_lib = None

OK, ERR_RANGE, ERR_DUPLICATE, ERR_ARG, ERR_CAPACITY, ERR_NOMEM = range(6)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with status {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile spc_oracle.c into a shared library (host gcc, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
               "-lm"]
        # row loops in parallel where the compiler has OpenMP; plain C otherwise
        if subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True).returncode != 0:
            subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_subm_map.argtypes = [_I32P, _i64, _i32, _I32P, _I32P, _I32P, _I32P, _I64P]
            lib.orc_out_shape.argtypes = [_I32P, _I32P, _I32P, _I32P, _I32P, _I32P]
            lib.orc_strided_out_coords.argtypes = [_I32P, _i64, _i32, _I32P, _I32P, _I32P, _I32P,
                                                   _I32P, _I32P, _i64, ctypes.POINTER(_i64)]
            lib.orc_strided_map.argtypes = [_I32P, _i64, _I32P, _i64, _i32, _I32P, _I32P, _I32P,
                                            _I32P, _I32P, _I32P, ctypes.c_void_p, _I64P]
            lib.orc_transpose_map.argtypes = [_I32P, _i64, _i64, _i64, _I32P]
            lib.orc_transpose_map.restype = None
            lib.orc_conv_fwd.argtypes = [_F64P, _F64P, ctypes.c_void_p, _I32P, _i64, _i64, _i64,
                                         _i32, _i32, _F64P]
            lib.orc_conv_fwd.restype = None
            lib.orc_conv_fwd_rows.argtypes = [_F64P, _F64P, ctypes.c_void_p, _I32P, _i64, _i64,
                                              _i64, _i32, _i32, _I64P, _i64, _F64P]
            lib.orc_conv_fwd_rows.restype = None
            lib.orc_maxpool_fwd.argtypes = [_F64P, _I32P, _i64, _i64, _i64, _i32, _F64P,
                                            ctypes.c_void_p]
            lib.orc_maxpool_fwd.restype = None
            lib.orc_maxpool_dgrad.argtypes = [_F64P, _I32P, ctypes.c_void_p, _i64, _i64, _i64, _i32,
                                              _F64P]
            lib.orc_maxpool_dgrad.restype = None
            lib.orc_conv_inverse.argtypes = [_F64P, _F64P, ctypes.c_void_p, _I32P, _i64, _i64, _i64,
                                             _i32, _i32, _F64P]
            lib.orc_conv_inverse.restype = None
            lib.orc_conv_dgrad.argtypes = [_F64P, _F64P, _I32P, _i64, _i64, _i64, _i32, _i32, _F64P]
            lib.orc_conv_dgrad.restype = None
            lib.orc_conv_dgrad_rows.argtypes = [_F64P, _F64P, _I32P, _i64, _i64, _i64, _i32, _i32,
                                                _I64P, _i64, _F64P]
            lib.orc_conv_dgrad_rows.restype = None
            lib.orc_conv_wgrad.argtypes = [_F64P, _F64P, _I32P, _i64, _i64, _i64, _i32, _i32, _F64P]
            lib.orc_conv_wgrad.restype = None
            lib.orc_conv_wgrad_entries.argtypes = [_F64P, _F64P, _I32P, _i64, _i64, _i64, _i32,
                                                   _i32, _I64P, _i64, _F64P]
            lib.orc_conv_wgrad_entries.restype = None
            _I8P = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
            _F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
            lib.orc_set_threads.argtypes = [_i32]
            lib.orc_set_threads.restype = _i32
            lib.orc_conv_fwd_int8.argtypes = [_I8P, _I8P, _F32P, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_float, _i32, ctypes.c_void_p, _i64, _i64,
                                              _i64, _i32, _i32, _I8P, _I32P]
            _lib = lib
    return _lib


def set_threads(n: int = 0) -> int:
    """Threads of the oracle's parallel row loops (n > 0 sets them); returns the
    count in effect (1 when it was compiled without OpenMP)."""
    return int(_load().orc_set_threads(int(n)))


def _triple(v) -> np.ndarray:
    if np.isscalar(v):
        v = (v, v, v)
    return np.ascontiguousarray(np.asarray(v, dtype=np.int32).reshape(3))


def _coords(c) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(c, dtype=np.int32).reshape(-1, 4))


def f64(t) -> np.ndarray:
    """Exact float64 copy of a CPU tensor / array of any float dtype."""
    if hasattr(t, "detach"):
        t = t.detach().to("cpu")
        import torch

        t = t.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def subm_map(coords, batch: int, shape, ksize=3, dil=1):
    """Submanifold indice map [K, N] int32 (-1 = no neighbour) and pair counts [K]."""
    lib = _load()
    c = _coords(coords)
    ks, dl = _triple(ksize), _triple(dil)
    K = int(np.prod(ks))
    n = c.shape[0]
    imap = np.empty((K, n), dtype=np.int32)
    cnt = np.empty(K, dtype=np.int64)
    st = lib.orc_subm_map(c, n, batch, _triple(shape), ks, dl, imap, cnt)
    if st != OK:
        raise OracleError(st, "subm_map")
    return imap, cnt


def out_shape(in_shape, ksize, stride, pad, dil=1):
    lib = _load()
    out = np.empty(3, dtype=np.int32)
    st = lib.orc_out_shape(_triple(in_shape), _triple(ksize), _triple(stride), _triple(pad),
                           _triple(dil), out)
    if st != OK:
        raise OracleError(st, "out_shape")
    return tuple(int(v) for v in out)


def strided_out_coords(coords, batch: int, in_shape, ksize=3, stride=2, pad=1, dil=1):
    """Output coordinate set of a strided sparse conv, sorted by (b, z, y, x)."""
    lib = _load()
    c = _coords(coords)
    ks = _triple(ksize)
    cap = max(1, c.shape[0] * int(np.prod(ks)))
    out = np.empty((cap, 4), dtype=np.int32)
    n_out = _i64(0)
    st = lib.orc_strided_out_coords(c, c.shape[0], batch, _triple(in_shape), ks, _triple(stride),
                                    _triple(pad), _triple(dil), out, cap, ctypes.byref(n_out))
    if st != OK:
        raise OracleError(st, "strided_out_coords")
    return out[: n_out.value].copy()


def strided_map(coords, out_coords, batch: int, in_shape, ksize=3, stride=2, pad=1, dil=1,
                with_transpose: bool = True):
    """out->in map [K, N_out], in->out map [K, N] (or None) and pair counts [K]."""
    lib = _load()
    c, oc = _coords(coords), _coords(out_coords)
    ks = _triple(ksize)
    K = int(np.prod(ks))
    imap = np.empty((K, oc.shape[0]), dtype=np.int32)
    imap_t = np.empty((K, c.shape[0]), dtype=np.int32) if with_transpose else None
    cnt = np.empty(K, dtype=np.int64)
    st = lib.orc_strided_map(c, c.shape[0], oc, oc.shape[0], batch, _triple(in_shape), ks,
                             _triple(stride), _triple(pad), _triple(dil), imap,
                             imap_t.ctypes.data if imap_t is not None else None, cnt)
    if st != OK:
        raise OracleError(st, "strided_map")
    return imap, imap_t, cnt


def transpose_map(imap, n_in: int):
    lib = _load()
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    out = np.empty((K, n_in), dtype=np.int32)
    lib.orc_transpose_map(m, K, n_in, n_out, out)
    return out


def conv_fwd(x, w, bias, imap, rows=None):
    """y = bias + sum over pairs of x[i] W[k]; all rows, or the listed output rows."""
    lib = _load()
    x, w = f64(x), f64(w)
    b = f64(bias) if bias is not None else None
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    n_in, cin = x.shape
    cout = w.shape[2]
    assert w.shape == (K, cin, cout)
    bptr = b.ctypes.data if b is not None else None
    if rows is None:
        y = np.empty((n_out, cout), dtype=np.float64)
        lib.orc_conv_fwd(x, w, bptr, m, K, n_in, n_out, cin, cout, y)
        return y
    r = np.ascontiguousarray(rows, dtype=np.int64)
    y = np.empty((r.shape[0], cout), dtype=np.float64)
    lib.orc_conv_fwd_rows(x, w, bptr, m, K, n_in, n_out, cin, cout, r, r.shape[0], y)
    return y


def conv_fwd_fused(x, w, bias, imap, residual=None, add_scale=1.0, relu=False):
    """Forward with the fused epilogue, as defined: act(conv + bias + add_scale residual),
    act = max(., 0) when relu; all in float64."""
    y = conv_fwd(x, w, bias, imap)
    if residual is not None:
        y = y + float(add_scale) * f64(residual)
    return np.maximum(y, 0.0) if relu else y


def maxpool_fwd(x, imap):
    """Max over each output row's pairs (occupied inputs only); returns (y, arg) with
    arg[o, c] the first offset reaching the max (255 when the row has no pair)."""
    lib = _load()
    x = f64(x)
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    n_in, c = x.shape
    y = np.empty((n_out, c), dtype=np.float64)
    arg = np.empty((n_out, c), dtype=np.uint8)
    lib.orc_maxpool_fwd(x, m, K, n_in, n_out, c, y, arg.ctypes.data)
    return y, arg


def maxpool_dgrad(dy, imap, arg, n_in: int):
    lib = _load()
    dy = f64(dy)
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    c = dy.shape[1]
    a = np.ascontiguousarray(arg, dtype=np.uint8)
    dx = np.empty((n_in, c), dtype=np.float64)
    lib.orc_maxpool_dgrad(dy, m, a.ctypes.data, K, n_in, n_out, c, dx)
    return dx


def conv_inverse(y, w, bias, imap, n_out: int):
    """Inverse conv of a strided conv with forward map imap [K, N_y]:
    out[i] = bias + sum over pairs imap[k, o] = i of y[o] W[k], out [n_out, Cout]."""
    lib = _load()
    y, w = f64(y), f64(w)
    b = f64(bias) if bias is not None else None
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_y = m.shape
    cy, cout = w.shape[1], w.shape[2]
    assert y.shape == (n_y, cy) and w.shape[0] == K
    out = np.empty((n_out, cout), dtype=np.float64)
    lib.orc_conv_inverse(y, w, b.ctypes.data if b is not None else None, m, K, n_y, n_out, cy, cout, out)
    return out


def conv_dgrad(dy, w, imap, n_in: int):
    lib = _load()
    dy, w = f64(dy), f64(w)
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    cin, cout = w.shape[1], w.shape[2]
    dx = np.empty((n_in, cin), dtype=np.float64)
    lib.orc_conv_dgrad(dy, w, m, K, n_in, n_out, cin, cout, dx)
    return dx


def conv_dgrad_rows(dy, w, imap_t, rows):
    """dinput at the listed input rows through a transposed map [K, N_in]."""
    lib = _load()
    dy, w = f64(dy), f64(w)
    mt = np.ascontiguousarray(imap_t, dtype=np.int32)
    K, n_in = mt.shape
    n_out = dy.shape[0]
    cin, cout = w.shape[1], w.shape[2]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    dx = np.empty((r.shape[0], cin), dtype=np.float64)
    lib.orc_conv_dgrad_rows(dy, w, mt, K, n_in, n_out, cin, cout, r, r.shape[0], dx)
    return dx


def conv_wgrad(x, dy, imap):
    lib = _load()
    x, dy = f64(x), f64(dy)
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    n_in, cin = x.shape
    cout = dy.shape[1]
    dw = np.empty((K, cin, cout), dtype=np.float64)
    lib.orc_conv_wgrad(x, dy, m, K, n_in, n_out, cin, cout, dw)
    return dw


def conv_wgrad_entries(x, dy, imap, entries):
    """dW at flat indices (k*cin + c)*cout + j."""
    lib = _load()
    x, dy = f64(x), f64(dy)
    m = np.ascontiguousarray(imap, dtype=np.int32)
    K, n_out = m.shape
    n_in, cin = x.shape
    cout = dy.shape[1]
    e = np.ascontiguousarray(entries, dtype=np.int64)
    v = np.empty(e.shape[0], dtype=np.float64)
    lib.orc_conv_wgrad_entries(x, dy, m, K, n_in, n_out, cin, cout, e, e.shape[0], v)
    return v


def _np(t, dtype):
    if hasattr(t, "detach"):
        t = t.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(t), dtype=dtype)


def conv_fwd_int8(x, w, scale, bias, imap, add=None, add_scale=0.0, relu=False):
    """Quantized forward (spconv's int8 implicit GEMM rule): int8 codes x [N_in, Cin]
    and w [K, Cin, Cout], fp32 per-channel scale [Cout] and bias [Cout] (or None),
    optional int8 residual add [N_out, Cout] with an fp32 scale, optional ReLU.
    imap [K, N_out], or None for K = 1 on the identity map.  Returns (y int8
    [N_out, Cout], acc int32 [N_out, Cout] -- the exact integer sums)."""
    lib = _load()
    xq, wq = _np(x, np.int8), _np(w, np.int8)
    K, cin, cout = wq.shape
    n_in = xq.shape[0]
    assert xq.shape[1] == cin
    if imap is None:
        assert K == 1
        m, n_out = None, n_in
    else:
        m = np.ascontiguousarray(imap, dtype=np.int32)
        assert m.shape[0] == K
        n_out = m.shape[1]
    sc = _np(scale, np.float32)
    b = _np(bias, np.float32) if bias is not None else None
    a = _np(add, np.int8) if add is not None else None
    y = np.empty((n_out, cout), dtype=np.int8)
    acc = np.empty((n_out, cout), dtype=np.int32)
    st = lib.orc_conv_fwd_int8(xq, wq, sc, b.ctypes.data if b is not None else None,
                               a.ctypes.data if a is not None else None, float(add_scale),
                               1 if relu else 0, m.ctypes.data if m is not None else None, K, n_in,
                               n_out, cin, cout, y, acc)
    if st != OK:
        raise OracleError(st, "conv_fwd_int8")
    return y, acc
