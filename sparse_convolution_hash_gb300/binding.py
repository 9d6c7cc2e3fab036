"""ctypes binding of libspc.so (the C ABI declared in include/spc.h).

Each ``spc_*`` function here has the name of the C entry point it calls and
only marshals arguments: it takes torch CUDA tensors, allocates the outputs and
workspace with torch (device memory only), passes raw pointers and the current
CUDA stream, and checks the returned status.  Every computation runs in the
library's CUDA kernels; there is no CPU fallback.  If libspc.so has not been
built, loading raises ``SpcLibraryMissing``.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libspc.so")

SPC_OK = 0
STATUS_NAMES = {
    0: "SPC_OK", 1: "SPC_ERR_INVALID_ARG", 2: "SPC_ERR_COORD_RANGE", 3: "SPC_ERR_DUPLICATE",
    4: "SPC_ERR_TABLE_FULL", 5: "SPC_ERR_CAPACITY", 6: "SPC_ERR_UNSUPPORTED", 7: "SPC_ERR_CUDA",
    8: "SPC_ERR_WORKSPACE", 9: "SPC_ERR_TIMEOUT",
}
SPC_F32, SPC_F16, SPC_BF16 = 0, 1, 2
SPC_PREC_EXACT, SPC_PREC_TF32 = 0, 1
SPC_MAP_TRANSPOSED, SPC_MAP_SUBM_MIRROR = 0, 1

_DTYPES = {torch.float32: SPC_F32, torch.float16: SPC_F16, torch.bfloat16: SPC_BF16}


class SpcLibraryMissing(RuntimeError):
    pass


class SpcError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class Geom(ctypes.Structure):
    _fields_ = [("ksize", ctypes.c_int32 * 3), ("stride", ctypes.c_int32 * 3),
                ("pad", ctypes.c_int32 * 3), ("dil", ctypes.c_int32 * 3)]


def _triple(v) -> tuple:
    if isinstance(v, int):
        return (v, v, v)
    t = tuple(int(a) for a in v)
    assert len(t) == 3
    return t


def make_geom(ksize=3, stride=1, pad=0, dil=1) -> Geom:
    g = Geom()
    for name, v in (("ksize", ksize), ("stride", stride), ("pad", pad), ("dil", dil)):
        arr = getattr(g, name)
        for a, x in enumerate(_triple(v)):
            arr[a] = x
    return g


_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_I3 = ctypes.c_int32 * 3
_GP = ctypes.POINTER(Geom)


def lib():
    """The loaded libspc.so (raises SpcLibraryMissing if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise SpcLibraryMissing(
                    f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                    "(there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            L.spc_status_string.argtypes = [_i32]
            L.spc_status_string.restype = ctypes.c_char_p
            L.spc_version.argtypes = []
            L.spc_version.restype = _i32
            L.spc_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.spc_set_wait_limit_ns.restype = _i32
            L.spc_get_wait_limit_ns.argtypes = []
            L.spc_get_wait_limit_ns.restype = ctypes.c_uint64
            L.spc_out_shape.argtypes = [_I3, _GP, _I3]
            L.spc_out_shape.restype = _i32
            L.spc_indice_map_workspace_size.argtypes = [_i64]
            L.spc_indice_map_workspace_size.restype = _sz
            L.spc_build_indice_map.argtypes = [_p, _i64, _i32, _I3, _GP, _i32, _p, _i64, _p, _p,
                                               _p, _p, _p, _p, _sz, _p]
            L.spc_build_indice_map.restype = _i32
            L.spc_strided_out_coords_workspace_size.argtypes = [_i64, _GP]
            L.spc_strided_out_coords_workspace_size.restype = _sz
            L.spc_strided_out_coords.argtypes = [_p, _i64, _i32, _I3, _GP, _I3, _p, _i64, _p, _p,
                                                 _p, _sz, _p]
            L.spc_strided_out_coords.restype = _i32
            L.spc_conv_workspace_size.argtypes = [_i32, _i64, _i64, _i32, _i32, _i32]
            L.spc_conv_workspace_size.restype = _sz
            L.spc_conv_fwd.argtypes = [_p, _p, _p, _p, _p, _i32, _i64, _i64, _i32, _i32, _i32,
                                       _i32, _p, _p, _p, _sz, _p]
            L.spc_conv_fwd.restype = _i32
            L.spc_conv_fwd_fused.argtypes = [_p, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i32, _i32, _i32,
                                             _i32, _p, ctypes.c_float, _i32, _p, _p, _p, _sz, _p]
            L.spc_conv_fwd_fused.restype = _i32
            L.spc_maxpool_fwd.argtypes = [_p, _p, _p, _i32, _i64, _i64, _i32, _i32, _p, _p, _p]
            L.spc_maxpool_fwd.restype = _i32
            L.spc_maxpool_dgrad.argtypes = [_p, _p, _p, _i32, _i64, _i64, _i32, _i32, _p, _p]
            L.spc_maxpool_dgrad.restype = _i32
            L.spc_conv_inverse.argtypes = [_p, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i32, _i32, _i32,
                                           _i32, _p, _p, _p, _sz, _p]
            L.spc_map_row_order_workspace_size.argtypes = [_i64]
            L.spc_map_row_order_workspace_size.restype = _sz
            L.spc_map_row_order.argtypes = [_p, _i32, _i64, _p, _p, _p, _sz, _p]
            L.spc_map_row_order.restype = _i32
            L.spc_conv_inverse.restype = _i32
            L.spc_conv_int8_workspace_size.argtypes = [_i32, _i32, _i32]
            L.spc_conv_int8_workspace_size.restype = _sz
            L.spc_conv_fwd_int8.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i32, _i32,
                                            _p, ctypes.c_float, _i32, _p, _p, _p, _sz, _p]
            L.spc_conv_fwd_int8.restype = _i32
            L.spc_conv_dgrad.argtypes = [_p, _p, _p, _i32, _p, _p, _i32, _i64, _i64, _i32, _i32,
                                         _i32, _i32, _p, _p, _p, _sz, _p]
            L.spc_conv_dgrad.restype = _i32
            L.spc_conv_wgrad_workspace_size.argtypes = [_i32, _i64, _i64, _i32, _i32, _i32]
            L.spc_conv_wgrad_workspace_size.restype = _sz
            L.spc_conv_wgrad.argtypes = [_p, _p, _p, _i32, _i64, _i64, _i32, _i32, _i32, _i32,
                                         _p, _p, _p, _sz, _p]
            L.spc_conv_wgrad.restype = _i32
            _lib = L
    return _lib


def _check(code: int, where: str):
    if code != SPC_OK:
        raise SpcError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.contiguous()


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def new_status(device) -> torch.Tensor:
    """A zeroed device status word (sticky error flag of the data-dependent checks)."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor, where: str = "spc"):
    """Synchronise on the status word and raise SpcError if a kernel reported an error."""
    code = int(status.item())
    if code != SPC_OK:
        raise SpcError(code, where)


def spc_status_string(code: int) -> str:
    return lib().spc_status_string(code).decode()


def spc_version() -> int:
    return int(lib().spc_version())


def spc_set_wait_limit_ns(ns: int) -> None:
    """Bound (ns) of the waits of one warp role on another in the pipelined
    tensor-core kernels launched afterwards (a wait that runs out sets
    SPC_ERR_TIMEOUT in the call's status word)."""
    _check(lib().spc_set_wait_limit_ns(int(ns)), "spc_set_wait_limit_ns")


def spc_get_wait_limit_ns() -> int:
    return int(lib().spc_get_wait_limit_ns())


def spc_out_shape(in_shape, ksize=3, stride=2, pad=1, dil=1) -> tuple:
    g = make_geom(ksize, stride, pad, dil)
    out = _I3()
    _check(lib().spc_out_shape(_I3(*_triple(in_shape)), ctypes.byref(g), out), "spc_out_shape")
    return tuple(out)


def spc_indice_map_workspace_size(n_in: int) -> int:
    return int(lib().spc_indice_map_workspace_size(n_in))


def spc_build_indice_map(coords: torch.Tensor, batch: int, in_shape: Sequence[int], ksize=3,
                         stride=1, pad=0, dil=1, subm: bool = True,
                         out_coords: Optional[torch.Tensor] = None, with_transpose: bool = False,
                         with_mask: bool = True, status: Optional[torch.Tensor] = None,
                         ws: Optional[torch.Tensor] = None, out: Optional[dict] = None) -> dict:
    """Indice map [K, N_out] (+ transpose [K, N_in], pair counts [K], row masks [N_out]).

    Returns a dict with keys imap, imap_t (or None), pair_count, mask (or None),
    status, ws.  Data errors land in `status`; call check_status() to raise them.
    Passing the dict of an earlier call as `out` reuses its buffers (no
    allocation, so the call can be captured in a CUDA graph).
    """
    coords = _cuda(coords, "coords").to(torch.int32)
    dev = coords.device
    n_in = coords.shape[0]
    g = make_geom(ksize, stride, pad, dil)
    K = g.ksize[0] * g.ksize[1] * g.ksize[2]
    if subm:
        n_out = n_in
        oc = None
    else:
        oc = _cuda(out_coords, "out_coords").to(torch.int32)
        n_out = oc.shape[0]
    if out is not None:
        imap, imap_t, pair_count, mask = out["imap"], out["imap_t"], out["pair_count"], out["mask"]
        status = out["status"] if status is None else status
        ws = out["ws"] if ws is None else ws
    else:
        imap = torch.empty((K, n_out), dtype=torch.int32, device=dev)
        imap_t = (torch.empty((K, n_in), dtype=torch.int32, device=dev)
                  if (with_transpose and not subm) else None)
        pair_count = torch.empty(K, dtype=torch.int32, device=dev)
        mask = torch.empty(n_out, dtype=torch.int32, device=dev) if (with_mask and K <= 32) else None
    status = new_status(dev) if status is None else status
    nbytes = spc_indice_map_workspace_size(n_in)
    if ws is None or ws.numel() < nbytes:
        ws = _workspace(nbytes, dev)
    code = lib().spc_build_indice_map(
        _ptr(coords), n_in, batch, _I3(*_triple(in_shape)), ctypes.byref(g), 1 if subm else 0,
        _ptr(oc), n_out, _ptr(imap), _ptr(imap_t), _ptr(pair_count), _ptr(mask), _ptr(status),
        _ptr(ws), ws.numel(), _stream(dev))
    _check(code, "spc_build_indice_map")
    return dict(imap=imap, imap_t=imap_t, pair_count=pair_count, mask=mask, status=status, ws=ws)


def spc_strided_out_coords(coords: torch.Tensor, batch: int, in_shape, ksize=3, stride=2, pad=1,
                           dil=1, cap: Optional[int] = None, status: Optional[torch.Tensor] = None):
    """Output coordinate set [N_out, 4] (sorted by (b, z, y, x)) and the output grid.

    Reads N_out back to the host (one synchronisation) to trim the buffer.
    """
    coords = _cuda(coords, "coords").to(torch.int32)
    dev = coords.device
    n_in = coords.shape[0]
    g = make_geom(ksize, stride, pad, dil)
    K = g.ksize[0] * g.ksize[1] * g.ksize[2]
    cap = n_in * K if cap is None else int(cap)
    out = torch.empty((max(cap, 1), 4), dtype=torch.int32, device=dev)
    n_out = torch.zeros(1, dtype=torch.int64, device=dev)
    status = new_status(dev) if status is None else status
    nbytes = int(lib().spc_strided_out_coords_workspace_size(n_in, ctypes.byref(g)))
    ws = _workspace(nbytes, dev)
    out_shape = _I3()
    code = lib().spc_strided_out_coords(
        _ptr(coords), n_in, batch, _I3(*_triple(in_shape)), ctypes.byref(g), out_shape, _ptr(out),
        cap, _ptr(n_out), _ptr(status), _ptr(ws), ws.numel(), _stream(dev))
    _check(code, "spc_strided_out_coords")
    n = int(n_out.item())
    check_status(status, "spc_strided_out_coords")
    return out[:n], tuple(out_shape)


def spc_conv_fwd(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                 imap: Optional[torch.Tensor], mask: Optional[torch.Tensor] = None,
                 n_out: Optional[int] = None, precision: int = SPC_PREC_EXACT,
                 out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None, perm: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y[o] = bias + sum over pairs of x[imap[k, o]] W[k]; y has x's dtype.

    Pass `out`, `ws` (spc_conv_workspace_size bytes) and `status` to call
    without allocating (e.g. inside CUDA-graph capture).  `perm` (with its
    `mask`) from spc_map_row_order(imap) computes the tiles in that row order
    (through spc_conv_fwd_fused, which takes it)."""
    if perm is not None:
        return spc_conv_fwd_fused(x, w, bias, imap, mask, n_out=n_out, precision=precision,
                                  out=out, status=status, ws=ws, perm=perm)
    x = _cuda(x, "x")
    w = _cuda(w, "w").to(x.dtype)
    b = _cuda(bias, "bias").to(x.dtype) if bias is not None else None
    K, cin, cout = w.shape
    if imap is not None:
        imap = _cuda(imap, "imap")
        n_out = imap.shape[1]
    elif n_out is None:
        n_out = x.shape[0]
    y = torch.empty((n_out, cout), dtype=x.dtype, device=x.device) if out is None else out
    dt = _DTYPES[x.dtype]
    nbytes = int(lib().spc_conv_workspace_size(K, x.shape[0], n_out, cin, cout, dt))
    if nbytes and (ws is None or ws.numel() < nbytes):
        ws = _workspace(nbytes, x.device)
    code = lib().spc_conv_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(imap), _ptr(mask), K, x.shape[0],
                              n_out, cin, cout, dt, precision, _ptr(y), _ptr(status), _ptr(ws),
                              0 if ws is None else ws.numel(), _stream(x.device))
    _check(code, "spc_conv_fwd")
    return y


SPC_ACT_NONE, SPC_ACT_RELU = 0, 1


def spc_conv_fwd_fused(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                       imap: Optional[torch.Tensor], mask: Optional[torch.Tensor] = None,
                       residual: Optional[torch.Tensor] = None, add_scale: float = 1.0,
                       act: int = SPC_ACT_NONE, n_out: Optional[int] = None,
                       precision: int = SPC_PREC_EXACT, out: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None,
                       ws: Optional[torch.Tensor] = None,
                       perm: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y[o] = act(bias + sum over pairs of x[imap[k, o]] W[k] + add_scale residual[o]);
    `perm` (with its `mask`) from spc_map_row_order(imap) groups the tiles' rows."""
    x = _cuda(x, "x")
    w = _cuda(w, "w").to(x.dtype)
    b = _cuda(bias, "bias").to(x.dtype) if bias is not None else None
    res = _cuda(residual, "residual").to(x.dtype) if residual is not None else None
    K, cin, cout = w.shape
    if imap is not None:
        imap = _cuda(imap, "imap")
        n_out = imap.shape[1]
    elif n_out is None:
        n_out = x.shape[0]
    y = torch.empty((n_out, cout), dtype=x.dtype, device=x.device) if out is None else out
    dt = _DTYPES[x.dtype]
    nbytes = int(lib().spc_conv_workspace_size(K, x.shape[0], n_out, cin, cout, dt))
    if nbytes and (ws is None or ws.numel() < nbytes):
        ws = _workspace(nbytes, x.device)
    code = lib().spc_conv_fwd_fused(_ptr(x), _ptr(w), _ptr(b), _ptr(imap), _ptr(mask), _ptr(perm), K,
                                    x.shape[0], n_out, cin, cout, dt, precision, _ptr(res),
                                    float(add_scale), int(act), _ptr(y), _ptr(status), _ptr(ws),
                                    0 if ws is None else ws.numel(), _stream(x.device))
    _check(code, "spc_conv_fwd_fused")
    return y


def spc_maxpool_fwd(x: torch.Tensor, imap: torch.Tensor, mask: Optional[torch.Tensor] = None,
                    with_arg: bool = True, out: Optional[torch.Tensor] = None,
                    arg: Optional[torch.Tensor] = None):
    """Sparse max pool on a strided map imap [K, N_out]: returns (y [N_out, C], arg) where
    arg [N_out, C] uint8 holds the offset each channel took (None unless with_arg)."""
    x = _cuda(x, "x")
    m = _cuda(imap, "imap")
    K, n_out = m.shape
    c = x.shape[1]
    y = torch.empty((n_out, c), dtype=x.dtype, device=x.device) if out is None else out
    if with_arg and arg is None:
        arg = torch.empty((n_out, c), dtype=torch.uint8, device=x.device)
    code = lib().spc_maxpool_fwd(_ptr(x), _ptr(m), _ptr(mask), K, x.shape[0], n_out, c,
                                 _DTYPES[x.dtype], _ptr(y), _ptr(arg if with_arg else None),
                                 _stream(x.device))
    _check(code, "spc_maxpool_fwd")
    return y, (arg if with_arg else None)


def spc_maxpool_dgrad(dy: torch.Tensor, imap_t: torch.Tensor, arg: torch.Tensor,
                      out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Gradient of spc_maxpool_fwd through the transposed map imap_t [K, N_in]."""
    dy = _cuda(dy, "dy")
    mt = _cuda(imap_t, "imap_t")
    K, n_in = mt.shape
    c = dy.shape[1]
    dx = torch.empty((n_in, c), dtype=dy.dtype, device=dy.device) if out is None else out
    code = lib().spc_maxpool_dgrad(_ptr(dy), _ptr(mt), _ptr(_cuda(arg, "arg")), K, n_in,
                                   dy.shape[0], c, _DTYPES[dy.dtype], _ptr(dx), _stream(dy.device))
    _check(code, "spc_maxpool_dgrad")
    return dx


def spc_map_row_order(map_: Optional[torch.Tensor], ws: Optional[torch.Tensor] = None,
                      mask: Optional[torch.Tensor] = None, K: Optional[int] = None,
                      perm: Optional[torch.Tensor] = None):
    """(mask [n] uint32, perm [n] int32): rows of map [K, n] grouped by offset mask.

    With map_ None, `mask` (the row masks spc_build_indice_map wrote) and `K`
    are read instead of the map.  Passing `ws` and `perm` (and `mask`) avoids
    allocation (e.g. inside CUDA-graph capture)."""
    if map_ is not None:
        m = _cuda(map_, "map")
        K, n = m.shape
        dev = m.device
        mask = torch.empty(n, dtype=torch.int32, device=dev) if mask is None else mask
    else:
        m = None
        assert mask is not None and K is not None
        n, dev = mask.shape[0], mask.device
    perm = torch.empty(n, dtype=torch.int32, device=dev) if perm is None else perm
    nbytes = int(lib().spc_map_row_order_workspace_size(n))
    if ws is None or ws.numel() < nbytes:
        ws = _workspace(nbytes, dev)
    code = lib().spc_map_row_order(_ptr(m), int(K), n, _ptr(mask), _ptr(perm), _ptr(ws), ws.numel(),
                                   _stream(dev))
    _check(code, "spc_map_row_order")
    return mask, perm


def spc_conv_inverse(y: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                     imap_t: torch.Tensor, precision: int = SPC_PREC_EXACT,
                     out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                     ws: Optional[torch.Tensor] = None, mask_t: Optional[torch.Tensor] = None,
                     perm: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Inverse of a strided conv through its transposed map imap_t [K, N_in]:
    out[i] = bias + sum over pairs imap_t[k, i] = o of y[o] W[k]; out [N_in, Cout].
    mask_t / perm from spc_map_row_order(imap_t) let the kernel skip unused offsets."""
    y = _cuda(y, "y")
    w = _cuda(w, "w").to(y.dtype)
    b = _cuda(bias, "bias").to(y.dtype) if bias is not None else None
    m = _cuda(imap_t, "imap_t")
    K, cy, cout = w.shape
    n_out = m.shape[1]
    o = torch.empty((n_out, cout), dtype=y.dtype, device=y.device) if out is None else out
    dt = _DTYPES[y.dtype]
    nbytes = int(lib().spc_conv_workspace_size(K, y.shape[0], n_out, cy, cout, dt))
    if nbytes and (ws is None or ws.numel() < nbytes):
        ws = _workspace(nbytes, y.device)
    code = lib().spc_conv_inverse(_ptr(y), _ptr(w), _ptr(b), _ptr(m), _ptr(mask_t), _ptr(perm), K,
                                  y.shape[0], n_out, cy, cout, dt, precision, _ptr(o),
                                  _ptr(status), _ptr(ws), 0 if ws is None else ws.numel(),
                                  _stream(y.device))
    _check(code, "spc_conv_inverse")
    return o


def spc_conv_fwd_int8(x: torch.Tensor, w: torch.Tensor, scale: torch.Tensor,
                      bias: Optional[torch.Tensor], imap: Optional[torch.Tensor],
                      mask: Optional[torch.Tensor] = None, perm: Optional[torch.Tensor] = None,
                      add: Optional[torch.Tensor] = None, add_scale: float = 0.0,
                      act: int = SPC_ACT_NONE, n_out: Optional[int] = None,
                      out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                      ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quantized forward: int8 x [n_in, cin], int8 w [K, cin, cout], fp32 per-channel
    scale and bias, optional int8 residual `add` with `add_scale`, optional ReLU;
    returns int8 [n_out, cout].  `perm` / `mask` from spc_map_row_order(imap)
    group rows by offset mask (spconv's do_sort); None keeps map order."""
    x = _cuda(x, "x")
    w = _cuda(w, "w")
    assert x.dtype == torch.int8 and w.dtype == torch.int8
    sc = _cuda(scale, "scale").to(torch.float32).contiguous()
    b = _cuda(bias, "bias").to(torch.float32).contiguous() if bias is not None else None
    K, cin, cout = w.shape
    if imap is not None:
        imap = _cuda(imap, "imap")
        n_out = imap.shape[1]
    elif n_out is None:
        n_out = x.shape[0]
    y = torch.empty((n_out, cout), dtype=torch.int8, device=x.device) if out is None else out
    nbytes = int(lib().spc_conv_int8_workspace_size(K, cin, cout))
    if ws is None or ws.numel() < nbytes:
        ws = _workspace(max(nbytes, 256), x.device)
    code = lib().spc_conv_fwd_int8(_ptr(x), _ptr(w), _ptr(sc), _ptr(b), _ptr(imap), _ptr(mask),
                                   _ptr(perm), K, x.shape[0], n_out, cin, cout, _ptr(add),
                                   float(add_scale), act, _ptr(y), _ptr(status), _ptr(ws),
                                   ws.numel(), _stream(x.device))
    _check(code, "spc_conv_fwd_int8")
    return y


def spc_conv_dgrad(dy: torch.Tensor, w: torch.Tensor, map_: Optional[torch.Tensor], kind: int,
                   n_in: int, precision: int = SPC_PREC_EXACT, mask: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None,
                   perm: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dx[i] = sum over pairs imap[k, o] = i of W[k] dy[o]; `perm` orders the
    input-row tiles (for a submanifold map, the forward's row order)."""
    dy = _cuda(dy, "dy")
    w = _cuda(w, "w").to(dy.dtype)
    K, cin, cout = w.shape
    m = _cuda(map_, "map") if map_ is not None else None
    dx = torch.empty((n_in, cin), dtype=dy.dtype, device=dy.device) if out is None else out
    dt = _DTYPES[dy.dtype]
    code = lib().spc_conv_dgrad(_ptr(dy), _ptr(w), _ptr(m), kind, _ptr(mask), _ptr(perm), K, n_in,
                                dy.shape[0], cin, cout, dt, precision, _ptr(dx), _ptr(status),
                                None, 0, _stream(dy.device))
    _check(code, "spc_conv_dgrad")
    return dx


def spc_conv_wgrad(x: torch.Tensor, dy: torch.Tensor, imap: Optional[torch.Tensor], K: int,
                   precision: int = SPC_PREC_EXACT, out: Optional[torch.Tensor] = None,
                   ws: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dW[k] = sum over pairs of x[imap[k, o]]^T dy[o], float32 [K, cin, cout]."""
    x = _cuda(x, "x")
    dy = _cuda(dy, "dy").to(x.dtype)
    m = _cuda(imap, "imap") if imap is not None else None
    cin, cout = x.shape[1], dy.shape[1]
    dw = torch.empty((K, cin, cout), dtype=torch.float32, device=x.device) if out is None else out
    dt = _DTYPES[x.dtype]
    nbytes = int(lib().spc_conv_wgrad_workspace_size(K, x.shape[0], dy.shape[0], cin, cout, dt))
    if ws is None or ws.numel() < nbytes:
        ws = _workspace(nbytes, x.device)
    code = lib().spc_conv_wgrad(_ptr(x), _ptr(dy), _ptr(m), K, x.shape[0], dy.shape[0], cin, cout,
                                dt, precision, _ptr(dw), _ptr(status), _ptr(ws), ws.numel(),
                                _stream(x.device))
    _check(code, "spc_conv_wgrad")
    return dw
