"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its host-only logic (output grid, workspace sizing, argument
checks that return before any work is enqueued) behaves as documented."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from sparse_convolution_hash_gb300 import binding
from sparse_convolution_hash_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return binding.lib()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"\b(spc_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (spc_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_status_strings_and_version(L):
    assert binding.spc_version() >= 100
    for code in range(10):
        assert binding.spc_status_string(code)
    assert binding.spc_status_string(99) == "unknown status"


@pytest.mark.parametrize("shape,ks,st,pd,dl", [
    ((8, 200, 200), 3, 2, (0, 1, 1), 1),
    ((41, 1600, 1408), 3, 2, 1, 1),
    ((32, 32, 32), 3, 2, 1, 1),
    ((5, 7, 9), (3, 2, 1), (3, 2, 1), (0, 1, 2), (2, 1, 1)),
    ((2, 2, 2), 5, 1, 0, 1),
])
def test_out_shape_matches_oracle(L, shape, ks, st, pd, dl):
    assert binding.spc_out_shape(shape, ks, st, pd, dl) == oracle.out_shape(shape, ks, st, pd, dl)


def test_workspace_sizes(L):
    assert binding.spc_indice_map_workspace_size(0) >= 256
    assert binding.spc_indice_map_workspace_size(400000) >= 8 * 2 * 400000
    g = binding.make_geom(3, 2, 1, 1)
    assert L.spc_strided_out_coords_workspace_size(2000, ctypes.byref(g)) >= 2 * 8 * 27 * 2000
    assert L.spc_conv_wgrad_workspace_size(27, 1000, 1000, 64, 64, binding.SPC_BF16) > 0
    assert L.spc_conv_wgrad_workspace_size(0, 1000, 1000, 64, 64, binding.SPC_BF16) == 0


def _i3(v):
    return (ctypes.c_int32 * 3)(*v)


def test_argument_errors_return_before_any_work(L):
    g = binding.make_geom(3, 1, 1, 1)
    E = 1  # SPC_ERR_INVALID_ARG
    # negative sizes, zero batch, bad grid
    assert L.spc_build_indice_map(None, -1, 1, _i3((4, 4, 4)), ctypes.byref(g), 1, None, -1, None,
                                  None, None, None, None, None, 0, None) == E
    assert L.spc_build_indice_map(None, 0, 0, _i3((4, 4, 4)), ctypes.byref(g), 1, None, 0, None,
                                  None, None, None, None, None, 0, None) == E
    assert L.spc_build_indice_map(None, 0, 1, _i3((0, 4, 4)), ctypes.byref(g), 1, None, 0, None,
                                  None, None, None, None, None, 0, None) == E
    # submanifold needs odd kernels and n_out == n_in
    g2 = binding.make_geom(2, 1, 0, 1)
    st = ctypes.c_void_p(16)
    assert L.spc_build_indice_map(ctypes.c_void_p(256), 4, 1, _i3((4, 4, 4)), ctypes.byref(g2), 1,
                                  None, 4, ctypes.c_void_p(256), None, ctypes.c_void_p(256), None,
                                  st, ctypes.c_void_p(256), 1 << 20, None) == E
    # misaligned coordinates
    assert L.spc_build_indice_map(ctypes.c_void_p(260), 4, 1, _i3((4, 4, 4)), ctypes.byref(g), 1,
                                  None, 4, ctypes.c_void_p(256), None, ctypes.c_void_p(256), None,
                                  st, ctypes.c_void_p(256), 1 << 20, None) == E
    # workspace too small
    assert L.spc_build_indice_map(ctypes.c_void_p(256), 4, 1, _i3((4, 4, 4)), ctypes.byref(g), 1,
                                  None, 4, ctypes.c_void_p(256), None, ctypes.c_void_p(256), None,
                                  st, ctypes.c_void_p(256), 8, None) == 8
    # mask only for K <= 32
    g5 = binding.make_geom(5, 1, 2, 1)
    assert L.spc_build_indice_map(ctypes.c_void_p(256), 4, 1, _i3((8, 8, 8)), ctypes.byref(g5), 1,
                                  None, 4, ctypes.c_void_p(256), None, ctypes.c_void_p(256),
                                  ctypes.c_void_p(256), st, ctypes.c_void_p(256), 1 << 20,
                                  None) == E
    # conv: bad dtype, missing map for K > 1, misaligned weight
    assert L.spc_conv_fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), None, None, None, 27, 4, 4,
                          8, 8, 7, 0, ctypes.c_void_p(256), None, None, 0, None) == E
    assert L.spc_conv_fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), None, None, None, 27, 4, 4,
                          8, 8, 0, 0, ctypes.c_void_p(256), None, None, 0, None) == E
    assert L.spc_conv_fwd(ctypes.c_void_p(256), ctypes.c_void_p(258), None, ctypes.c_void_p(256),
                          None, 27, 4, 4, 8, 8, 0, 0, ctypes.c_void_p(256), None, None, 0,
                          None) == E
    # fused forward: unknown activation, misaligned residual, residual aliasing the output
    fz = L.spc_conv_fwd_fused
    assert fz(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256), None, None, 27, 4,
              4, 8, 8, 0, 0, None, 1.0, 2, ctypes.c_void_p(512), None, None, 0, None) == E
    assert fz(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256), None, None, 27, 4,
              4, 8, 8, 0, 0, ctypes.c_void_p(260), 1.0, 1, ctypes.c_void_p(512), None, None, 0,
              None) == E
    assert fz(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256), None, None, 27, 4,
              4, 8, 8, 0, 0, ctypes.c_void_p(512), 1.0, 1, ctypes.c_void_p(512), None, None, 0,
              None) == E
    # max pool: offsets beyond the uint8 argmax, a mask with K > 32, a missing map
    assert L.spc_maxpool_fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), None, 255, 4, 4, 8, 0,
                             ctypes.c_void_p(512), None, None) == E
    assert L.spc_maxpool_fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256), 125,
                             4, 4, 8, 0, ctypes.c_void_p(512), None, None) == E
    assert L.spc_maxpool_fwd(ctypes.c_void_p(256), None, None, 27, 4, 4, 8, 0,
                             ctypes.c_void_p(512), None, None) == E
    assert L.spc_maxpool_dgrad(ctypes.c_void_p(256), None, ctypes.c_void_p(256), 27, 4, 4, 8, 0,
                               ctypes.c_void_p(512), None) == E
    # inverse conv: the transposed map is required; bad dtype, misaligned weight, and a
    # row order with K > 32 rejected
    inv = L.spc_conv_inverse
    assert inv(ctypes.c_void_p(256), ctypes.c_void_p(256), None, None, None, None, 27, 4, 4, 8, 8,
               0, 0, ctypes.c_void_p(256), None, None, 0, None) == E
    assert inv(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256), None, None,
               27, 4, 4, 8, 8, 7, 0, ctypes.c_void_p(256), None, None, 0, None) == E
    assert inv(ctypes.c_void_p(256), ctypes.c_void_p(258), None, ctypes.c_void_p(256), None, None,
               27, 4, 4, 8, 8, 0, 0, ctypes.c_void_p(256), None, None, 0, None) == E
    assert inv(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256), None,
               ctypes.c_void_p(256), 125, 4, 4, 8, 8, 0, 0, ctypes.c_void_p(256), None, None, 0,
               None) == E
    # row order: K beyond the mask bits, missing output, too small a workspace
    assert L.spc_map_row_order(ctypes.c_void_p(256), 33, 4, None, ctypes.c_void_p(256),
                               ctypes.c_void_p(256), 1 << 20, None) == E
    assert L.spc_map_row_order(ctypes.c_void_p(256), 27, 4, None, None, ctypes.c_void_p(256),
                               1 << 20, None) == E
    assert L.spc_map_row_order(ctypes.c_void_p(256), 27, 4, None, ctypes.c_void_p(256),
                               ctypes.c_void_p(256), 8, None) == 8
    assert L.spc_map_row_order_workspace_size(1000) >= 16 * 1000
    # a row order needs the map or, instead, the build's masks as input
    assert L.spc_map_row_order(None, 27, 4, None, ctypes.c_void_p(256), ctypes.c_void_p(256),
                               1 << 20, None) == E
    # 16-bit rows of multiples of 64 channels read W as stored: no workspace;
    # the 32-channel rows take a transposed copy (as does tf32), which the
    # tensor-core path requires
    assert L.spc_conv_workspace_size(27, 4, 4, 128, 128, binding.SPC_BF16) == 0
    assert L.spc_conv_workspace_size(27, 4, 4, 32, 128, binding.SPC_BF16) == 27 * 32 * 128 * 2
    assert L.spc_conv_workspace_size(27, 4, 4, 64, 64, binding.SPC_F32) == 27 * 64 * 64 * 4
    assert L.spc_conv_fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256),
                          None, 27, 4, 4, 32, 128, binding.SPC_BF16, 0, ctypes.c_void_p(256),
                          None, None, 0, None) == 8
    assert L.spc_conv_dgrad(ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
                            binding.SPC_MAP_SUBM_MIRROR, None, None, 27, 4, 5, 8, 8, 0, 0,
                            ctypes.c_void_p(256), None, None, 0, None) == E
    # a mask or a row order needs K <= 32
    assert L.spc_conv_dgrad(ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
                            binding.SPC_MAP_TRANSPOSED, None, ctypes.c_void_p(256), 125, 4, 4, 8, 8,
                            0, 0, ctypes.c_void_p(256), None, None, 0, None) == E
    assert fz(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.c_void_p(256), None,
              ctypes.c_void_p(256), 125, 4, 4, 8, 8, 0, 0, None, 1.0, 0, ctypes.c_void_p(512),
              None, None, 0, None) == E
    assert L.spc_conv_wgrad(ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256), 27,
                            4, 4, 8, 8, 2, 0, ctypes.c_void_p(256), None, None, 0, None) == 8
    # strided out coords: null n_out / status
    gs = binding.make_geom(3, 2, 1, 1)
    assert L.spc_strided_out_coords(ctypes.c_void_p(256), 4, 1, _i3((8, 8, 8)), ctypes.byref(gs),
                                    _i3((0, 0, 0)), ctypes.c_void_p(256), 10, None, None, None, 0,
                                    None) == E


def test_hash_key_capacity_is_checked(L):
    # a grid too large for the packed key beside the row field is refused, not mis-keyed
    g = binding.make_geom(3, 1, 1, 1)
    big = _i3((2 ** 30, 2 ** 30, 2 ** 10))
    st = ctypes.c_void_p(16)
    r = L.spc_build_indice_map(ctypes.c_void_p(256), 4, 1, big, ctypes.byref(g), 1, None, 4,
                               ctypes.c_void_p(256), None, ctypes.c_void_p(256), None, st,
                               ctypes.c_void_p(256), 1 << 20, None)
    assert r == 6  # SPC_ERR_UNSUPPORTED


def test_binding_refuses_without_library(monkeypatch):
    monkeypatch.setattr(binding, "LIB_PATH", "/nonexistent/libspc.so")
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(binding.SpcLibraryMissing):
        binding.lib()


def test_noalloc_context_cache_logic(tmp_path):
    """The allocation-free build caches its table's device address per CUDA
    context id; compiled and run on the host with the library's own header."""
    exe = tmp_path / "ctx_cache_check"
    src = os.path.join(ROOT, "tests", "ctx_cache_check.cpp")
    inc = os.path.join(ROOT, "sparse_convolution_hash_gb300", "csrc")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", inc, src, "-o", str(exe), "-lpthread"],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "ctx cache ok" in out.stdout


def test_wait_limit_setting(L):
    old = binding.spc_get_wait_limit_ns()
    assert old == 2_000_000_000
    try:
        binding.spc_set_wait_limit_ns(12345)
        assert binding.spc_get_wait_limit_ns() == 12345
        with pytest.raises(binding.SpcError):
            binding.spc_set_wait_limit_ns(61_000_000_000)
        assert binding.spc_get_wait_limit_ns() == 12345
    finally:
        binding.spc_set_wait_limit_ns(old)
    assert binding.spc_get_wait_limit_ns() == old


def test_int8_host_checks(L):
    """The quantized forward's argument checks and workspace size (no launch)."""
    P = ctypes.c_void_p
    f = L.spc_conv_fwd_int8
    assert L.spc_conv_int8_workspace_size(27, 128, 128) == 27 * 2 * 128 * 128 * 2
    # K * cin beyond the exact range, or channels not multiples of 64: unsupported, size 0
    assert L.spc_conv_int8_workspace_size(27, 320, 64) == 0
    assert L.spc_conv_int8_workspace_size(27, 48, 64) == 0
    args = lambda **o: [o.get("x", P(256)), o.get("w", P(256)), o.get("scale", P(256)), None,
                        P(256), None, None, o.get("K", 27), 4, 4, o.get("cin", 64),
                        o.get("cout", 64), o.get("add"), 1.0, o.get("act", 0), o.get("y", P(512)),
                        None, o.get("ws", None), o.get("wsb", 0), None]
    assert f(*args(scale=None)) == 1          # scale required
    assert f(*args(w=P(258))) == 1            # misaligned weights
    assert f(*args(act=2)) == 1               # unknown activation
    assert f(*args(add=P(512))) == 1          # residual aliasing the output
    assert f(*args(cin=320)) == 6             # K * cin > 8192
    assert f(*args(cout=96)) == 6             # cout not a multiple of 64
    assert f(*args()) == 8                    # workspace missing
    assert f(*args(ws=P(256), wsb=1024)) == 8  # workspace too small
