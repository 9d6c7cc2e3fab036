"""The allocation-free indice-map build (spc_build_indice_map_noalloc).

Some callers cannot allocate device memory when they need an indice map (an
engine's enqueue step that must not call cudaMalloc, a framework that owns all
device memory and offers no workspace).  This entry point keeps its hash table
in a fixed array inside the library instead of a caller workspace.  It must
give exactly the maps, pair counts and row masks of spc_build_indice_map, on
two calls in a row with different coordinate sets (the shared table is reused
and must be cleared in between).  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import scenes
import sparse_convolution_hash_gb300 as spc
from sparse_convolution_hash_gb300 import binding

pytestmark = pytest.mark.gpu

MAX_VOXELS = 1048576  # SPC_NOALLOC_MAX_VOXELS in include/spc.h


@pytest.fixture(scope="module")
def noalloc():
    import __graft_entry__

    __graft_entry__.build()
    L = binding.lib()
    f = L.spc_build_indice_map_noalloc
    p = ctypes.c_void_p
    f.argtypes = [p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32 * 3,
                  ctypes.POINTER(binding.Geom), ctypes.c_int32, p, ctypes.c_int64, p, p, p, p, p, p]
    f.restype = ctypes.c_int32
    return f


def call_noalloc(f, coords, batch, shape):
    dev = torch.device("cuda:0")
    c = torch.from_numpy(coords).to(dev)
    n = c.shape[0]
    g = binding.make_geom(3, 1, 1, 1)
    imap = torch.empty((27, n), dtype=torch.int32, device=dev)
    cnt = torch.empty(27, dtype=torch.int32, device=dev)
    mask = torch.empty(n, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    code = f(c.data_ptr(), n, batch, (ctypes.c_int32 * 3)(*shape), ctypes.byref(g), 1, None, n,
             imap.data_ptr(), None, cnt.data_ptr(), mask.data_ptr(), status.data_ptr(), stream)
    assert code == 0, binding.spc_status_string(code)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return imap, cnt, mask


def test_noalloc_matches_workspace_build_twice(noalloc):
    cases = [(scenes.coords_for("lidar"), 2, (41, 1600, 1408)),
             (scenes.coords_for("uniform32"), 1, (32, 32, 32))]
    for coords, batch, shape in cases:
        imap, cnt, mask = call_noalloc(noalloc, coords, batch, shape)
        ref = spc.spc_build_indice_map(torch.from_numpy(coords).cuda(), batch, shape)
        spc.check_status(ref["status"])
        assert torch.equal(imap, ref["imap"])
        assert torch.equal(cnt, ref["pair_count"])
        assert torch.equal(mask, ref["mask"])


def test_noalloc_rejects_oversized_input(noalloc):
    g = binding.make_geom(3, 1, 1, 1)
    code = noalloc(None, MAX_VOXELS + 1, 1, (ctypes.c_int32 * 3)(1024, 1024, 1024),
                   ctypes.byref(g), 1, None, MAX_VOXELS + 1, None, None, None, None, None, None)
    assert code == 8  # SPC_ERR_WORKSPACE
