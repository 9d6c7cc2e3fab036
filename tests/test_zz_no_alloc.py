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


def call_noalloc(f, coords, batch, shape, ksize=3, stride=1, pad=1, subm=True, out_coords=None,
                 with_transpose=False):
    dev = torch.device("cuda:0")
    c = torch.from_numpy(coords).to(dev) if isinstance(coords, np.ndarray) else coords
    n = c.shape[0]
    g = binding.make_geom(ksize, stride, pad, 1)
    K = ksize ** 3
    oc = None if subm else out_coords
    n_out = n if subm else oc.shape[0]
    imap = torch.empty((K, n_out), dtype=torch.int32, device=dev)
    imap_t = torch.empty((K, n), dtype=torch.int32, device=dev) if with_transpose else None
    cnt = torch.empty(K, dtype=torch.int32, device=dev)
    mask = torch.empty(n_out, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    ptr = (lambda t: None if t is None else t.data_ptr())
    code = f(c.data_ptr(), n, batch, (ctypes.c_int32 * 3)(*shape), ctypes.byref(g), 1 if subm else 0,
             ptr(oc), n_out, imap.data_ptr(), ptr(imap_t), cnt.data_ptr(), mask.data_ptr(),
             status.data_ptr(), stream)
    assert code == 0, binding.spc_status_string(code)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return imap, cnt, mask, imap_t


def test_noalloc_matches_workspace_build_twice(noalloc):
    cases = [(scenes.coords_for("lidar"), 2, (41, 1600, 1408)),
             (scenes.coords_for("uniform32"), 1, (32, 32, 32))]
    for coords, batch, shape in cases:
        imap, cnt, mask, _ = call_noalloc(noalloc, coords, batch, shape)
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


def test_noalloc_strided_map_with_transpose(noalloc):
    """k3 s2 p1 on the 2,000-voxel set: the table is sized from the input set
    while the map has the (different) number of output rows."""
    coords = scenes.coords_for("uniform32")
    shape = (32, 32, 32)
    c = torch.from_numpy(coords).cuda()
    oc, _ = spc.spc_strided_out_coords(c, 1, shape, 3, 2, 1, 1)
    assert oc.shape[0] != c.shape[0]
    for _ in range(2):
        imap, cnt, mask, imap_t = call_noalloc(noalloc, c, 1, shape, ksize=3, stride=2, pad=1,
                                               subm=False, out_coords=oc, with_transpose=True)
        ref = spc.spc_build_indice_map(c, 1, shape, ksize=3, stride=2, pad=1, subm=False,
                                       out_coords=oc, with_transpose=True)
        spc.check_status(ref["status"])
        assert torch.equal(imap, ref["imap"])
        assert torch.equal(imap_t, ref["imap_t"])
        assert torch.equal(cnt, ref["pair_count"])
        assert torch.equal(mask, ref["mask"])


def test_noalloc_accepts_exactly_the_maximum(noalloc):
    """MAX_VOXELS distinct voxels fill the fixed table to its load-factor limit."""
    rng = np.random.default_rng(20261202)
    side = 192
    cells = rng.choice(side ** 3, size=MAX_VOXELS, replace=False)
    coords = np.zeros((MAX_VOXELS, 4), dtype=np.int32)
    coords[:, 1] = cells // (side * side)
    coords[:, 2] = (cells // side) % side
    coords[:, 3] = cells % side
    c = torch.from_numpy(coords).cuda()
    imap, cnt, mask, _ = call_noalloc(noalloc, c, 1, (side, side, side))
    ref = spc.spc_build_indice_map(c, 1, (side, side, side))
    spc.check_status(ref["status"])
    assert torch.equal(imap, ref["imap"])
    assert torch.equal(cnt, ref["pair_count"])
    assert torch.equal(mask, ref["mask"])


def test_noalloc_allocates_nothing(noalloc):
    """After a first call (which looks up the table's address), further calls
    leave both torch's allocator and the device's free memory unchanged."""
    dev = torch.device("cuda:0")
    coords = scenes.coords_for("lidar")
    c = torch.from_numpy(coords).to(dev)
    n = c.shape[0]
    g = binding.make_geom(3, 1, 1, 1)
    imap = torch.empty((27, n), dtype=torch.int32, device=dev)
    cnt = torch.empty(27, dtype=torch.int32, device=dev)
    mask = torch.empty(n, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    shape = (ctypes.c_int32 * 3)(41, 1600, 1408)

    def once():
        code = noalloc(c.data_ptr(), n, 2, shape, ctypes.byref(g), 1, None, n, imap.data_ptr(), None,
                       cnt.data_ptr(), mask.data_ptr(), status.data_ptr(), stream)
        assert code == 0, binding.spc_status_string(code)

    once()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(5):
        once()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.cuda.memory_allocated(dev) == alloc0
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
