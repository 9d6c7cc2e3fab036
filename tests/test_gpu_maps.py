"""GPU parity of the indice-map and output-set kernels against the oracle.

Integer results must be bit-exact: the submanifold map [K, N], the strided
out->in map [K, N_out] and its transpose [K, N], the pair counts, the row masks
and the strided output coordinate set (sorted by (b, z, y, x))."""

import numpy as np
import pytest
import torch

import oracle
import scenes
import sparse_convolution_hash_gb300 as spc
from gpu_util import dev, rand_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def check_subm(coords, batch, shape, ks=3, dil=1):
    m = spc.spc_build_indice_map(torch.from_numpy(coords).to(dev()), batch, shape, ksize=ks,
                                 dil=dil, subm=True)
    spc.check_status(m["status"], "build")
    imap_ref, cnt_ref = oracle.subm_map(coords, batch, shape, ks, dil)
    imap = m["imap"].cpu().numpy()
    np.testing.assert_array_equal(imap, imap_ref)
    np.testing.assert_array_equal(m["pair_count"].cpu().numpy(), cnt_ref)
    if m["mask"] is not None:
        mask = m["mask"].cpu().numpy().astype(np.uint32)
        want = np.zeros(coords.shape[0], dtype=np.uint32)
        for k in range(imap_ref.shape[0]):
            want |= (imap_ref[k] >= 0).astype(np.uint32) << np.uint32(k)
        np.testing.assert_array_equal(mask, want)
    return m


@pytest.mark.parametrize("n,batch,shape,ks,dil", [
    (1, 1, (4, 4, 4), 3, 1),
    (7, 1, (4, 4, 4), 3, 1),
    (333, 2, (9, 8, 7), 3, 1),
    (1000, 3, (10, 10, 10), (3, 1, 5), (1, 2, 1)),
    (2501, 1, (17, 13, 13), 5, 1),
    (64, 1, (4, 4, 4), 3, 1),          # every cell of the grid occupied
    (500, 2, (12, 12, 12), 1, 1),
])
def test_subm_map_small(n, batch, shape, ks, dil):
    g = np.random.default_rng(n)
    check_subm(rand_coords(g, n, batch, shape), batch, shape, ks, dil)


@pytest.mark.parametrize("kind", ["uniform32", "lidar", "shell256", "shell192x4"])
def test_subm_map_workloads(kind):
    c = scenes.coords_for(kind)
    batch = int(c[:, 0].max()) + 1
    shape = {"uniform32": (32, 32, 32), "lidar": (41, 1600, 1408), "shell256": (256, 256, 256),
             "shell192x4": (192, 192, 192)}[kind]
    check_subm(c, batch, shape)


def test_subm_map_empty_and_deterministic():
    c = np.zeros((0, 4), dtype=np.int32)
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(dev()), 1, (4, 4, 4), subm=True)
    spc.check_status(m["status"])
    assert m["imap"].shape == (27, 0)
    assert int(m["pair_count"].sum()) == 0
    c = scenes.coords_for("uniform32")
    a = spc.spc_build_indice_map(torch.from_numpy(c).to(dev()), 1, (32, 32, 32))
    b = spc.spc_build_indice_map(torch.from_numpy(c).to(dev()), 1, (32, 32, 32))
    assert torch.equal(a["imap"], b["imap"]) and torch.equal(a["mask"], b["mask"])


def test_subm_map_errors():
    c = np.array([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=np.int32)
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(dev()), 1, (4, 4, 4))
    with pytest.raises(spc.SpcError) as e:
        spc.check_status(m["status"])
    assert e.value.code == 3
    c = np.array([[0, 1, 1, 1], [0, 2, 4, 2]], dtype=np.int32)
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(dev()), 1, (4, 4, 4))
    with pytest.raises(spc.SpcError) as e:
        spc.check_status(m["status"])
    assert e.value.code == 2
    c = np.array([[1, 1, 1, 1]], dtype=np.int32)
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(dev()), 1, (4, 4, 4))
    with pytest.raises(spc.SpcError) as e:
        spc.check_status(m["status"])
    assert e.value.code == 2


def check_strided(coords, batch, shape, ks, st, pd, dl):
    dc = torch.from_numpy(coords).to(dev())
    oc, out_shape = spc.spc_strided_out_coords(dc, batch, shape, ks, st, pd, dl)
    oc_ref = oracle.strided_out_coords(coords, batch, shape, ks, st, pd, dl)
    assert out_shape == oracle.out_shape(shape, ks, st, pd, dl)
    np.testing.assert_array_equal(oc.cpu().numpy(), oc_ref)
    m = spc.spc_build_indice_map(dc, batch, shape, ksize=ks, stride=st, pad=pd, dil=dl, subm=False,
                                 out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    imap_ref, imap_t_ref, cnt_ref = oracle.strided_map(coords, oc_ref, batch, shape, ks, st, pd, dl)
    np.testing.assert_array_equal(m["imap"].cpu().numpy(), imap_ref)
    np.testing.assert_array_equal(m["imap_t"].cpu().numpy(), imap_t_ref)
    np.testing.assert_array_equal(m["pair_count"].cpu().numpy(), cnt_ref)
    return oc, m


@pytest.mark.parametrize("n,batch,shape,ks,st,pd,dl", [
    (1, 1, (5, 5, 5), 3, 2, 1, 1),
    (300, 2, (9, 10, 11), 3, 2, 1, 1),
    (700, 1, (16, 9, 12), (3, 2, 3), (2, 2, 1), (0, 1, 1), (1, 1, 2)),
    (5000, 3, (20, 20, 20), 2, 2, 0, 1),
    (4097, 1, (33, 31, 29), 3, 3, 1, 1),
    # few voxels in a large grid: the output-grid bitmap would not fit the
    # candidates' key space, so these take the radix-sort path
    (3, 1, (200, 210, 190), 3, 2, 1, 1),
    (40, 2, (128, 128, 128), 2, 2, 0, 1),
])
def test_strided_small(n, batch, shape, ks, st, pd, dl):
    g = np.random.default_rng(n + 7)
    check_strided(rand_coords(g, n, batch, shape), batch, shape, ks, st, pd, dl)


def test_strided_uniform32_k3s2p1():
    oc, m = check_strided(scenes.coords_for("uniform32"), 1, (32, 32, 32), 3, 2, 1, 1)
    assert oc.shape[0] > 2000


def test_strided_lidar_k3s2p1():
    c = scenes.coords_for("lidar")
    check_strided(c, 2, (41, 1600, 1408), 3, 2, 1, 1)


def test_strided_golden_empty_output():
    c = torch.tensor([[0, 7, 153, 142]], dtype=torch.int32, device=dev())
    oc, out_shape = spc.spc_strided_out_coords(c, 1, (8, 200, 200), 3, 2, (0, 1, 1), 1)
    assert oc.shape[0] == 0
    assert out_shape == (3, 100, 100)
    m = spc.spc_build_indice_map(c, 1, (8, 200, 200), ksize=3, stride=2, pad=(0, 1, 1),
                                 subm=False, out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    assert m["imap"].shape == (27, 0)
    assert (m["imap_t"] == -1).all()


def test_strided_capacity_error_reports_size():
    c = scenes.coords_for("uniform32")
    n_ref = oracle.strided_out_coords(c, 1, (32, 32, 32), 3, 2, 1, 1).shape[0]
    with pytest.raises(spc.SpcError) as e:
        spc.spc_strided_out_coords(torch.from_numpy(c).to(dev()), 1, (32, 32, 32), 3, 2, 1, 1,
                                   cap=n_ref - 1)
    assert e.value.code == 5
    oc, _ = spc.spc_strided_out_coords(torch.from_numpy(c).to(dev()), 1, (32, 32, 32), 3, 2, 1, 1,
                                       cap=n_ref)
    assert oc.shape[0] == n_ref


def test_strided_range_error():
    c = torch.tensor([[0, 1, 1, 1], [0, 9, 1, 1]], dtype=torch.int32, device=dev())
    with pytest.raises(spc.SpcError) as e:
        spc.spc_strided_out_coords(c, 1, (8, 8, 8), 3, 2, 1, 1)
    assert e.value.code == 2


@pytest.mark.parametrize("case", ["full grid sorted", "sorted", "shuffled", "x-pairs"])
def test_subm_map_x_runs(case):
    """Submanifold 3x3x3 maps of at least 4,096 rows take side columns of each
    line from the neighbouring rows of an x-run: rows in (b, z, y, x) order
    (every row adjacent on a full grid; runs broken at random in a sparse set),
    the same set shuffled (no adjacency), and runs of two (adjacent pairs that
    straddle warp boundaries)."""
    g = np.random.default_rng(31)
    if case == "full grid sorted":
        z, y, x = np.meshgrid(np.arange(16), np.arange(16), np.arange(16), indexing="ij")
        coords = np.stack([np.zeros(4096), z.ravel(), y.ravel(), x.ravel()], 1).astype(np.int32)
        batch, shape = 1, (16, 16, 16)
    elif case == "x-pairs":
        batch, shape = 2, (24, 24, 24)
        cells = g.choice(batch * 24 * 24 * 12, size=6000, replace=False)
        b, zz, yy, xx = np.unravel_index(cells, (batch, 24, 24, 12))
        left = np.stack([b, zz, yy, 2 * xx], 1)
        coords = np.concatenate([left, left + np.array([0, 0, 0, 1])]).astype(np.int32)
        order = np.lexsort((coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]))
        coords = np.ascontiguousarray(coords[order])
    else:
        batch, shape = 2, (30, 30, 30)
        coords = rand_coords(g, 20000, batch, shape)
        order = np.lexsort((coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]))
        coords = np.ascontiguousarray(coords[order] if case == "sorted" else coords)
    check_subm(coords, batch, shape)
