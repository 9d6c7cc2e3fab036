"""GPU parity of the convolution kernels against the fp64 oracle.

Floating-point results are compared normwise, ||gpu - oracle|| / ||oracle||,
within 1e-5 (fp32 exact), 2e-3 (tf32) and 2e-2 (fp16 / bf16).  Small cases
are compared in full; the full-size workloads on sampled rows (first and last
tiles, the ragged tail, and random rows) or sampled dW entries, which the
oracle computes one by one.  Run-to-run bit identity is checked too."""

import numpy as np
import pytest
import torch

import oracle
import scenes
import sparse_convolution_hash_gb300 as spc
from gpu_util import TOL, DT, dev, normwise, rand_coords, rand_tensor, sample_rows, to_np

pytestmark = pytest.mark.gpu

SHAPES = {"uniform32": (32, 32, 32), "lidar": (41, 1600, 1408), "shell256": (256, 256, 256),
          "shell192x4": (192, 192, 192)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def subm_case(coords, batch, shape, cin, cout, dtype, ks=3, seed=0, bias=True):
    g = np.random.default_rng(seed)
    n = coords.shape[0]
    K = ks ** 3
    x = rand_tensor(g, (n, cin), dtype)
    w = rand_tensor(g, (K, cin, cout), dtype, std=float(np.sqrt(1.0 / (K * cin))))
    b = rand_tensor(g, (cout,), dtype, std=0.1) if bias else None
    dy = rand_tensor(g, (n, cout), dtype)
    m = spc.spc_build_indice_map(torch.from_numpy(coords).to(dev()), batch, shape, ksize=ks)
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(coords, batch, shape, ks)
    return x, w, b, dy, m, imap_ref


@pytest.mark.parametrize("dtype,prec", [("f32", "exact"), ("f32", "tf32"), ("f16", "exact"),
                                        ("bf16", "exact")])
@pytest.mark.parametrize("n,cin,cout", [(1, 8, 8), (777, 16, 16), (1500, 24, 40),
                                        (2100, 64, 128), (900, 128, 96), (640, 32, 32),
                                        (333, 16, 32), (1029, 32, 16), (515, 8, 16),
                                        (1000, 128, 128), (3000, 64, 64), (700, 192, 64),
                                        (513, 64, 256), (129, 128, 64), (600, 16, 64),
                                        (450, 32, 128)])
def test_subm_small_full(dtype, prec, n, cin, cout):
    g = np.random.default_rng(n)
    batch, shape = 2, (12, 11, 13)
    coords = rand_coords(g, n, batch, shape)
    x, w, b, dy, m, imap_ref = subm_case(coords, batch, shape, cin, cout, dtype, seed=n)
    p = spc.SPC_PREC_TF32 if prec == "tf32" else spc.SPC_PREC_EXACT
    d = dev()
    tol = TOL[(dtype, prec)]
    y_ref = oracle.conv_fwd(x, w, b, imap_ref)
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], m["mask"], precision=p)
    assert normwise(to_np(y), y_ref) < tol
    y_nomask = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], None, precision=p)
    assert normwise(to_np(y_nomask), y_ref) < tol
    dx_ref = oracle.conv_dgrad(dy, w, imap_ref, n)
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap"], spc.SPC_MAP_SUBM_MIRROR, n, precision=p)
    assert normwise(to_np(dx), dx_ref) < tol
    dxm = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap"], spc.SPC_MAP_SUBM_MIRROR, n, precision=p,
                             mask=m["mask"])
    assert normwise(to_np(dxm), dx_ref) < tol
    dw = spc.spc_conv_wgrad(x.to(d), dy.to(d), m["imap"], 27, precision=p)
    assert normwise(to_np(dw), oracle.conv_wgrad(x, dy, imap_ref)) < tol


@pytest.mark.parametrize("dtype,cin,cout", [("f32", 16, 16), ("bf16", 64, 64), ("f16", 32, 16)])
def test_subm_k5(dtype, cin, cout):
    """5^3 kernel (K = 125, beyond the 32-bit offset masks): forward, mirrored
    dinput and dfilter (its offset groups of 3 and 4) in full."""
    g = np.random.default_rng(cin * 7 + cout)
    batch, shape = 1, (9, 10, 8)
    coords = rand_coords(g, 400, batch, shape)
    x, w, b, dy, m, imap_ref = subm_case(coords, batch, shape, cin, cout, dtype, ks=5, seed=cin)
    d = dev()
    tol = TOL[(dtype, "exact")]
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], None)
    assert normwise(to_np(y), oracle.conv_fwd(x, w, b, imap_ref)) < tol
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap"], spc.SPC_MAP_SUBM_MIRROR, 400)
    assert normwise(to_np(dx), oracle.conv_dgrad(dy, w, imap_ref, 400)) < tol
    dw = spc.spc_conv_wgrad(x.to(d), dy.to(d), m["imap"], 125)
    assert normwise(to_np(dw), oracle.conv_wgrad(x, dy, imap_ref)) < tol


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_k1_gemm_shortcut(dtype):
    g = np.random.default_rng(5)
    n, cin, cout = 1234, 32, 48
    x = rand_tensor(g, (n, cin), dtype)
    w = rand_tensor(g, (1, cin, cout), dtype, std=0.2)
    b = rand_tensor(g, (cout,), dtype, std=0.1)
    d = dev()
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), None)
    ref = x.double().numpy() @ w[0].double().numpy() + b.double().numpy()
    assert normwise(to_np(y), ref) < TOL[(dtype, "exact")]
    dy = rand_tensor(g, (n, cout), dtype)
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), None, spc.SPC_MAP_TRANSPOSED, n)
    assert normwise(to_np(dx), dy.double().numpy() @ w[0].double().numpy().T) < TOL[(dtype, "exact")]
    dw = spc.spc_conv_wgrad(x.to(d), dy.to(d), None, 1)
    assert normwise(to_np(dw)[0], x.double().numpy().T @ dy.double().numpy()) < TOL[(dtype, "exact")]


def test_uniform32_subm_f32_full():
    """2,000 voxels in 32^3, fp32 16->16 with bias: the whole output at 1e-5."""
    w = scenes.workload("uniform32_subm_f32")
    d = dev()
    m = spc.spc_build_indice_map(torch.from_numpy(w["coords"]).to(d), 1, (32, 32, 32))
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(w["coords"], 1, (32, 32, 32))
    y = spc.spc_conv_fwd(w["x"].to(d), w["w"].to(d), w["bias"].to(d), m["imap"], m["mask"])
    assert normwise(to_np(y), oracle.conv_fwd(w["x"], w["w"], w["bias"], imap_ref)) < 1e-5
    y2 = spc.spc_conv_fwd(w["x"].to(d), w["w"].to(d), w["bias"].to(d), m["imap"], m["mask"])
    assert torch.equal(y, y2)


def test_uniform32_strided_bf16():
    """k3 s2 p1 on the 2,000-voxel set, bf16 64->128: fwd, dinput, dfilter in full."""
    w = scenes.workload("uniform32_strided_bf16")
    c = w["coords"]
    d = dev()
    dc = torch.from_numpy(c).to(d)
    oc, _ = spc.spc_strided_out_coords(dc, 1, (32, 32, 32), 3, 2, 1, 1)
    m = spc.spc_build_indice_map(dc, 1, (32, 32, 32), ksize=3, stride=2, pad=1, subm=False,
                                 out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    oc_ref = oracle.strided_out_coords(c, 1, (32, 32, 32), 3, 2, 1, 1)
    imap_ref, imap_t_ref, _ = oracle.strided_map(c, oc_ref, 1, (32, 32, 32), 3, 2, 1, 1)
    y = spc.spc_conv_fwd(w["x"].to(d), w["w"].to(d), None, m["imap"], m["mask"])
    assert normwise(to_np(y), oracle.conv_fwd(w["x"], w["w"], None, imap_ref)) < 2e-2
    g = np.random.default_rng(3)
    dy = rand_tensor(g, (oc.shape[0], 128), "bf16")
    dx = spc.spc_conv_dgrad(dy.to(d), w["w"].to(d), m["imap_t"], spc.SPC_MAP_TRANSPOSED, c.shape[0])
    assert normwise(to_np(dx), oracle.conv_dgrad(dy, w["w"], imap_ref, c.shape[0])) < 2e-2
    dw = spc.spc_conv_wgrad(w["x"].to(d), dy.to(d), m["imap"], 27)
    assert normwise(to_np(dw), oracle.conv_wgrad(w["x"], dy, imap_ref)) < 2e-2


@pytest.mark.parametrize("dtype,cin,cout", [("bf16", 128, 128), ("f16", 64, 128), ("bf16", 128, 64)])
def test_strided_k2_wide(dtype, cin, cout):
    """k2 s2 (8 offsets) with wide channels, which selects the tensor-core tile
    shapes for few offsets (two CTAs of 2 x 128 rows per SM, also with 128-wide
    weight stages): forward and dinput in full, several tiles and a ragged tail."""
    g = np.random.default_rng(cin + 3 * cout)
    batch, shape, n = 2, (24, 22, 26), 3000
    c = rand_coords(g, n, batch, shape)
    d = dev()
    dc = torch.from_numpy(c).to(d)
    oc, _ = spc.spc_strided_out_coords(dc, batch, shape, 2, 2, 0, 1)
    m = spc.spc_build_indice_map(dc, batch, shape, ksize=2, stride=2, pad=0, subm=False,
                                 out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    oc_ref = oracle.strided_out_coords(c, batch, shape, 2, 2, 0, 1)
    imap_ref, _, _ = oracle.strided_map(c, oc_ref, batch, shape, 2, 2, 0, 1)
    assert oc_ref.shape[0] > 4 * 256
    x = rand_tensor(g, (n, cin), dtype)
    w = rand_tensor(g, (8, cin, cout), dtype, std=float(np.sqrt(1.0 / (8 * cin))))
    b = rand_tensor(g, (cout,), dtype, std=0.1)
    tol = TOL[(dtype, "exact")]
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], m["mask"])
    assert normwise(to_np(y), oracle.conv_fwd(x, w, b, imap_ref)) < tol
    dy = rand_tensor(g, (oc_ref.shape[0], cout), dtype)
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap_t"], spc.SPC_MAP_TRANSPOSED, n)
    assert normwise(to_np(dx), oracle.conv_dgrad(dy, w, imap_ref, n)) < tol


@pytest.mark.parametrize("dtype,cin,cout", [("bf16", 128, 128), ("f16", 128, 64)])
def test_subm_k1_wide_full(dtype, cin, cout):
    """1 x 1 x 1 submanifold conv through its (identity) map with wide channels:
    the one-offset tensor-core tiles, whole output and dinput."""
    g = np.random.default_rng(cout)
    batch, shape = 2, (12, 11, 13)
    coords = rand_coords(g, 1700, batch, shape)
    x, w, b, dy, m, imap_ref = subm_case(coords, batch, shape, cin, cout, dtype, ks=1, seed=cin)
    d = dev()
    tol = TOL[(dtype, "exact")]
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], m["mask"])
    assert normwise(to_np(y), oracle.conv_fwd(x, w, b, imap_ref)) < tol
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap"], spc.SPC_MAP_SUBM_MIRROR, 1700)
    assert normwise(to_np(dx), oracle.conv_dgrad(dy, w, imap_ref, 1700)) < tol


@pytest.mark.parametrize("n,cin,cout,dtype,prec", [(777, 16, 16, "f16", "exact"),
                                                  (1000, 128, 128, "bf16", "exact"),
                                                  (3000, 64, 64, "bf16", "exact"),
                                                  (600, 16, 64, "f16", "exact"),
                                                  (1500, 24, 40, "f32", "exact"),
                                                  (800, 64, 128, "f32", "tf32")])
@pytest.mark.parametrize("res_scale,relu", [(1.0, True), (None, True), (0.5, False)])
def test_fused_epilogue(n, cin, cout, dtype, prec, res_scale, relu):
    """Residual add and ReLU in the forward's epilogue, on every forward kernel."""
    g = np.random.default_rng(n + cin)
    batch, shape = 2, (12, 11, 13)
    coords = rand_coords(g, n, batch, shape)
    x, w, b, _, m, imap_ref = subm_case(coords, batch, shape, cin, cout, dtype, seed=n)
    res = rand_tensor(g, (n, cout), dtype) if res_scale is not None else None
    d = dev()
    p = spc.SPC_PREC_TF32 if prec == "tf32" else spc.SPC_PREC_EXACT
    y = spc.spc_conv_fwd_fused(x.to(d), w.to(d), b.to(d), m["imap"], m["mask"],
                               residual=res.to(d) if res is not None else None,
                               add_scale=res_scale if res_scale is not None else 1.0,
                               act=spc.SPC_ACT_RELU if relu else spc.SPC_ACT_NONE, precision=p)
    ref = oracle.conv_fwd_fused(x, w, b, imap_ref, res, res_scale or 1.0, relu)
    assert normwise(to_np(y), ref) < TOL[(dtype, prec)]
    if relu:
        assert (to_np(y) >= 0).all()


@pytest.mark.parametrize("dtype,cy,cout", [("bf16", 128, 64), ("f16", 64, 64), ("f32", 16, 16),
                                           ("bf16", 32, 32), ("bf16", 64, 16), ("f16", 24, 40),
                                           ("bf16", 64, 128), ("f32", 64, 192)])
def test_inverse_conv_strided(dtype, cy, cout):
    """Inverse of the k3 s2 p1 conv on the 2,000-voxel set: output, and both
    gradients through the documented spc_conv_dgrad / spc_conv_wgrad calls."""
    w = scenes.workload("uniform32_strided_bf16")
    c = w["coords"]
    d = dev()
    dc = torch.from_numpy(c).to(d)
    oc, _ = spc.spc_strided_out_coords(dc, 1, (32, 32, 32), 3, 2, 1, 1)
    m = spc.spc_build_indice_map(dc, 1, (32, 32, 32), ksize=3, stride=2, pad=1, subm=False,
                                 out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    oc_ref = oracle.strided_out_coords(c, 1, (32, 32, 32), 3, 2, 1, 1)
    imap_ref, imap_t_ref, _ = oracle.strided_map(c, oc_ref, 1, (32, 32, 32), 3, 2, 1, 1)
    g = np.random.default_rng(cy * 1000 + cout)
    n_y, n = oc.shape[0], c.shape[0]
    y = rand_tensor(g, (n_y, cy), dtype)
    wt = rand_tensor(g, (27, cy, cout), dtype, std=float(np.sqrt(1.0 / (27 * cy))))
    b = rand_tensor(g, (cout,), dtype, std=0.1)
    tol = TOL[(dtype, "exact")]
    out = spc.spc_conv_inverse(y.to(d), wt.to(d), b.to(d), m["imap_t"])
    assert out.shape == (n, cout)
    ref = oracle.conv_inverse(y, wt, b, imap_ref, n)
    assert normwise(to_np(out), ref) < tol
    assert torch.equal(out, spc.spc_conv_inverse(y.to(d), wt.to(d), b.to(d), m["imap_t"]))
    # rows grouped by offset mask: a permutation, masks non-decreasing along it,
    # stable within a group, and the same result
    mask_t, perm = spc.spc_map_row_order(m["imap_t"])
    p_np, mk = perm.cpu().numpy(), mask_t.cpu().numpy().astype(np.uint32)
    assert np.array_equal(np.sort(p_np), np.arange(n))
    exp_mask = ((imap_t_ref >= 0) * (1 << np.arange(27, dtype=np.int64))[:, None]).sum(0)
    assert np.array_equal(mk.astype(np.int64), exp_mask)
    assert np.array_equal(p_np, np.lexsort((np.arange(n), exp_mask)))
    out_g = spc.spc_conv_inverse(y.to(d), wt.to(d), b.to(d), m["imap_t"], mask_t=mask_t, perm=perm)
    assert normwise(to_np(out_g), ref) < tol
    dout = rand_tensor(g, (n, cout), dtype)
    # dy[o] = sum over pairs imap[k, o] = i of W[k] dout[i]: the forward map read as transposed
    dy = spc.spc_conv_dgrad(dout.to(d), wt.to(d), m["imap"], spc.SPC_MAP_TRANSPOSED, n_y)
    wt_t = wt.double().numpy().transpose(0, 2, 1)
    assert normwise(to_np(dy), oracle.conv_fwd(dout, wt_t, None, imap_ref)) < tol
    # dW[k] = sum over pairs of y[o]^T dout[i]
    dw = spc.spc_conv_wgrad(y.to(d), dout.to(d), m["imap_t"], 27)
    assert normwise(to_np(dw), oracle.conv_wgrad(y, dout, imap_t_ref)) < tol


@pytest.mark.parametrize("ks,stride,pad", [(3, 2, 1), (2, 2, 0)])
@pytest.mark.parametrize("dtype,c", [("bf16", 64), ("f32", 16), ("f16", 24), ("f16", 7)])
def test_maxpool(ks, stride, pad, dtype, c):
    """Max pool on the 2,000-voxel set: values bit-exact (a max is exact in any
    precision), argmax offsets exact, gradient within the dtype's tolerance."""
    w = scenes.workload("uniform32_strided_bf16")
    coords = w["coords"]
    d = dev()
    dc = torch.from_numpy(coords).to(d)
    oc, _ = spc.spc_strided_out_coords(dc, 1, (32, 32, 32), ks, stride, pad, 1)
    m = spc.spc_build_indice_map(dc, 1, (32, 32, 32), ksize=ks, stride=stride, pad=pad, subm=False,
                                 out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    oc_ref = oracle.strided_out_coords(coords, 1, (32, 32, 32), ks, stride, pad, 1)
    imap_ref, _, _ = oracle.strided_map(coords, oc_ref, 1, (32, 32, 32), ks, stride, pad, 1)
    g = np.random.default_rng(ks * 100 + c)
    x = rand_tensor(g, (coords.shape[0], c), dtype)
    y_ref, arg_ref = oracle.maxpool_fwd(x, imap_ref)
    for mask in (None, m["mask"]):
        y, arg = spc.spc_maxpool_fwd(x.to(d), m["imap"], mask)
        assert np.array_equal(to_np(y), y_ref)
        assert np.array_equal(arg.cpu().numpy(), arg_ref)
    dy = rand_tensor(g, (oc.shape[0], c), dtype)
    dx = spc.spc_maxpool_dgrad(dy.to(d), m["imap_t"], arg)
    assert normwise(to_np(dx), oracle.maxpool_dgrad(dy, imap_ref, arg_ref, coords.shape[0])) < \
        TOL[(dtype, "exact")]


@pytest.mark.parametrize("name", ["lidar_subm_f16", "shell256_subm_bf16", "shell256_k1_bf16"])
def test_forward_workloads_sampled(name):
    w = scenes.workload(name)
    c = w["coords"]
    kind = name.split("_")[0]
    batch, shape = int(c[:, 0].max()) + 1, SHAPES[kind]
    ks = w["k"]
    d = dev()
    imap_ref, _ = oracle.subm_map(c, batch, shape, ks)
    if ks == 1:
        imap_dev, mask = None, None
    else:
        m = spc.spc_build_indice_map(torch.from_numpy(c).to(d), batch, shape, ksize=ks)
        spc.check_status(m["status"])
        imap_dev, mask = m["imap"], m["mask"]
    x, wt = w["x"].to(d), w["w"].to(d)
    b = w["bias"].to(d) if w["bias"] is not None else None
    y = spc.spc_conv_fwd(x, wt, b, imap_dev, mask, n_out=c.shape[0])
    rows = sample_rows(c.shape[0])
    ref = oracle.conv_fwd(w["x"], w["w"], w["bias"], imap_ref, rows=rows)
    assert normwise(to_np(y[torch.from_numpy(rows).to(d)]), ref) < TOL[(w["dtype"], "exact")]
    y2 = spc.spc_conv_fwd(x, wt, b, imap_dev, mask, n_out=c.shape[0])
    assert torch.equal(y, y2)


def test_training_step_shell192x4_sampled():
    """4 x 192^3 shells, bf16 64->64: fwd, dinput (mirror map) and dfilter."""
    w = scenes.workload("shell192x4_train_bf16")
    c = w["coords"]
    n = c.shape[0]
    d = dev()
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(d), 4, (192, 192, 192))
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(c, 4, (192, 192, 192))
    x, wt, dy = w["x"].to(d), w["w"].to(d), w["dy"].to(d)
    y = spc.spc_conv_fwd(x, wt, None, m["imap"], m["mask"])
    dx = spc.spc_conv_dgrad(dy, wt, m["imap"], spc.SPC_MAP_SUBM_MIRROR, n, mask=m["mask"])
    dw = spc.spc_conv_wgrad(x, dy, m["imap"], 27)
    rows = sample_rows(n, seed=1)
    r = torch.from_numpy(rows).to(d)
    assert normwise(to_np(y[r]), oracle.conv_fwd(w["x"], w["w"], None, imap_ref, rows=rows)) < 2e-2
    imap_t_ref = oracle.transpose_map(imap_ref, n)
    assert normwise(to_np(dx[r]), oracle.conv_dgrad_rows(w["dy"], w["w"], imap_t_ref, rows)) < 2e-2
    g = np.random.default_rng(2)
    ent = np.unique(np.concatenate([np.arange(64), g.integers(0, 27 * 64 * 64, size=400)]))
    ref = oracle.conv_wgrad_entries(w["x"], w["dy"], imap_ref, ent)
    assert normwise(to_np(dw).reshape(-1)[ent], ref) < 2e-2
    dw2 = spc.spc_conv_wgrad(x, dy, m["imap"], 27)
    dx2 = spc.spc_conv_dgrad(dy, wt, m["imap"], spc.SPC_MAP_SUBM_MIRROR, n, mask=m["mask"])
    assert torch.equal(dw, dw2) and torch.equal(dx, dx2)


def test_empty_conv():
    d = dev()
    x = torch.zeros((0, 16), dtype=torch.bfloat16, device=d)
    w = torch.zeros((27, 16, 16), dtype=torch.bfloat16, device=d)
    imap = torch.zeros((27, 0), dtype=torch.int32, device=d)
    assert spc.spc_conv_fwd(x, w, None, imap).shape == (0, 16)
    dw = spc.spc_conv_wgrad(x, torch.zeros((0, 16), dtype=torch.bfloat16, device=d), imap, 27)
    assert (dw == 0).all()


def test_dfilter_whole_offsets_shell192x4():
    """Every dW entry of three whole offsets (a corner, a face and the centre) on
    the full 4 x 192^3 training workload, where the split-row reduction is
    longest: against the oracle's per-entry sums, normwise per offset."""
    w = scenes.workload("shell192x4_train_bf16")
    c = w["coords"]
    d = dev()
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(d), 4, (192, 192, 192))
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(c, 4, (192, 192, 192))
    dw = to_np(spc.spc_conv_wgrad(w["x"].to(d), w["dy"].to(d), m["imap"], 27))
    cin, cout = w["cin"], w["cout"]
    for k in (0, 4, 13):
        ent = k * cin * cout + np.arange(cin * cout)
        ref = oracle.conv_wgrad_entries(w["x"], w["dy"], imap_ref, ent)
        assert normwise(dw.reshape(-1)[ent], ref) < 2e-2, k


def test_wait_limit_runs_out_with_a_status_and_the_context_survives():
    """With the wait limit at 0 the pipelined tensor-core kernels give up at the
    first stage handoff that is not already complete: the call's status word
    reads SPC_ERR_TIMEOUT and the kernels return (no hang, no fault).  With the
    limit restored the same context computes correct results."""
    g = np.random.default_rng(5)
    batch, shape = 2, (12, 11, 13)
    coords = rand_coords(g, 3000, batch, shape)
    x, w, b, dy, m, imap_ref = subm_case(coords, batch, shape, 64, 64, "bf16", seed=5, bias=False)
    d = dev()
    xd, wd, dyd = x.to(d), w.to(d), dy.to(d)
    old = spc.binding.spc_get_wait_limit_ns()
    assert old == 2_000_000_000
    timeouts = {"fwd": 0, "dgrad": 0, "wgrad": 0}
    try:
        spc.binding.spc_set_wait_limit_ns(0)
        for _ in range(3):
            for what in timeouts:
                st = spc.new_status(d)
                if what == "fwd":
                    spc.spc_conv_fwd(xd, wd, None, m["imap"], m["mask"], status=st)
                elif what == "dgrad":
                    spc.spc_conv_dgrad(dyd, wd, m["imap"], spc.SPC_MAP_SUBM_MIRROR, coords.shape[0],
                                       mask=m["mask"], status=st)
                else:
                    spc.spc_conv_wgrad(xd, dyd, m["imap"], 27, status=st)
                torch.cuda.synchronize()
                code = int(st.item())
                assert code in (0, 9), code  # SPC_OK or SPC_ERR_TIMEOUT
                timeouts[what] += code == 9
    finally:
        spc.binding.spc_set_wait_limit_ns(old)
    assert all(v > 0 for v in timeouts.values()), timeouts
    st = spc.new_status(d)
    y = spc.spc_conv_fwd(xd, wd, None, m["imap"], m["mask"], status=st)
    dw = spc.spc_conv_wgrad(xd, dyd, m["imap"], 27, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert normwise(to_np(y), oracle.conv_fwd(x, w, None, imap_ref)) < 2e-2
    assert normwise(to_np(dw), oracle.conv_wgrad(x, dy, imap_ref)) < 2e-2


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("n,cin,cout", [(1, 64, 64), (129, 128, 128), (1000, 64, 192),
                                        (3001, 128, 64), (700, 192, 128)])
def test_k1_dense_rows(dtype, n, cin, cout):
    """K = 1 on the identity map (no map): the tensor-core kernel loads whole row
    blocks with TMA; forward and dinput against the oracle, ragged tails included."""
    g = np.random.default_rng(n + cin + cout)
    x = rand_tensor(g, (n, cin), dtype)
    w = rand_tensor(g, (1, cin, cout), dtype, std=float(np.sqrt(1.0 / cin)))
    b = rand_tensor(g, (cout,), dtype, std=0.1)
    dy = rand_tensor(g, (n, cout), dtype)
    ident = np.arange(n, dtype=np.int32)[None, :]
    d = dev()
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), None, n_out=n)
    assert normwise(to_np(y), oracle.conv_fwd(x, w, b, ident)) < TOL[(dtype, "exact")]
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), None, spc.SPC_MAP_SUBM_MIRROR, n)
    assert normwise(to_np(dx), oracle.conv_dgrad(dy, w, ident, n)) < TOL[(dtype, "exact")]


@pytest.mark.parametrize("n,cin,cout", [(2100, 64, 128), (3000, 64, 64), (1000, 128, 128),
                                        (700, 192, 64), (600, 16, 64)])
def test_row_order_forward_and_dinput(n, cin, cout):
    """Tiles in mask-grouped row order (spc_map_row_order, from the map or from
    the build's masks): forward and dinput against the oracle and equal to the
    map-order results."""
    g = np.random.default_rng(n + 7)
    batch, shape = 2, (12, 11, 13)
    coords = rand_coords(g, n, batch, shape)
    x, w, b, dy, m, imap_ref = subm_case(coords, batch, shape, cin, cout, "bf16", seed=n)
    d = dev()
    mask_g, perm = spc.spc_map_row_order(m["imap"])
    mask_b, perm_b = spc.spc_map_row_order(None, mask=m["mask"].clone(), K=27)
    assert torch.equal(perm, perm_b) and torch.equal(mask_g, mask_b)
    assert torch.equal(torch.sort(perm.long()).values, torch.arange(n, device=d))
    y0 = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], m["mask"])
    y = spc.spc_conv_fwd(x.to(d), w.to(d), b.to(d), m["imap"], mask_g, perm=perm)
    assert normwise(to_np(y), oracle.conv_fwd(x, w, b, imap_ref)) < 2e-2
    assert torch.equal(y, y0)
    dx0 = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap"], spc.SPC_MAP_SUBM_MIRROR, n, mask=m["mask"])
    dx = spc.spc_conv_dgrad(dy.to(d), w.to(d), m["imap"], spc.SPC_MAP_SUBM_MIRROR, n, mask=mask_g,
                            perm=perm)
    assert normwise(to_np(dx), oracle.conv_dgrad(dy, w, imap_ref, n)) < 2e-2
    assert torch.equal(dx, dx0)


@pytest.mark.parametrize("cin,cout,dtype", [(64, 64, "bf16"), (16, 16, "f16"), (64, 128, "bf16")])
def test_inverse_of_an_empty_strided_output(cin, cout, dtype):
    """spconv's worked example (shape [8, 200, 200], k3 s2 pad [0, 1, 1], one point
    at z = 7) has an empty strided output; the inverse conv through its maps
    reads no row and writes the bias at the input site, and the forward of the
    empty set writes nothing."""
    d = dev()
    coords = np.array([[0, 7, 100, 100]], dtype=np.int32)
    shape = (8, 200, 200)
    dc = torch.from_numpy(coords).to(d)
    oc, oshape = spc.spc_strided_out_coords(dc, 1, shape, 3, 2, (0, 1, 1), 1)
    assert oc.shape[0] == 0
    m = spc.spc_build_indice_map(dc, 1, shape, ksize=3, stride=2, pad=(0, 1, 1), subm=False,
                                 out_coords=oc, with_transpose=True)
    spc.check_status(m["status"])
    assert int(m["pair_count"].sum().item()) == 0
    assert (m["imap_t"] == -1).all()
    g = np.random.default_rng(cin + cout)
    wt = rand_tensor(g, (27, cin, cout), dtype, std=0.1)
    b = rand_tensor(g, (cout,), dtype, std=0.5)
    y = torch.zeros((0, cin), dtype=DT[dtype], device=d)
    st = spc.new_status(d)
    out = spc.spc_conv_inverse(y, wt.to(d), b.to(d), m["imap_t"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert out.shape == (1, cout)
    ref = oracle.conv_inverse(y.cpu(), wt, b, m["imap"].cpu().numpy(), 1)
    assert np.array_equal(to_np(out), ref)
    assert np.array_equal(to_np(out)[0], to_np(b))
    fwd = spc.spc_conv_fwd(torch.ones((1, cin), dtype=DT[dtype], device=d), wt.to(d), b.to(d), m["imap"])
    assert fwd.shape == (0, cout)
