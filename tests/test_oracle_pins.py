"""Pins of the CPU oracle against things other than itself.

Each check fixes the oracle to an independent fact:
  * brute-force all-pairs neighbour search on tiny grids, with the offset order
    written the way the MLX SubMConv3d page builds it (numpy meshgrid 'ij');
  * torch's dense conv3d (a library cross-correlation) on a zero-filled grid,
    read back at occupied sites (submanifold) or over the dense output (strided);
  * torch autograd of that dense conv3d for dinput / dfilter;
  * closed forms: the 1x1 kernel is a plain GEMM, a centre-only identity kernel
    returns the input, translations leave maps and outputs unchanged, the
    forward is linear (central differences are exact), and the adjoint
    identities <dy, conv(x)> = <dgrad(dy), x> and <dy, conv_W(x)> = <dW, W>;
  * the worked example of spconv's COMMON_PROBLEMS page (empty output).
"""

import itertools
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import scenes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def page_offsets(ks, dil=(1, 1, 1)):
    """Offsets as the MLX page builds them: centred ranges, meshgrid 'ij', C order."""
    rz, ry, rx = (np.arange(k) - k // 2 for k in ks)
    grid = np.meshgrid(rz * dil[0], ry * dil[1], rx * dil[2], indexing="ij")
    return np.stack(grid, axis=-1).reshape(-1, 3)


def rand_coords(g, n, batch, shape):
    cells = g.choice(batch * int(np.prod(shape)), size=n, replace=False)
    b, z, y, x = np.unravel_index(cells, (batch,) + tuple(shape))
    return np.stack([b, z, y, x], axis=1).astype(np.int32)


def brute_subm_map(coords, shape, ks, dil):
    offs = page_offsets(ks, dil)
    n = coords.shape[0]
    imap = np.full((offs.shape[0], n), -1, dtype=np.int32)
    for o in range(n):
        for k, d in enumerate(offs):
            want = (coords[o, 0], coords[o, 1] + d[0], coords[o, 2] + d[1], coords[o, 3] + d[2])
            for i in range(n):
                if tuple(coords[i]) == want:
                    imap[k, o] = i
    return imap


def dense_grid(coords, feats, batch, shape):
    """[B, C, D, H, W] float64 grid with feats at the occupied cells, zero elsewhere."""
    c = feats.shape[1]
    g = torch.zeros((batch, c) + tuple(shape), dtype=torch.float64)
    t = torch.as_tensor(coords, dtype=torch.long)
    g[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]] = torch.as_tensor(feats, dtype=torch.float64)
    return g


def dense_weight(w, ks):
    """[K, Cin, Cout] with k in C order over (kz, ky, kx) -> conv3d weight [Cout, Cin, kz, ky, kx]."""
    K, cin, cout = w.shape
    wt = torch.as_tensor(w, dtype=torch.float64).reshape(ks[0], ks[1], ks[2], cin, cout)
    return wt.permute(4, 3, 0, 1, 2).contiguous()


# --------------------------------------------------------------------------- maps


@pytest.mark.parametrize("ks,dil,shape,batch,n", [
    ((3, 3, 3), (1, 1, 1), (5, 5, 5), 1, 50),
    ((3, 1, 3), (2, 1, 1), (6, 4, 7), 2, 60),
    ((1, 1, 1), (1, 1, 1), (4, 4, 4), 2, 30),
    ((5, 3, 3), (1, 1, 2), (7, 5, 6), 1, 80),
])
def test_subm_map_brute_force(ks, dil, shape, batch, n):
    g = np.random.default_rng(11)
    coords = rand_coords(g, n, batch, shape)
    imap, cnt = oracle.subm_map(coords, batch, shape, ks, dil)
    want = brute_subm_map(coords, shape, ks, dil)
    np.testing.assert_array_equal(imap, want)
    np.testing.assert_array_equal(cnt, (want >= 0).sum(axis=1))


def test_subm_map_symmetry_and_centre():
    c = scenes.uniform_cells(2000, (32, 32, 32), seed=1)
    imap, cnt = oracle.subm_map(c, 1, (32, 32, 32))
    K, n = imap.shape
    assert cnt[K // 2] == n
    np.testing.assert_array_equal(imap[K // 2], np.arange(n))
    for k in range(K):
        o = np.nonzero(imap[k] >= 0)[0]
        i = imap[k, o]
        np.testing.assert_array_equal(imap[K - 1 - k, i], o)
    # counts of mirrored offsets are equal
    np.testing.assert_array_equal(cnt, cnt[::-1])


def test_subm_map_translation_invariance():
    g = np.random.default_rng(5)
    c = rand_coords(g, 120, 2, (6, 6, 6))
    imap, cnt = oracle.subm_map(c, 2, (12, 12, 12))
    shifted = c.copy()
    shifted[:, 1:] += np.array([3, 5, 2], dtype=np.int32)
    imap2, cnt2 = oracle.subm_map(shifted, 2, (12, 12, 12))
    np.testing.assert_array_equal(imap, imap2)
    np.testing.assert_array_equal(cnt, cnt2)


def test_map_errors():
    c = np.array([[0, 1, 1, 1], [0, 1, 1, 1]], dtype=np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.subm_map(c, 1, (4, 4, 4))
    assert e.value.code == oracle.ERR_DUPLICATE
    c = np.array([[0, 1, 4, 1]], dtype=np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.subm_map(c, 1, (4, 4, 4))
    assert e.value.code == oracle.ERR_RANGE
    c = np.array([[1, 0, 0, 0]], dtype=np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.subm_map(c, 1, (4, 4, 4))
    assert e.value.code == oracle.ERR_RANGE


def test_empty_sets():
    c = np.zeros((0, 4), dtype=np.int32)
    imap, cnt = oracle.subm_map(c, 1, (4, 4, 4))
    assert imap.shape == (27, 0) and (cnt == 0).all()
    assert oracle.strided_out_coords(c, 1, (4, 4, 4)).shape == (0, 4)


# ------------------------------------------------------------- strided output set


def dense_reach(coords, batch, shape, ks, stride, pad, dil):
    occ = dense_grid(coords, np.ones((coords.shape[0], 1)), batch, shape)
    ones = torch.ones((1, 1) + tuple(ks), dtype=torch.float64)
    r = F.conv3d(occ, ones, stride=stride, padding=pad, dilation=dil)
    return r[:, 0]


@pytest.mark.parametrize("shape,ks,stride,pad,dil,batch,n", [
    ((8, 8, 8), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), 1, 40),
    ((9, 7, 10), (3, 3, 3), (2, 2, 2), (0, 1, 1), (1, 1, 1), 2, 70),
    ((10, 10, 6), (2, 2, 2), (2, 2, 2), (0, 0, 0), (1, 1, 1), 1, 50),
    ((11, 9, 9), (3, 3, 3), (3, 2, 1), (1, 0, 1), (1, 2, 1), 2, 90),
    ((7, 7, 7), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 1, 30),
])
def test_strided_out_set_dense_reach(shape, ks, stride, pad, dil, batch, n):
    g = np.random.default_rng(7)
    coords = rand_coords(g, n, batch, shape)
    reach = dense_reach(coords, batch, shape, ks, stride, pad, dil)
    assert oracle.out_shape(shape, ks, stride, pad, dil) == tuple(reach.shape[1:])
    want = np.argwhere(reach.numpy() > 0).astype(np.int32)  # C order = sorted (b, z, y, x)
    got = oracle.strided_out_coords(coords, batch, shape, ks, stride, pad, dil)
    np.testing.assert_array_equal(got, want)


def test_golden_common_problems_empty_output():
    spec = {}
    with open(os.path.join(GOLDEN, "spconv_common_problems_empty_output.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            spec[key] = [int(v) for v in vals]
    coords = np.array([spec["coord"]], dtype=np.int32)
    got = oracle.strided_out_coords(coords, spec["batch"][0], spec["spatial_shape"], spec["ksize"],
                                    spec["stride"], spec["padding"], spec["dilation"])
    assert got.shape[0] == spec["expected_n_out"][0]
    # the out-of-range axis is z: with padding 1 on z the point would survive
    got = oracle.strided_out_coords(coords, 1, spec["spatial_shape"], 3, 2, 1, 1)
    assert got.shape[0] > 0


def test_strided_map_vs_brute_force():
    g = np.random.default_rng(3)
    shape, ks, st, pd, dl = (9, 8, 7), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1)
    coords = rand_coords(g, 60, 2, shape)
    oc = oracle.strided_out_coords(coords, 2, shape, ks, st, pd, dl)
    imap, imap_t, cnt = oracle.strided_map(coords, oc, 2, shape, ks, st, pd, dl)
    offs = list(itertools.product(*(range(k) for k in ks)))
    want = np.full((len(offs), oc.shape[0]), -1, dtype=np.int32)
    for o in range(oc.shape[0]):
        for k, (a, b, c) in enumerate(offs):
            p = (oc[o, 0], oc[o, 1] * 2 - 1 + a, oc[o, 2] * 2 - 1 + b, oc[o, 3] * 2 - 1 + c)
            for i in range(coords.shape[0]):
                if tuple(coords[i]) == p:
                    want[k, o] = i
    np.testing.assert_array_equal(imap, want)
    np.testing.assert_array_equal(cnt, (want >= 0).sum(axis=1))
    np.testing.assert_array_equal(imap_t, oracle.transpose_map(want, coords.shape[0]))
    # every input reaches at least one output, so every input has some pair
    assert ((imap_t >= 0).sum(axis=0) > 0).all()


# ------------------------------------------------------------------- forward sums


def feats(g, n, c):
    return g.standard_normal((n, c))


@pytest.mark.parametrize("ks,dil,batch", [((3, 3, 3), (1, 1, 1), 2), ((3, 1, 5), (1, 2, 1), 1)])
def test_subm_fwd_vs_dense_conv3d(ks, dil, batch):
    g = np.random.default_rng(21)
    shape = (7, 6, 8)
    coords = rand_coords(g, 90, batch, shape)
    cin, cout = 3, 5
    x = feats(g, 90, cin)
    K = int(np.prod(ks))
    w = g.standard_normal((K, cin, cout))
    b = g.standard_normal(cout)
    imap, _ = oracle.subm_map(coords, batch, shape, ks, dil)
    y = oracle.conv_fwd(x, w, b, imap)
    pad = tuple((k // 2) * d for k, d in zip(ks, dil))
    dense = F.conv3d(dense_grid(coords, x, batch, shape), dense_weight(w, ks),
                     torch.as_tensor(b), padding=pad, dilation=dil)
    t = torch.as_tensor(coords, dtype=torch.long)
    want = dense[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]].numpy()
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape,ks,stride,pad,dil,batch", [
    ((8, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), 2),
    ((9, 7, 8), (2, 3, 3), (2, 1, 3), (0, 1, 2), (1, 1, 1), 1),
])
def test_strided_fwd_vs_dense_conv3d(shape, ks, stride, pad, dil, batch):
    g = np.random.default_rng(22)
    coords = rand_coords(g, 80, batch, shape)
    cin, cout = 4, 3
    x = feats(g, 80, cin)
    w = g.standard_normal((int(np.prod(ks)), cin, cout))
    oc = oracle.strided_out_coords(coords, batch, shape, ks, stride, pad, dil)
    imap, _, _ = oracle.strided_map(coords, oc, batch, shape, ks, stride, pad, dil)
    y = oracle.conv_fwd(x, w, None, imap)
    dense = F.conv3d(dense_grid(coords, x, batch, shape), dense_weight(w, ks),
                     stride=stride, padding=pad, dilation=dil)
    t = torch.as_tensor(oc, dtype=torch.long)
    np.testing.assert_allclose(y, dense[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]].numpy(),
                               rtol=1e-12, atol=1e-12)
    # the dense output vanishes everywhere outside the output set
    mask = torch.ones(dense.shape[0], *dense.shape[2:], dtype=torch.bool)
    mask[t[:, 0], t[:, 1], t[:, 2], t[:, 3]] = False
    assert dense.permute(0, 2, 3, 4, 1)[mask].abs().max().item() == 0.0


@pytest.mark.parametrize("shape,ks,stride,pad,dil,batch", [
    ((8, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), 2),
    ((10, 9, 11), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), 1),
    ((9, 7, 8), (2, 3, 3), (2, 1, 3), (0, 1, 2), (1, 1, 1), 1),
])
def test_inverse_vs_dense_conv_transpose3d(shape, ks, stride, pad, dil, batch):
    """The inverse conv of a strided conv (same maps) is the dense transposed
    convolution of the strided output, read back at the input sites."""
    g = np.random.default_rng(23)
    coords = rand_coords(g, 80, batch, shape)
    cy, cout = 4, 3
    oc = oracle.strided_out_coords(coords, batch, shape, ks, stride, pad, dil)
    imap, imap_t, _ = oracle.strided_map(coords, oc, batch, shape, ks, stride, pad, dil,
                                         with_transpose=True)
    y = feats(g, oc.shape[0], cy)
    w = g.standard_normal((int(np.prod(ks)), cy, cout))
    b = g.standard_normal(cout)
    out = oracle.conv_inverse(y, w, b, imap, coords.shape[0])
    oshape = oracle.out_shape(shape, ks, stride, pad, dil)
    opad = [shape[a] - ((oshape[a] - 1) * stride[a] - 2 * pad[a] + dil[a] * (ks[a] - 1) + 1)
            for a in range(3)]
    assert all(0 <= opad[a] < max(stride[a], dil[a]) for a in range(3))
    wt = torch.as_tensor(w, dtype=torch.float64).reshape(*ks, cy, cout).permute(3, 4, 0, 1, 2)
    dense = F.conv_transpose3d(dense_grid(oc, y, batch, oshape), wt.contiguous(),
                               torch.as_tensor(b, dtype=torch.float64), stride=stride,
                               padding=pad, output_padding=opad, dilation=dil)
    t = torch.as_tensor(coords, dtype=torch.long)
    np.testing.assert_allclose(out, dense[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]].numpy(),
                               rtol=1e-12, atol=1e-12)
    # the gather form over the transposed map gives the same rows
    np.testing.assert_allclose(out, oracle.conv_fwd(y, w, b, imap_t), rtol=1e-12, atol=1e-12)


def test_fused_epilogue_vs_dense_conv3d_relu():
    """conv + bias + s * residual, then ReLU: torch's dense conv3d and relu on a
    zero-filled grid, read at the occupied cells."""
    g = np.random.default_rng(31)
    shape, batch, ks = (7, 6, 8), 2, (3, 3, 3)
    coords = rand_coords(g, 90, batch, shape)
    cin, cout = 4, 5
    x = feats(g, 90, cin)
    w = g.standard_normal((27, cin, cout))
    b = g.standard_normal(cout)
    res = g.standard_normal((90, cout))
    imap, _ = oracle.subm_map(coords, batch, shape, 3)
    dense = F.conv3d(dense_grid(coords, x, batch, shape), dense_weight(w, ks),
                     torch.as_tensor(b, dtype=torch.float64), padding=1)
    t = torch.as_tensor(coords, dtype=torch.long)
    at = dense[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]]
    ref = torch.relu(at + 0.75 * torch.as_tensor(res)).numpy()
    got = oracle.conv_fwd_fused(x, w, b, imap, res, 0.75, relu=True)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert (got == 0).any() and (got > 0).any()  # the activation acts
    np.testing.assert_allclose(oracle.conv_fwd_fused(x, w, b, imap), at.numpy(), rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("shape,ks,stride,pad,batch", [
    ((8, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), 2),
    ((9, 8, 7), (2, 2, 2), (2, 2, 2), (0, 0, 0), 1),
])
def test_maxpool_vs_dense_max_pool3d(shape, ks, stride, pad, batch):
    """Sparse max pool = torch's dense max_pool3d over a grid holding -inf at empty
    cells, read at the strided output set; its gradient = torch autograd's."""
    g = np.random.default_rng(41)
    coords = rand_coords(g, 120, batch, shape)
    c = 5
    x = g.standard_normal((120, c))
    oc = oracle.strided_out_coords(coords, batch, shape, ks, stride, pad, 1)
    imap, _, _ = oracle.strided_map(coords, oc, batch, shape, ks, stride, pad, 1, False)
    y, arg = oracle.maxpool_fwd(x, imap)
    t = torch.as_tensor(coords, dtype=torch.long)
    xt = torch.as_tensor(x).clone().requires_grad_(True)
    # scatter x into the -inf grid differentiably
    flat = torch.full((batch * c * int(np.prod(shape)),), float("-inf"), dtype=torch.float64)
    cell = ((t[:, 0] * c)[:, None] + torch.arange(c)[None, :]) * int(np.prod(shape)) + \
        (((t[:, 1] * shape[1] + t[:, 2]) * shape[2]) + t[:, 3])[:, None]
    dense = flat.index_put((cell.reshape(-1),), xt.reshape(-1)).reshape((batch, c) + tuple(shape))
    pooled = F.max_pool3d(dense, ks, stride=stride, padding=pad)
    to = torch.as_tensor(oc, dtype=torch.long)
    at = pooled[to[:, 0], :, to[:, 1], to[:, 2], to[:, 3]]
    np.testing.assert_array_equal(y, at.detach().numpy())
    dy = g.standard_normal(at.shape)
    at.backward(torch.as_tensor(dy))
    np.testing.assert_allclose(oracle.maxpool_dgrad(dy, imap, arg, 120), xt.grad.numpy(),
                               rtol=1e-12, atol=1e-12)
    assert (arg < 255).all()  # every output of the strided set has an input


def test_k1_is_gemm():
    g = np.random.default_rng(23)
    coords = rand_coords(g, 200, 2, (9, 9, 9))
    x, w, b = feats(g, 200, 6), g.standard_normal((1, 6, 7)), g.standard_normal(7)
    imap, cnt = oracle.subm_map(coords, 2, (9, 9, 9), 1)
    assert cnt[0] == 200
    np.testing.assert_allclose(oracle.conv_fwd(x, w, b, imap), x @ w[0] + b, rtol=1e-13, atol=1e-13)


def test_centre_only_identity():
    c = scenes.uniform_cells(2000, (32, 32, 32), seed=1)
    g = np.random.default_rng(24)
    x, b = feats(g, 2000, 8), g.standard_normal(8)
    w = np.zeros((27, 8, 8))
    w[13] = np.eye(8)
    imap, _ = oracle.subm_map(c, 1, (32, 32, 32))
    np.testing.assert_array_equal(oracle.conv_fwd(x, w, b, imap), x + b)


def test_fwd_translation_invariance():
    g = np.random.default_rng(25)
    c = rand_coords(g, 150, 1, (7, 7, 7))
    x, w = feats(g, 150, 4), g.standard_normal((27, 4, 4))
    y1 = oracle.conv_fwd(x, w, None, oracle.subm_map(c, 1, (16, 16, 16))[0])
    c2 = c.copy()
    c2[:, 1:] += np.array([8, 1, 4], dtype=np.int32)
    y2 = oracle.conv_fwd(x, w, None, oracle.subm_map(c2, 1, (16, 16, 16))[0])
    np.testing.assert_array_equal(y1, y2)


def test_fwd_rows_matches_full():
    g = np.random.default_rng(26)
    c = rand_coords(g, 300, 1, (8, 8, 8))
    x, w, b = feats(g, 300, 5), g.standard_normal((27, 5, 6)), g.standard_normal(6)
    imap, _ = oracle.subm_map(c, 1, (8, 8, 8))
    rows = np.array([0, 17, 299, 5, 5])
    np.testing.assert_array_equal(oracle.conv_fwd(x, w, b, imap, rows=rows),
                                  oracle.conv_fwd(x, w, b, imap)[rows])


# ----------------------------------------------------------------------- backward


def _subm_case(seed, n=110, batch=2, shape=(6, 7, 6), cin=3, cout=4):
    g = np.random.default_rng(seed)
    coords = rand_coords(g, n, batch, shape)
    x, w = feats(g, n, cin), g.standard_normal((27, cin, cout))
    dy = g.standard_normal((n, cout))
    imap, _ = oracle.subm_map(coords, batch, shape)
    return coords, x, w, dy, imap


def test_backward_vs_dense_autograd_subm():
    coords, x, w, dy, imap = _subm_case(31)
    batch, shape = 2, (6, 7, 6)
    xg = dense_grid(coords, x, batch, shape).requires_grad_(True)
    wt = dense_weight(w, (3, 3, 3)).requires_grad_(True)
    out = F.conv3d(xg, wt, padding=1)
    t = torch.as_tensor(coords, dtype=torch.long)
    loss = (out[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]] * torch.as_tensor(dy)).sum()
    loss.backward()
    dx_want = xg.grad[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]].numpy()
    dw_want = wt.grad.permute(2, 3, 4, 1, 0).reshape(27, 3, 4).numpy()
    np.testing.assert_allclose(oracle.conv_dgrad(dy, w, imap, x.shape[0]), dx_want,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.conv_wgrad(x, dy, imap), dw_want, rtol=1e-12, atol=1e-11)


def test_backward_vs_dense_autograd_strided():
    g = np.random.default_rng(32)
    shape, batch, cin, cout = (9, 8, 7), 2, 3, 5
    coords = rand_coords(g, 90, batch, shape)
    x, w = feats(g, 90, cin), g.standard_normal((27, cin, cout))
    oc = oracle.strided_out_coords(coords, batch, shape, 3, 2, 1, 1)
    imap, imap_t, _ = oracle.strided_map(coords, oc, batch, shape, 3, 2, 1, 1)
    dy = g.standard_normal((oc.shape[0], cout))
    xg = dense_grid(coords, x, batch, shape).requires_grad_(True)
    wt = dense_weight(w, (3, 3, 3)).requires_grad_(True)
    out = F.conv3d(xg, wt, stride=2, padding=1)
    to = torch.as_tensor(oc, dtype=torch.long)
    (out[to[:, 0], :, to[:, 1], to[:, 2], to[:, 3]] * torch.as_tensor(dy)).sum().backward()
    t = torch.as_tensor(coords, dtype=torch.long)
    dx_want = xg.grad[t[:, 0], :, t[:, 1], t[:, 2], t[:, 3]].numpy()
    np.testing.assert_allclose(oracle.conv_dgrad(dy, w, imap, 90), dx_want, rtol=1e-12, atol=1e-12)
    rows = np.arange(90)
    np.testing.assert_allclose(oracle.conv_dgrad_rows(dy, w, imap_t, rows), dx_want,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.conv_wgrad(x, dy, imap),
                               wt.grad.permute(2, 3, 4, 1, 0).reshape(27, cin, cout).numpy(),
                               rtol=1e-12, atol=1e-11)


def test_central_differences():
    coords, x, w, dy, imap = _subm_case(33, n=60, shape=(5, 5, 5), cin=2, cout=3)
    L = lambda xx, ww: float((oracle.conv_fwd(xx, ww, None, imap) * dy).sum())
    dx = oracle.conv_dgrad(dy, w, imap, x.shape[0])
    dw = oracle.conv_wgrad(x, dy, imap)
    h = 0.5  # the loss is linear in x and in w, so central differences are exact
    for (i, c) in [(0, 0), (7, 1), (59, 0), (31, 1)]:
        xp, xm = x.copy(), x.copy()
        xp[i, c] += h
        xm[i, c] -= h
        assert abs((L(xp, w) - L(xm, w)) / (2 * h) - dx[i, c]) < 1e-10
    for (k, c, j) in [(0, 0, 0), (13, 1, 2), (26, 0, 1), (4, 1, 1)]:
        wp, wm = w.copy(), w.copy()
        wp[k, c, j] += h
        wm[k, c, j] -= h
        assert abs((L(x, wp) - L(x, wm)) / (2 * h) - dw[k, c, j]) < 1e-10


def test_adjoint_identities():
    coords, x, w, dy, imap = _subm_case(34, n=300, shape=(8, 8, 8), cin=5, cout=6)
    y = oracle.conv_fwd(x, w, None, imap)
    dx = oracle.conv_dgrad(dy, w, imap, x.shape[0])
    dw = oracle.conv_wgrad(x, dy, imap)
    lhs = float((dy * y).sum())
    assert abs(lhs - float((dx * x).sum())) <= 1e-11 * max(1.0, abs(lhs))
    assert abs(lhs - float((dw * w).sum())) <= 1e-11 * max(1.0, abs(lhs))


def test_subm_dgrad_is_fwd_with_mirrored_transposed_weight():
    coords, x, w, dy, imap = _subm_case(35, n=200, shape=(7, 7, 7), cin=4, cout=3)
    w_m = np.ascontiguousarray(w[::-1].transpose(0, 2, 1))
    np.testing.assert_allclose(oracle.conv_dgrad(dy, w, imap, 200),
                               oracle.conv_fwd(dy, w_m, None, imap), rtol=1e-12, atol=1e-12)


def test_sampled_helpers_match_full():
    coords, x, w, dy, imap = _subm_case(36, n=150, shape=(7, 6, 7), cin=3, cout=4)
    imap_t = oracle.transpose_map(imap, 150)
    rows = np.array([3, 0, 149, 77])
    np.testing.assert_allclose(oracle.conv_dgrad_rows(dy, w, imap_t, rows),
                               oracle.conv_dgrad(dy, w, imap, 150)[rows], rtol=1e-13, atol=1e-13)
    ent = np.array([0, 5, 27 * 12 - 1, 13 * 12 + 7])
    np.testing.assert_allclose(oracle.conv_wgrad_entries(x, dy, imap, ent),
                               oracle.conv_wgrad(x, dy, imap).reshape(-1)[ent], rtol=1e-13,
                               atol=1e-13)


# ------------------------------------------------------------------ int8 rule

def test_int8_golden_two_voxels():
    """Hand-worked cases of the int8 rule (rounding ties, ReLU, saturation, the
    residual add) on a two-voxel scene: tests/golden/int8_two_voxel_rule.txt."""
    c = np.array([[0, 0, 0, 0], [0, 0, 0, 1]], dtype=np.int32)
    imap, _ = oracle.subm_map(c, 1, (4, 4, 4))
    x = np.array([[3], [-5]], dtype=np.int8)
    w = np.zeros((27, 1, 1), dtype=np.int8)
    w[13], w[14], w[12] = 2, 7, -1
    rows = 0
    for line in open(os.path.join(GOLDEN, "int8_two_voxel_rule.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        sc, b, a0, a1, asc, relu, y0, y1 = line
        add = None if a0 == "none" else np.array([[int(a0)], [int(a1)]], dtype=np.int8)
        y, acc = oracle.conv_fwd_int8(x, w, np.array([float(sc)], np.float32),
                                      np.array([float(b)], np.float32), imap, add=add,
                                      add_scale=float(asc), relu=relu == "1")
        assert acc.ravel().tolist() == [-29, -13]
        assert y.ravel().tolist() == [int(y0), int(y1)], line
        rows += 1
    assert rows == 6


def _int8_case(seed, n=300, batch=2, shape=(7, 8, 9), cin=24, cout=20):
    g = np.random.default_rng(seed)
    coords = rand_coords(g, n, batch, shape)
    imap, _ = oracle.subm_map(coords, batch, shape)
    x = g.integers(-128, 128, size=(n, cin)).astype(np.int8)
    w = g.integers(-128, 128, size=(27, cin, cout)).astype(np.int8)
    return coords, imap, x, w, g


def test_int8_sums_equal_the_fp64_forward():
    """The integer sums are the pinned float forward of the same integer values
    (every partial sum is an integer far below 2^53, so fp64 is exact)."""
    _, imap, x, w, _ = _int8_case(11)
    _, acc = oracle.conv_fwd_int8(x, w, np.ones(w.shape[2], np.float32), None, imap)
    ref = oracle.conv_fwd(x.astype(np.float64), w.astype(np.float64), None, imap)
    assert np.array_equal(acc.astype(np.float64), ref)


def test_int8_k1_is_integer_gemm():
    g = np.random.default_rng(12)
    x = g.integers(-128, 128, size=(50, 16)).astype(np.int8)
    w = g.integers(-128, 128, size=(1, 16, 8)).astype(np.int8)
    _, acc = oracle.conv_fwd_int8(x, w, np.ones(8, np.float32), None, None)
    assert np.array_equal(acc, x.astype(np.int64) @ w[0].astype(np.int64))


def test_int8_scales_reproduce_the_dequantized_float_conv():
    """scale = input_scale * weight_scale[j] / output_scale and bias / output_scale
    (the page's conversion from a quantized layer) make the code the quantized
    float conv of the dequantized tensors: equal codes except within fp32
    rounding of a rounding tie, and never more than one code apart."""
    _, imap, x, w, g = _int8_case(13, cin=16, cout=12)
    w = (w // 8).astype(np.int8)  # keep outputs mostly inside the int8 range
    s_in = np.float32(0.05)
    s_w = g.uniform(0.002, 0.02, size=w.shape[2]).astype(np.float32)
    s_out = np.float32(0.09)
    bias_fp = g.normal(0, 0.5, size=w.shape[2])
    scale = (s_in * s_w / s_out).astype(np.float32)
    bias = (bias_fp / s_out).astype(np.float32)
    y, _ = oracle.conv_fwd_int8(x, w, scale, bias, imap)
    real = oracle.conv_fwd(x.astype(np.float64) * float(s_in),
                           w.astype(np.float64) * s_w.astype(np.float64)[None, None, :],
                           bias_fp, imap) / float(s_out)
    q = np.clip(np.where(real >= 0, np.floor(real + 0.5), np.ceil(real - 0.5)), -128, 127)
    diff = np.abs(y.astype(np.int64) - q.astype(np.int64))
    assert diff.max() <= 1
    near_tie = np.abs(np.abs(real - np.trunc(real)) - 0.5) < 1e-3
    assert np.all(near_tie[diff > 0])
    assert (diff == 0).mean() > 0.99
    assert np.unique(y).size > 50  # the case spans the code range


def test_int8_residual_relu_translation():
    """ReLU output is nonnegative, saturated codes sit at the ends, and a
    translated scene gives the same codes."""
    coords, imap, x, w, g = _int8_case(14, cin=8, cout=8)
    add = g.integers(-128, 128, size=(coords.shape[0], 8)).astype(np.int8)
    sc = np.full(8, 0.003, np.float32)
    y, acc = oracle.conv_fwd_int8(x, w, sc, None, imap, add=add, add_scale=0.5, relu=True)
    assert y.min() >= 0
    shifted = coords.copy()
    shifted[:, 1:] += 1
    imap2, _ = oracle.subm_map(shifted, 2, (8, 9, 10))
    y2, acc2 = oracle.conv_fwd_int8(x, w, sc, None, imap2, add=add, add_scale=0.5, relu=True)
    assert np.array_equal(y, y2) and np.array_equal(acc, acc2)


def test_oracle_threads_do_not_change_results():
    """The oracle's parallel row loops give the same bits at any thread count."""
    coords, imap, x, w, g = _int8_case(15, n=400, cin=8, cout=6)
    xf = g.standard_normal((400, 8))
    wf = g.standard_normal((27, 8, 6))
    shape, batch = (7, 8, 9), 2
    try:
        oracle.set_threads(1)
        m1, c1 = oracle.subm_map(coords, batch, shape)
        y1 = oracle.conv_fwd(xf, wf, None, m1)
        q1, a1 = oracle.conv_fwd_int8(x, w, np.full(6, 0.01, np.float32), None, m1)
        oracle.set_threads(4)
        m4, c4 = oracle.subm_map(coords, batch, shape)
        y4 = oracle.conv_fwd(xf, wf, None, m4)
        q4, a4 = oracle.conv_fwd_int8(x, w, np.full(6, 0.01, np.float32), None, m4)
    finally:
        oracle.set_threads(1)
    assert np.array_equal(m1, m4) and np.array_equal(c1, c4)
    assert np.array_equal(y1, y4) and np.array_equal(q1, q4) and np.array_equal(a1, a4)
