"""GPU parity of the quantized (int8) forward against the oracle's int8 rule.

The output codes are integers decided in fp32 by the same expression on both
sides, so they must match bit for bit; the integer sums are exact on the GPU
for K * Cin <= 8192 (the kernel's split of the weights into 4-bit halves), which
the extreme-value case checks at its limit.  Small cases are compared in full;
the 256^3 shell at full size on sampled rows (first and last tiles, the ragged
tail, random rows), which the oracle evaluates on the sampled map columns."""

import numpy as np
import pytest
import torch

import oracle
import scenes
import sparse_convolution_hash_gb300 as spc
from gpu_util import dev, rand_coords, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def int8_case(g, n, cin, cout, K, spread=40.0):
    x = np.clip(np.rint(g.standard_normal((n, cin)) * spread), -128, 127).astype(np.int8)
    w = np.clip(np.rint(g.standard_normal((K, cin, cout)) * 30.0), -128, 127).astype(np.int8)
    # output scale so that codes spread over the int8 range
    scale = (g.uniform(0.5, 1.5, size=cout) / (spread * 30.0 * np.sqrt(K * cin) / 40.0)).astype(np.float32)
    bias = g.normal(0.0, 5.0, size=cout).astype(np.float32)
    return x, w, scale, bias


def run(x, w, scale, bias, imap, **kw):
    d = dev()
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(d)
    st = spc.new_status(d)
    y = spc.spc_conv_fwd_int8(t(x), t(w), t(scale), t(bias), imap, status=st, **kw)
    torch.cuda.synchronize()
    spc.check_status(st, "int8 forward")
    return y


@pytest.mark.parametrize("n,cin,cout", [(1, 64, 64), (700, 64, 64), (1500, 128, 128),
                                        (1029, 64, 192), (333, 192, 64), (2100, 128, 256),
                                        (129, 256, 128)])
@pytest.mark.parametrize("relu,residual", [(False, False), (True, True)])
def test_int8_subm_small_full(n, cin, cout, relu, residual):
    g = np.random.default_rng(n + cin)
    batch, shape = 2, (12, 11, 13)
    coords = rand_coords(g, n, batch, shape)
    x, w, scale, bias = int8_case(g, n, cin, cout, 27)
    add = g.integers(-128, 128, size=(n, cout)).astype(np.int8) if residual else None
    m = spc.spc_build_indice_map(torch.from_numpy(coords).to(dev()), batch, shape)
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(coords, batch, shape)
    ref, acc = oracle.conv_fwd_int8(x, w, scale, bias, imap_ref, add=add, add_scale=0.37, relu=relu)
    d = dev()
    kw = dict(add=None if add is None else torch.from_numpy(add).to(d), add_scale=0.37,
              act=spc.SPC_ACT_RELU if relu else spc.SPC_ACT_NONE)
    y = run(x, w, scale, bias, m["imap"], mask=m["mask"], **kw)
    assert np.array_equal(y.cpu().numpy(), ref)
    # grouped row order (spconv's do_sort): same codes
    mask_g, perm = spc.spc_map_row_order(m["imap"])
    y2 = run(x, w, scale, bias, m["imap"], mask=mask_g, perm=perm, **kw)
    assert torch.equal(y, y2)
    # the case exercises the code range (not all saturated or zero)
    assert len(np.unique(ref)) > 20 and np.abs(acc).max() > 0


def test_int8_exactness_at_the_limit():
    """Integer sums at the edge of the exact range, K * Cin = 27 * 256 = 6,912, on
    a fully occupied 6^3 grid (interior rows have all 27 neighbours) with every
    feature -128.  Channel 0 has every weight -1 (low half 15): its low-half
    fp32 sums reach 13.3M, near 2^24.  Channel 1 has every weight -128 (high
    half -8).  A bias of minus the interior rows' exact sum at unit scale makes
    those rows' codes 0 exactly when the sum is exact (an error of one unit in
    channel 0, or of one high-half unit in channel 1, moves the code)."""
    z, y_, x_ = np.meshgrid(np.arange(6), np.arange(6), np.arange(6), indexing="ij")
    coords = np.stack([np.zeros(216), z.ravel(), y_.ravel(), x_.ravel()], 1).astype(np.int32)
    cin, cout = 256, 64
    g = np.random.default_rng(3)
    w = g.choice(np.array([-128, -1, 127], np.int8), size=(27, cin, cout))
    w[:, :, 0] = -1
    w[:, :, 1] = -128
    m = spc.spc_build_indice_map(torch.from_numpy(coords).to(dev()), 1, (6, 6, 6))
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(coords, 1, (6, 6, 6))
    interior = (imap_ref >= 0).all(axis=0)
    assert interior.sum() == 64
    scale = np.ones(cout, np.float32)
    bias = np.zeros(cout, np.float32)
    bias[0], bias[1] = -(128.0 * 6912), -(128.0 * 128 * 6912)
    for xv in ("all -128", "random signs"):
        x = (np.full((216, cin), -128, np.int8) if xv == "all -128"
             else g.choice(np.array([-128, 127], np.int8), size=(216, cin)))
        ref, acc = oracle.conv_fwd_int8(x, w, scale, bias, imap_ref)
        y = run(x, w, scale, bias, m["imap"])
        assert np.array_equal(y.cpu().numpy(), ref), xv
        if xv == "all -128":
            assert (ref[interior, :2] == 0).all() and acc[interior, 0].max() == 128 * 6912
    # at a scale that keeps codes in range for all channels
    ref, _ = oracle.conv_fwd_int8(x, w, np.full(cout, 2.0 ** -20, np.float32), None, imap_ref)
    y = run(x, w, np.full(cout, 2.0 ** -20, np.float32), None, m["imap"])
    assert np.array_equal(y.cpu().numpy(), ref)


def test_int8_k1_and_strided():
    g = np.random.default_rng(9)
    d = dev()
    # k = 1 without a map: a per-voxel integer GEMM
    x, w, scale, bias = int8_case(g, 1000, 128, 64, 1)
    ref, _ = oracle.conv_fwd_int8(x, w, scale, bias, None)
    y = run(x, w, scale, bias, None, n_out=1000)
    assert np.array_equal(y.cpu().numpy(), ref)
    # strided k3 s2 p1 on the 2,000-voxel set
    coords = scenes.coords_for("uniform32")
    c = torch.from_numpy(coords).to(d)
    oc, _ = spc.spc_strided_out_coords(c, 1, (32, 32, 32), 3, 2, 1, 1)
    m = spc.spc_build_indice_map(c, 1, (32, 32, 32), ksize=3, stride=2, pad=1, subm=False,
                                 out_coords=oc)
    spc.check_status(m["status"])
    imap_ref, _, _ = oracle.strided_map(coords, oc.cpu().numpy(), 1, (32, 32, 32), 3, 2, 1, 1, False)
    x, w, scale, bias = int8_case(g, coords.shape[0], 64, 128, 27)
    ref, _ = oracle.conv_fwd_int8(x, w, scale, bias, imap_ref, relu=True)
    y = run(x, w, scale, bias, m["imap"], act=spc.SPC_ACT_RELU)
    assert np.array_equal(y.cpu().numpy(), ref)


def test_int8_empty_and_unsupported():
    d = dev()
    x = torch.zeros((0, 64), dtype=torch.int8, device=d)
    w = torch.zeros((27, 64, 64), dtype=torch.int8, device=d)
    sc = torch.ones(64, device=d)
    imap = torch.zeros((27, 0), dtype=torch.int32, device=d)
    assert spc.spc_conv_fwd_int8(x, w, sc, None, imap).shape == (0, 64)
    with pytest.raises(spc.SpcError):  # K * cin beyond the exact range
        spc.spc_conv_fwd_int8(torch.zeros((4, 320), dtype=torch.int8, device=d),
                              torch.zeros((27, 320, 64), dtype=torch.int8, device=d), sc, None,
                              torch.zeros((27, 4), dtype=torch.int32, device=d))


def test_int8_shell256_sampled():
    """256^3 shell (398,833 voxels), 128 -> 128, full size in the launch shape
    the benchmark times; sampled rows against the oracle, run-to-run identical."""
    w = scenes.workload("shell256_int8")
    c = w["coords"]
    d = dev()
    m = spc.spc_build_indice_map(torch.from_numpy(c).to(d), 1, (256, 256, 256))
    spc.check_status(m["status"])
    imap_ref, _ = oracle.subm_map(c, 1, (256, 256, 256))
    args = (w["x"].to(d), w["w"].to(d), w["scale"].to(d), w["bias"].to(d), m["imap"])
    y = spc.spc_conv_fwd_int8(*args, mask=m["mask"], act=spc.SPC_ACT_RELU)
    rows = sample_rows(c.shape[0], seed=4)
    ref, _ = oracle.conv_fwd_int8(w["x"], w["w"], w["scale"], w["bias"], imap_ref[:, rows],
                                  relu=True)
    assert np.array_equal(y[torch.from_numpy(rows).to(d)].cpu().numpy(), ref)
    y2 = spc.spc_conv_fwd_int8(*args, mask=m["mask"], act=spc.SPC_ACT_RELU)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("cout", [64, 128])
def test_int8_weight_split_path(cout):
    """K * Cin = 8192 (k = 1, 8192 input channels): beyond the accumulator-split
    range, so the kernel splits the weights into 4-bit halves; extreme codes."""
    g = np.random.default_rng(cout)
    n, cin = 300, 8192
    x = g.choice(np.array([-128, 127, -1, 5], np.int8), size=(n, cin))
    w = g.choice(np.array([-128, 127, -1, 15], np.int8), size=(1, cin, cout))
    _, acc = oracle.conv_fwd_int8(x, w, np.ones(cout, np.float32), None, None)
    assert np.abs(acc).max() > 2 ** 21
    scale = np.full(cout, 60.0 / acc.std(), np.float32)  # codes spread over the range
    ref, _ = oracle.conv_fwd_int8(x, w, scale, None, None)
    assert len(np.unique(ref)) > 100
    y = run(x, w, scale, None, None, n_out=n)
    assert np.array_equal(y.cpu().numpy(), ref)
