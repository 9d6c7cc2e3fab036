"""Seeded synthetic voxel scenes and feature tensors.

This module only draws inputs: coordinate sets with the shapes, sizes and
sparsity structure of the five sparse-convolution workloads, and the feature,
weight, bias and upstream-gradient tensors that go with them.  It holds none of
the convolution arithmetic, so both the CPU oracle and the CUDA path can take
their inputs from it.

Coordinates are int32 rows (b, z, y, x), batch index in column 0, as in the
spconv "SparseConvTensor" description (indices [N, ndim+1], batch first).
Every random draw uses numpy's PCG64 with a fixed seed; floating-point tensors
are drawn in float64 and then rounded once to the workload dtype, so that the
values handed to both sides are exactly representable in that dtype.

Workloads (sizes as the five configurations state them):

  uniform32   2,000 distinct cells drawn without replacement from a 32^3 grid,
              batch 1, rows in draw order (seed 1).
  lidar       batch 2 in a 41 x 1600 x 1408 (z, y, x) grid, 60,000 voxels per
              sample: a ground layer (each xy cell with probability 0.02, z
              uniform in {0, 1}) plus the surfaces of 40 axis-aligned boxes with
              integer sides in [8, 60]; box-surface cells not on the ground are
              subsampled uniformly to top each sample up to exactly 60,000.
              Rows sorted by (b, z, y, x) (seed 2).
  shell256    cells within one cell of the surface of a seeded union of six
              randomly rotated ellipsoids in a 256^3 grid (about 400k voxels),
              batch 1, rows sorted (seed 4).
  shell192x4  four such shells in 192^3 grids (seeds 5..8, about 125k voxels
              each), batch index 0..3 in column 0, rows sorted.

A cell is "within one cell of the surface" when its 3x3x3 neighbourhood holds
both a cell centre inside the union and one outside it.
"""

from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "rng",
    "uniform_cells",
    "lidar_scene",
    "ellipsoid_shell",
    "shell_batch",
    "normal",
    "WORKLOADS",
    "workload",
]


def rng(seed: int, tag: int = 0) -> np.random.Generator:
    """A PCG64 generator for (seed, tag); tags separate the streams of one workload."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tag)])))


def _decode_cells(flat: np.ndarray, shape) -> np.ndarray:
    z, y, x = np.unravel_index(flat, shape)
    return np.stack([z, y, x], axis=1)


def uniform_cells(n: int, shape=(32, 32, 32), seed: int = 1) -> np.ndarray:
    """n distinct cells of one sample, uniform without replacement, in draw order."""
    g = rng(seed, 0)
    total = int(np.prod(shape))
    flat = g.choice(total, size=n, replace=False)
    zyx = _decode_cells(flat, shape)
    out = np.zeros((n, 4), dtype=np.int32)
    out[:, 1:] = zyx
    return out


def _box_surface(g: np.random.Generator, shape) -> np.ndarray:
    """Flat indices of the surface cells of one random axis-aligned box."""
    D, H, W = shape
    sz, sy, sx = (int(v) for v in g.integers(8, 61, size=3))
    z0 = int(g.integers(0, D))
    y0 = int(g.integers(0, H - sy + 1))
    x0 = int(g.integers(0, W - sx + 1))
    z1 = min(D, z0 + sz)
    zz, yy, xx = np.meshgrid(
        np.arange(z0, z1), np.arange(y0, y0 + sy), np.arange(x0, x0 + sx), indexing="ij"
    )
    on_face = (
        (zz == z0) | (zz == z0 + sz - 1) | (yy == y0) | (yy == y0 + sy - 1)
        | (xx == x0) | (xx == x0 + sx - 1)
    )
    return np.ravel_multi_index((zz[on_face], yy[on_face], xx[on_face]), shape)


def lidar_scene(batch: int = 2, shape=(41, 1600, 1408), per_sample: int = 60000,
                ground_density: float = 0.02, n_boxes: int = 40, seed: int = 2) -> np.ndarray:
    """LiDAR-like scene: ground layer + sparsely sampled box surfaces, rows sorted."""
    D, H, W = shape
    rows = []
    for b in range(batch):
        g = rng(seed, 100 + b)
        chosen = g.random((H, W)) < ground_density
        gy, gx = np.nonzero(chosen)
        gz = g.integers(0, 2, size=gy.shape[0])
        ground = np.ravel_multi_index((gz, gy, gx), shape)
        boxes = np.unique(np.concatenate([_box_surface(g, shape) for _ in range(n_boxes)]))
        extra = np.setdiff1d(boxes, ground, assume_unique=False)
        need = per_sample - ground.shape[0]
        if need < 0:
            ground = g.choice(ground, size=per_sample, replace=False)
            need = 0
        need = min(need, extra.shape[0])
        top = g.choice(extra, size=need, replace=False)
        flat = np.sort(np.concatenate([ground, top]))
        zyx = _decode_cells(flat, shape)
        blk = np.empty((flat.shape[0], 4), dtype=np.int32)
        blk[:, 0] = b
        blk[:, 1:] = zyx
        rows.append(blk)
    return np.concatenate(rows, axis=0)


def _random_rotation(g: np.random.Generator) -> np.ndarray:
    q, r = np.linalg.qr(g.standard_normal((3, 3)))
    q = q * np.sign(np.diag(r))
    if np.linalg.det(q) < 0:
        q[:, 0] = -q[:, 0]
    return q


def _neigh_any(mask: np.ndarray) -> np.ndarray:
    """True where some cell of the 3x3x3 neighbourhood is True (outside the grid = False)."""
    out = mask
    for axis in range(3):
        p = np.pad(out, [(1, 1) if a == axis else (0, 0) for a in range(3)])
        sl = lambda s: tuple(slice(s, s + out.shape[axis]) if a == axis else slice(None) for a in range(3))
        out = p[sl(0)] | p[sl(1)] | p[sl(2)]
    return out


def ellipsoid_shell(dim: int, n_ellipsoids: int, scale: float, seed: int) -> np.ndarray:
    """(z, y, x) cells within one cell of a union of rotated ellipsoids, sorted."""
    g = rng(seed, 200)
    ax = np.arange(dim, dtype=np.float64)
    inside = np.zeros((dim, dim, dim), dtype=bool)
    zz, yy, xx = np.meshgrid(ax, ax, ax, indexing="ij", sparse=True)
    for _ in range(n_ellipsoids):
        c = g.uniform(0.22, 0.78, size=3) * dim
        semi = scale * dim * g.uniform(0.6, 1.4, size=3)
        R = _random_rotation(g)
        dz, dy, dx = zz - c[0], yy - c[1], xx - c[2]
        acc = np.zeros((dim, dim, dim), dtype=np.float64)
        for j in range(3):
            u = R[j, 0] * dz + R[j, 1] * dy + R[j, 2] * dx
            acc += (u / semi[j]) ** 2
        inside |= acc <= 1.0
    shell = _neigh_any(inside) & _neigh_any(~inside)
    z, y, x = np.nonzero(shell)
    return np.stack([z, y, x], axis=1).astype(np.int32)


# Scale factors fixed once so that the shells land on their target sizes
# (about 400k voxels at 256^3, about 125k per sample at 192^3).
SHELL256_SCALE = 0.18
SHELL192_SCALE = 0.1255


def shell_batch(dim: int, seeds, scale: float, n_ellipsoids: int = 6) -> np.ndarray:
    """Concatenate one shell per seed, batch index = position in `seeds`."""
    rows = []
    for b, s in enumerate(seeds):
        zyx = ellipsoid_shell(dim, n_ellipsoids, scale, s)
        blk = np.empty((zyx.shape[0], 4), dtype=np.int32)
        blk[:, 0] = b
        blk[:, 1:] = zyx
        rows.append(blk)
    return np.concatenate(rows, axis=0)


_TORCH_DTYPES = {
    "f32": torch.float32,
    "f16": torch.float16,
    "bf16": torch.bfloat16,
}


def normal(shape, std: float, dtype: str, seed: int, tag: int) -> torch.Tensor:
    """N(0, std^2) draws in float64, rounded once to `dtype`; returned on the CPU."""
    a = rng(seed, tag).standard_normal(shape) * std
    return torch.from_numpy(a).to(_TORCH_DTYPES[dtype])


# Workload table: name -> coordinate recipe and tensor recipe.
# "var" entries are variances, as in the workload statements N(0, var).
WORKLOADS = {
    "uniform32_subm_f32": dict(coords=("uniform32",), batch=1, shape=(32, 32, 32), k=3, stride=1,
                               pad=1, subm=True, dtype="f32", cin=16, cout=16, bias_var=0.01,
                               seed=1),
    "lidar_subm_f16": dict(coords=("lidar",), batch=2, shape=(41, 1600, 1408), k=3, stride=1,
                           pad=1, subm=True, dtype="f16", cin=16, cout=16, bias_var=None, seed=2),
    "uniform32_strided_bf16": dict(coords=("uniform32",), batch=1, shape=(32, 32, 32), k=3,
                                   stride=2, pad=1, subm=False, dtype="bf16", cin=64, cout=128,
                                   bias_var=None, seed=3),
    "shell256_subm_bf16": dict(coords=("shell256",), batch=1, shape=(256, 256, 256), k=3,
                               stride=1, pad=1, subm=True, dtype="bf16", cin=128, cout=128,
                               bias_var=None, seed=4),
    "shell256_k1_bf16": dict(coords=("shell256",), batch=1, shape=(256, 256, 256), k=1,
                             stride=1, pad=0, subm=True, dtype="bf16", cin=128, cout=128,
                             bias_var=None, seed=4),
    "shell192x4_train_bf16": dict(coords=("shell192x4",), batch=4, shape=(192, 192, 192), k=3,
                                  stride=1, pad=1, subm=True, dtype="bf16", cin=64, cout=64,
                                  bias_var=None, seed=5, train=True),
    # residual block tail on the 4 x 192^3 shells: relu(conv(x) + x) in one pass
    "shell192x4_resblock_bf16": dict(coords=("shell192x4",), batch=4, shape=(192, 192, 192), k=3,
                                     stride=1, pad=1, subm=True, dtype="bf16", cin=64, cout=64,
                                     bias_var=None, seed=10, resblock=True),
    # max pool k2 s2 (forward + gradient) on the 256^3 shell, 128 channels
    "shell256_maxpool_bf16": dict(coords=("shell256",), batch=1, shape=(256, 256, 256), k=2,
                                  stride=2, pad=0, subm=False, dtype="bf16", cin=128, cout=128,
                                  bias_var=None, seed=11, maxpool=True),
    # inverse of a k3 s2 p1 conv on the 256^3 shell: features on the strided output set
    # (cin channels) go back to the shell's voxels (cout channels)
    "shell256_inverse_bf16": dict(coords=("shell256",), batch=1, shape=(256, 256, 256), k=3,
                                  stride=2, pad=1, subm=False, dtype="bf16", cin=128, cout=128,
                                  bias_var=None, seed=9, inverse=True),
    # quantized inference layer on the 256^3 shell: int8 codes in and out, fp32
    # per-channel scale and bias, ReLU
    "shell256_int8": dict(coords=("shell256",), batch=1, shape=(256, 256, 256), k=3, stride=1,
                          pad=1, subm=True, dtype="i8", cin=128, cout=128, bias_var=None, seed=12,
                          int8=True),
}


def int8_codes(shape, std: float, seed: int, tag: int) -> torch.Tensor:
    """Integer codes rint(N(0, std^2)) clipped to [-128, 127], as int8 (CPU)."""
    a = np.clip(np.rint(rng(seed, tag).standard_normal(shape) * std), -128, 127)
    return torch.from_numpy(a.astype(np.int8))

_COORD_CACHE: dict = {}


def coords_for(kind: str) -> np.ndarray:
    """The coordinate set of one scene kind (cached per process)."""
    if kind not in _COORD_CACHE:
        if kind == "uniform32":
            c = uniform_cells(2000, (32, 32, 32), seed=1)
        elif kind == "lidar":
            c = lidar_scene(2, (41, 1600, 1408), 60000, 0.02, 40, seed=2)
        elif kind == "shell256":
            c = shell_batch(256, [4], SHELL256_SCALE)
        elif kind == "shell192x4":
            c = shell_batch(192, [5, 6, 7, 8], SHELL192_SCALE)
        else:
            raise KeyError(kind)
        _COORD_CACHE[kind] = c
    return _COORD_CACHE[kind]


def workload(name: str) -> dict:
    """Coordinates and CPU tensors of a named workload.

    Returns a dict with coords [N,4] int32 (numpy), x [N,cin], w [K,cin,cout],
    bias [cout] or None, dy [N_out?] is left to the caller for strided outputs
    (its row count depends on the output set); for subm workloads dy [N,cout]
    is included.
    """
    spec = WORKLOADS[name]
    coords = coords_for(spec["coords"][0])
    n = coords.shape[0]
    K = spec["k"] ** 3
    cin, cout, dt, seed = spec["cin"], spec["cout"], spec["dtype"], spec["seed"]
    out = dict(spec)
    out["name"] = name
    out["coords"] = coords
    if spec.get("int8"):
        # codes of std 32 (features) and 24 (weights); per-channel output scales
        # put the integer sums' typical size (about 32 * 24 * sqrt(20 Cin) on the
        # shells' ~20 pairs per voxel) at about 40 codes; bias of a few codes
        out["x"] = int8_codes((n, cin), 32.0, seed, 1)
        out["w"] = int8_codes((K, cin, cout), 24.0, seed, 2)
        g = rng(seed, 3)
        typical = 32.0 * 24.0 * np.sqrt(20.0 * cin)
        out["scale"] = torch.from_numpy((g.uniform(0.5, 1.5, size=cout) * 40.0 / typical)
                                        .astype(np.float32))
        out["bias"] = torch.from_numpy(g.normal(0.0, 4.0, size=cout).astype(np.float32))
        return out
    out["x"] = normal((n, cin), 1.0, dt, seed, 1)
    out["w"] = normal((K, cin, cout), float(np.sqrt(1.0 / (27 * cin))), dt, seed, 2)
    out["bias"] = (normal((cout,), float(np.sqrt(spec["bias_var"])), dt, seed, 3)
                   if spec["bias_var"] is not None else None)
    if spec["subm"]:
        out["dy"] = normal((n, cout), 1.0, dt, seed, 4)
    if spec.get("inverse"):
        # features on the strided output set, whose size the caller finds first
        out["y_for"] = lambda n_y: normal((n_y, cin), 1.0, dt, seed, 5)
    return out
