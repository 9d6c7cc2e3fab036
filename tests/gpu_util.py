"""Helpers shared by the GPU parity tests (no method arithmetic here)."""

import numpy as np
import torch

# Normwise relative tolerances against the fp64 oracle, by feature dtype and precision.
TOL = {("f32", "exact"): 1e-5, ("f32", "tf32"): 2e-3, ("f16", "exact"): 2e-2,
       ("bf16", "exact"): 2e-2, ("f16", "tf32"): 2e-2, ("bf16", "tf32"): 2e-2}

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def dev():
    return torch.device("cuda:0")


def normwise(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy() if t.is_floating_point() else t.cpu().numpy()


def sample_rows(n: int, seed: int = 0, n_rand: int = 1000, edge: int = 300) -> np.ndarray:
    """First and last `edge` rows (ragged tail included) plus random rows, sorted, unique."""
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    g = np.random.default_rng(seed)
    parts = [np.arange(min(edge, n)), np.arange(max(0, n - edge), n),
             g.integers(0, n, size=min(n_rand, n))]
    return np.unique(np.concatenate(parts)).astype(np.int64)


def rand_coords(g, n, batch, shape):
    cells = g.choice(batch * int(np.prod(shape)), size=n, replace=False)
    b, z, y, x = np.unravel_index(cells, (batch,) + tuple(shape))
    return np.stack([b, z, y, x], axis=1).astype(np.int32)


def rand_tensor(g, shape, dtype: str, std: float = 1.0) -> torch.Tensor:
    return torch.from_numpy(g.standard_normal(shape) * std).to(DT[dtype])
