"""Shared helpers for the GPU parity tests (not collected by pytest)."""
import numpy as np
import torch


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def sample_rows(N: int, n: int, seed: int) -> np.ndarray:
    """First/last rows, tile edges and ``n`` seeded random rows of [0, N)."""
    g = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, 129, N // 2, N - 2, N - 1]
    rnd = g.integers(0, N, size=n).tolist()
    return np.unique(np.clip(np.array(fixed + rnd), 0, N - 1))


def sample_heads(B: int, H: int, n: int, seed: int):
    g = np.random.default_rng(seed)
    heads = {(0, 0), (B - 1, H - 1)}
    while len(heads) < min(n, B * H):
        heads.add((int(g.integers(0, B)), int(g.integers(0, H))))
    return sorted(heads)
