"""Shared helpers for the GPU parity tests (not collected by pytest)."""
import json
import os

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


def record(name: str, values: dict) -> None:
    """Write measured values (errors, ratios) of a test to
    $ATTN_RECORD_DIR/<name>.json when that variable is set; a no-op
    otherwise.  The records are measurements, never expected values."""
    out = os.environ.get("ATTN_RECORD_DIR")
    if not out:
        return
    os.makedirs(out, exist_ok=True)
    with open(os.path.join(out, f"{name}.json"), "w") as f:
        json.dump(values, f, indent=1, sort_keys=True)
