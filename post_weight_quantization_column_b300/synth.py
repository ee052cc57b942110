"""Seeded synthetic workloads shaped like LLM linear layers.

This module only draws random numbers and rounds them to bf16.  It holds none
of the calibration arithmetic, so both the CUDA path and the CPU oracle can be
fed from it without sharing any of the method.

Recipe (every workload): ``numpy.random.default_rng(seed)`` (PCG64), draws in
float32, then a round-to-nearest-even cast to bfloat16 through torch.

* X ~ N(0, 1), or |a|*b with a, b iid N(0, 1) for the SiLU-gated
  down-projection input;
* k = round(0.01 * D_in) outlier channels chosen without replacement; they are
  multiplied by a fixed factor (tiny layer: 50) or by 10**U(1, 2) (log-uniform
  in [10, 100]);
* W ~ N(0, sigma), laid out [D_in, D_out] row-major (input channel = row).

The outlier structure mirrors the pages' observation that roughly 1% of the
input channels carry activations far larger than the rest.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    N: int          # calibration rows
    D_in: int       # input channels (rows of W)
    D_out: int      # output channels (columns of W)
    w_sigma: float
    x_kind: str     # "normal" or "gated"
    n_outliers: int
    outlier_factor: float | None   # fixed factor, or None for log-uniform [10, 100]
    symmetric: bool
    group_size: int = 128
    bits: int = 4


WORKLOADS = {
    "tiny": Workload("tiny", 0, 64, 256, 256, 0.02, "normal", 3, 50.0, False),
    "attn_proj": Workload("attn_proj", 1, 4096, 4096, 4096, 0.02, "normal", 41, None, False),
    "mlp_gate_up": Workload("mlp_gate_up", 2, 16384, 4096, 22016, 0.02, "normal", 41, None, False),
    "mlp_down": Workload("mlp_down", 3, 16384, 11008, 4096, 0.015, "gated", 110, None, False),
    "large_mlp": Workload("large_mlp", 4, 16384, 8192, 28672, 0.01, "normal", 82, None, True),
}
ORDER = ["tiny", "attn_proj", "mlp_gate_up", "mlp_down", "large_mlp"]


def custom(name, seed, N, D_in, D_out, *, w_sigma=0.02, x_kind="normal",
           n_outliers=None, outlier_factor=None, symmetric=False, group_size=128):
    """A workload of arbitrary shape with the same recipe (ragged test cases)."""
    if n_outliers is None:
        n_outliers = int(round(0.01 * D_in))
    return Workload(name, seed, N, D_in, D_out, w_sigma, x_kind, n_outliers,
                    outlier_factor, symmetric, group_size)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bfloat16 torch tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    """bfloat16 torch tensor -> float32 numpy (exact widening)."""
    return t.detach().to("cpu").to(torch.float32).numpy()


def generate(w: Workload):
    """Return (X, W) as CPU bfloat16 tensors, X [N, D_in], W [D_in, D_out]."""
    rng = np.random.default_rng(w.seed)
    if w.x_kind == "gated":
        a = rng.standard_normal((w.N, w.D_in), dtype=np.float32)
        b = rng.standard_normal((w.N, w.D_in), dtype=np.float32)
        X = np.abs(a) * b
        del a, b
    else:
        X = rng.standard_normal((w.N, w.D_in), dtype=np.float32)
    k = min(w.n_outliers, w.D_in)
    if k > 0:
        idx = rng.choice(w.D_in, size=k, replace=False)
        if w.outlier_factor is not None:
            fac = np.full(k, w.outlier_factor, dtype=np.float32)
        else:
            fac = (10.0 ** rng.uniform(1.0, 2.0, size=k)).astype(np.float32)
        X[:, idx] *= fac[None, :]
    Wm = rng.standard_normal((w.D_in, w.D_out), dtype=np.float32)
    Wm *= np.float32(w.w_sigma)
    return to_bf16(X), to_bf16(Wm)


def sample_columns(D_out: int, n: int, seed: int) -> np.ndarray:
    """Sorted seeded sample of output columns for sampled parity checks."""
    rng = np.random.default_rng(10_000 + seed)
    n = min(n, D_out)
    return np.sort(rng.choice(D_out, size=n, replace=False)).astype(np.int64)
