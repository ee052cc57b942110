"""Shared helpers of the GPU parity tests (inputs from the seeded generator,
expected values from the CPU oracle only)."""
from __future__ import annotations

import functools
import os

import numpy as np
import pytest
import torch

from post_weight_quantization_column_b300 import synth

PARITY_COLS = int(os.environ.get("AWQ_PARITY_COLS", "512"))
LOSS_RTOL = 1e-2          # per-alpha losses (spec tolerance)
STATS_RTOL = 1e-5         # mean |X| (fp32 in-slice sums, fp64 across slices)


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_column_b300 as awq
    if not os.path.exists(awq.LIB_PATH):
        from post_weight_quantization_column_b300 import build
        build.build()
    return awq


@functools.lru_cache(maxsize=1)
def workload_cpu(name: str):
    """(workload, X bf16 CPU, W bf16 CPU, X fp32 numpy, W fp32 numpy) for a named workload."""
    w = synth.WORKLOADS[name]
    X, W = synth.generate(w)
    return w, X, W, synth.bf16_to_f32(X), synth.bf16_to_f32(W)


def custom_cpu(w):
    X, W = synth.generate(w)
    return w, X, W, synth.bf16_to_f32(X), synth.bf16_to_f32(W)


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-300)


def check_alpha_star(gpu_best: int, oracle_losses: np.ndarray, rtol=LOSS_RTOL):
    """alpha* equal to the oracle's, or with an oracle loss within rtol of its minimum."""
    ob = int(np.argmin(oracle_losses))
    if gpu_best == ob:
        return
    assert oracle_losses[gpu_best] <= oracle_losses[ob] * (1 + rtol), (gpu_best, ob, oracle_losses)


def record(kind: str, **fields):
    """Append one JSON line to the file named by AWQ_TEST_RECORD, if set (a
    record of measured agreement, e.g. the share of columns within rtol)."""
    path = os.environ.get("AWQ_TEST_RECORD")
    if not path:
        return
    import json
    with open(path, "a") as f:
        f.write(json.dumps({"kind": kind, **fields}) + "\n")


def check_column_losses(got, want, rtol=LOSS_RTOL, min_frac=0.98, label=""):
    """Per-column losses: the search may round a code the other way where w'/step
    sits within ~1e-6 of a half step (reciprocal multiply instead of IEEE
    division), which moves that column's loss by a few percent.  Require most
    columns within rtol and every column within 25%."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    big = want > 1e-3 * want.max()
    e = rel_err(got[big], want[big])
    frac = float(np.mean(e <= rtol))
    record("column_losses", label=label, columns=int(e.size), outside=int(np.count_nonzero(e > rtol)),
           frac_within=frac, max_rel=float(e.max()))
    assert frac >= min_frac, (frac, float(e.max()))
    assert e.max() <= 0.25, float(e.max())
    return frac, float(e.max())
