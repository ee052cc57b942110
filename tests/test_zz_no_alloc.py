"""awq_act_stats_noalloc: the activation statistic for callers that cannot
allocate device memory (its scratch is static device memory inside the
library).  It runs the same row-slice plan and kernel as awq_act_stats and
sums in the same order, so its output must equal awq_act_stats' bit for bit,
on consecutive calls that share the array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import post_weight_quantization_column_b300 as awq
from post_weight_quantization_column_b300 import synth



def _fn():
    L = awq.lib()
    f = L.awq_act_stats_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Host-side checks, no GPU needed: too many channels for the static array."""
    f = _fn()
    fake = ctypes.c_void_p(0x1000)
    assert f(fake, 16, (1 << 20) + 8, (1 << 20) + 8, fake, None) == 2   # AWQ_ERR_SHAPE
    assert f(fake, 0, 256, 256, fake, None) == 2
    assert f(None, 16, 256, 256, fake, None) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(4096, 4096), (300, 776), (16384, 8192)])
def test_noalloc_matches_act_stats_twice(shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    N, D = shape
    f = _fn()
    rng = np.random.default_rng(N + D)
    Xf = rng.standard_normal((N, D), dtype=np.float32)
    Xf[:, rng.choice(D, size=max(1, D // 100), replace=False)] *= 30.0
    X = synth.to_bf16(Xf).cuda()
    ref = awq.act_stats(X)                              # the workspace entry point
    for _ in range(2):                                  # two calls in a row share the array
        out = torch.full((D,), float("nan"), dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream()
        rc = f(ctypes.c_void_p(X.data_ptr()), N, D, D, ctypes.c_void_p(out.data_ptr()),
               ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), ((out - ref).abs() / ref.abs()).max().item()


@pytest.mark.gpu
def test_noalloc_wide_layer():
    """A very wide layer (65536 channels) through the static scratch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = _fn()
    N, D = 2048, 65536
    rng = np.random.default_rng(3)
    X = synth.to_bf16(rng.standard_normal((N, D), dtype=np.float32)).cuda()
    ref = awq.act_stats(X)
    for _ in range(2):
        out = torch.empty(D, dtype=torch.float32, device="cuda")
        rc = f(ctypes.c_void_p(X.data_ptr()), N, D, D, ctypes.c_void_p(out.data_ptr()),
               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
