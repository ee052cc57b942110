"""The search through the Gram factor of X (awq_search_gram), CUDA path
against the CPU oracle's losses (the same quantity, ||X S^-1 W'hat - X W||^2,
evaluated there directly): losses within 1e-2, alpha* by the same rule, s*
bit-exact, and the searched pack after it bit-exact."""
import numpy as np
import pytest
import torch

from gpu_common import LOSS_RTOL, check_alpha_star, check_column_losses, custom_cpu, rel_err, require_gpu, workload_cpu
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import AwqError, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


CASES = [
    synth.custom("gram_asym", 71, 512, 256, 264, symmetric=False, group_size=128),
    synth.custom("gram_sym_g64", 72, 1024, 384, 784, symmetric=True, group_size=64, w_sigma=0.015),
    synth.custom("gram_g256_square", 73, 512, 512, 520, symmetric=False, group_size=256),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_gram_search_matches_oracle(awq, w):
    _, X, W, Xf, Wf = custom_cpu(w)
    Xd, Wd = X.cuda(), W.cuda()
    a_gpu = awq.act_stats(Xd)
    a = a_gpu.cpu().numpy()
    grid = orc.alpha_grid(21)
    res = awq.search(Xd, Wd, a_gpu, list(grid), group_size=w.group_size, symmetric=w.symmetric, col_losses=True,
                     gram=True)
    ref = orc.search(Xf, Wf, a, grid, group_size=w.group_size, symmetric=w.symmetric)
    L = res.losses.cpu().numpy()
    assert rel_err(L, ref["losses"]).max() <= LOSS_RTOL, (L, ref["losses"])
    check_alpha_star(res.best, ref["losses"])
    s_star = res.s_star.cpu().numpy()
    assert np.array_equal(s_star, orc.scales(a, grid[res.best]))
    check_column_losses(res.col_losses.cpu().numpy(), ref["col_losses"], label=f"gram {w.name}")
    # the searched pack reads the group parameters from the same workspace
    qw, sc, z = awq.quantize_pack_searched(Wd, res, w.group_size, w.symmetric)
    oq, osc, oz = orc.pack(Wf, s_star, w.group_size, w.symmetric)
    assert np.array_equal(qw.cpu().numpy(), oq)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
    # and it agrees with the direct search
    direct = awq.search(Xd, Wd, a_gpu, list(grid), group_size=w.group_size, symmetric=w.symmetric)
    assert rel_err(L, direct.losses.cpu().numpy()).max() <= LOSS_RTOL


def test_gram_search_full_size_sampled(awq):
    """The MLP gate+up layer (N = 4 D_in, where the Gram form saves 4x the
    flops): per-column losses of a seeded column sample against the oracle."""
    w, X, W, Xf, Wf = workload_cpu("mlp_gate_up")
    a_gpu = awq.act_stats(X.cuda())
    a = a_gpu.cpu().numpy()
    grid = orc.alpha_grid(21)
    res = awq.search(X.cuda(), W.cuda(), a_gpu, list(grid), group_size=w.group_size, symmetric=w.symmetric,
                     col_losses=True, gram=True)
    col = res.col_losses.cpu().numpy()
    L = res.losses.cpu().numpy()
    torch.cuda.empty_cache()
    cols = synth.sample_columns(w.D_out, 512, w.seed)
    ref = orc.search(Xf, Wf, a, grid, group_size=w.group_size, symmetric=w.symmetric, cols=cols)
    check_column_losses(col[:, cols], ref["col_losses"], label="gram sampled")
    np.testing.assert_allclose(col.sum(axis=1), L, rtol=1e-9)


def test_gram_rank_deficient_is_range_error(awq):
    """A channel that is zero in every row makes H singular: the factor is
    not positive definite and the call reports AWQ_ERR_RANGE."""
    w = synth.custom("gram_singular", 74, 256, 256, 136)
    _, X, W, Xf, Wf = custom_cpu(w)
    X = X.clone()
    X[:, 17] = 0
    a = awq.act_stats(X.cuda())
    with pytest.raises(AwqError) as e:
        awq.search(X.cuda(), W.cuda(), a, gram=True)
    assert e.value.name == "AWQ_ERR_RANGE"
