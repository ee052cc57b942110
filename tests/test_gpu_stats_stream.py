"""The statistic over a stream of calibration batches, and the max |x|
variant, CUDA path against the CPU oracle."""
import numpy as np
import pytest
import torch

from gpu_common import LOSS_RTOL, STATS_RTOL, check_alpha_star, custom_cpu, rel_err, require_gpu, workload_cpu
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import AwqError, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


@pytest.mark.parametrize("name,cuts", [("attn_proj", [1000, 37, 3059]), ("mlp_down", [8192, 8192]),
                                       ("tiny", [1, 63])])
def test_stream_mean_and_max(awq, name, cuts):
    w, X, W, Xf, Wf = workload_cpu(name)
    acc = awq.StatsAccumulator(w.D_in, "cuda", track_max=True)
    Xd = X.cuda()
    edges = np.cumsum([0] + cuts)
    assert edges[-1] == w.N
    for a, b in zip(edges[:-1], edges[1:]):
        acc.add_batch(Xd[a:b].contiguous())
    mean = acc.mean().cpu().numpy()
    want = orc.act_stats_stream([Xf[a:b] for a, b in zip(edges[:-1], edges[1:])])
    assert rel_err(mean, want).max() <= STATS_RTOL
    # and the one-shot statistic of the whole X
    assert rel_err(mean, awq.act_stats(Xd).cpu().numpy()).max() <= STATS_RTOL
    # the maximum is exact
    assert np.array_equal(acc.max_abs.cpu().numpy(), orc.act_stats_max(Xf))


def test_max_statistic_ragged_channels(awq):
    w = synth.custom("maxstat", 41, 300, 384, 264)
    _, X, W, Xf, Wf = custom_cpu(w)
    got = awq.act_stats_max(X.cuda()).cpu().numpy()
    assert np.array_equal(got, orc.act_stats_max(Xf))


def test_search_on_the_max_statistic(awq):
    """s_j = max(max|X_j|, floor)^alpha: the search takes any statistic vector."""
    w = synth.custom("maxsearch", 42, 256, 512, 520, symmetric=False)
    _, X, W, Xf, Wf = custom_cpu(w)
    m_gpu = awq.act_stats_max(X.cuda())
    m = m_gpu.cpu().numpy()
    assert np.array_equal(m, orc.act_stats_max(Xf))
    res = awq.search(X.cuda(), W.cuda(), m_gpu)
    ref = orc.search(Xf, Wf, m, orc.alpha_grid(21))
    assert rel_err(res.losses.cpu().numpy(), ref["losses"]).max() <= LOSS_RTOL
    check_alpha_star(res.best, ref["losses"])
    assert np.array_equal(res.s_star.cpu().numpy(), orc.scales(m, orc.alpha_grid(21)[res.best]))


def test_stream_nonfinite_batch_is_reported(awq):
    acc = awq.StatsAccumulator(256, "cuda")
    X = torch.randn(64, 256).to(torch.bfloat16).cuda()
    acc.add_batch(X)
    Xn = X.clone()
    Xn[5, 9] = float("inf")
    with pytest.raises(AwqError) as e:
        acc.add_batch(Xn)
    assert e.value.name == "AWQ_ERR_NONFINITE"
