"""The scale table s = fp32(pow(fp64(max(a, floor)), alpha)) bit for bit
against the oracle, over statistics spread across many binades (and zero
channels with a zero floor) and over grid and off-grid exponents: a search
with a one-point grid returns that point's scale row as s*."""
import numpy as np
import pytest
import torch

from gpu_common import require_gpu
from oracle import awq_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


@pytest.mark.parametrize("floor", [1e-4, 0.0])
def test_scale_table_matches_pow(awq, floor):
    rng = np.random.default_rng(61)
    D_in = 4096
    a = (10.0 ** rng.uniform(-7.0, 6.0, D_in)).astype(np.float32)
    a[:16] = np.float32(1.0)
    a[16:32] = np.float32(0.0)
    a[32:48] = np.float32(1e-40)          # subnormal statistics
    a[48:64] = rng.integers(1, 50, 16).astype(np.float32)
    X = torch.randn(16, D_in, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    W = (torch.randn(D_in, 8, generator=torch.Generator().manual_seed(2)) * 0.02).to(torch.bfloat16).cuda()
    ad = torch.from_numpy(a).cuda()
    alphas = list(orc.alpha_grid(21)) + [0.123456789, 0.999999, 1e-9, 1.0 / 3.0]
    bad = 0
    for alpha in alphas:
        # a zero floor lets zero or tiny channels give s = 0 or 1/s = inf, and the
        # losses are then not finite; only the scale row is checked here
        res = awq.search(X, W, ad, [float(alpha)], group_size=128, symmetric=True, act_floor=floor, check=False)
        got = res.s_star.cpu().numpy()
        want = orc.scales(a, alpha, act_floor=floor)
        bad += int(np.count_nonzero(got.view(np.uint32) != want.view(np.uint32)))
    assert bad == 0, bad
