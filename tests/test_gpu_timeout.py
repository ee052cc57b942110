"""The CTA-pair kernels' failure path, run on purpose (no fault, no trap):
waits that never complete expire after a short limit, AWQ_ERR_TIMEOUT
reaches the workspace's status word, every CTA leaves its roles, waits for
its bulk copy, meets its peer and frees TMEM; the same process and the same
workspace then run the whole path, which must still match the oracle."""
import numpy as np
import pytest
import torch

from gpu_common import LOSS_RTOL, check_alpha_star, rel_err, require_gpu, workload_cpu
from oracle import awq_oracle as orc

pytestmark = pytest.mark.gpu

AWQ_ERR_TIMEOUT = 9
LIMIT_NS = 1_000_000   # 1 ms instead of the product kernels' 2 s
PAIRS = 8


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


def test_expired_wait_then_the_path(awq):
    w, X, W, Xf, Wf = workload_cpu("tiny")
    Xd, Wd = X.cuda(), W.cuda()
    nb = awq.search_workspace_size(w.N, w.D_in, w.D_out, 21, w.group_size, w.symmetric)
    ws = torch.empty(max(nb, 256 + 4096), dtype=torch.uint8, device="cuda")
    ws[256:256 + 4096] = torch.randint(0, 256, (4096,), dtype=torch.uint8, device="cuda")

    rec = awq.selftest_wait_timeout(LIMIT_NS, PAIRS, ws)
    assert awq.workspace_status(ws) == AWQ_ERR_TIMEOUT
    # every CTA finished and freed its TMEM; the next kernels need all of it
    assert rec[0] == 2 * PAIRS, rec
    assert rec[1] == 2 * PAIRS, rec              # no wait of this kernel can complete
    assert rec[3] == 2 * PAIRS, rec              # the copy in flight was waited for
    assert 1_000 <= rec[2] < 200_000, rec        # the short limit applied (us), not the 2 s one

    # the same workspace: the search clears the status word and runs normally
    a = awq.act_stats(Xd)
    grid = orc.alpha_grid(21)
    res = awq.search(Xd, Wd, a, list(grid), group_size=w.group_size, symmetric=w.symmetric, ws=ws)
    qw, sc, z = awq.quantize_pack_searched(Wd, res, w.group_size, w.symmetric)
    torch.cuda.synchronize()
    assert awq.workspace_status(ws) == 0
    a_h = a.cpu().numpy()
    ref = orc.search(Xf, Wf, a_h, grid, group_size=w.group_size, symmetric=w.symmetric)
    L = res.losses.cpu().numpy()
    assert rel_err(L, ref["losses"]).max() <= LOSS_RTOL
    check_alpha_star(res.best, ref["losses"])
    s_star = res.s_star.cpu().numpy()
    assert np.array_equal(s_star, orc.scales(a_h, grid[res.best]))
    oq, osc, oz = orc.pack(Wf, s_star, group_size=w.group_size, symmetric=w.symmetric)
    assert np.array_equal(qw.cpu().numpy(), oq)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
    assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))
