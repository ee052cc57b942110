"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: pack codes / scales / zeros bit-exact given the same s; per-alpha
losses within 1e-2 relative; alpha* equal or within 1e-2 on the oracle's
loss; s* bit-exact; mean |X| within 1e-5 relative.
"""
import numpy as np
import pytest
import torch

from gpu_common import (LOSS_RTOL, PARITY_COLS, STATS_RTOL, check_alpha_star, check_column_losses, custom_cpu,
                        rel_err, require_gpu, workload_cpu)
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import synth

pytestmark = pytest.mark.gpu

NAMES = synth.ORDER
RAGGED = [
    # several tiles in every dimension plus a ragged tail (rows, columns)
    synth.custom("ragged_asym", 11, 300, 512, 776, symmetric=False, group_size=128),
    synth.custom("ragged_sym_g64", 12, 200, 384, 264, symmetric=True, group_size=64, w_sigma=0.015),
    synth.custom("short_rows_g256", 13, 40, 768, 520, symmetric=False, group_size=256),
]


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


# ---------------------------------------------------------------------------- GEMM main loop
@pytest.mark.parametrize("b_mn", [True, False], ids=["B_N_major", "B_K_major"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 328, 192), (512, 1024, 1024)])
def test_selftest_gemm_matches_matmul(awq, b_mn, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    Bdev = B.cuda() if b_mn else B.t().contiguous().cuda()
    C = awq.selftest_gemm(A.cuda(), Bdev, b_mn_major=b_mn).cpu().double()
    ref = A.double() @ B.double()
    err = (C - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() + 1e-6, err


# ---------------------------------------------------------------------------- step 1
@pytest.mark.parametrize("name", NAMES)
def test_act_stats(awq, name):
    w, X, W, Xf, Wf = workload_cpu(name)
    got = awq.act_stats(X.cuda()).cpu().numpy()
    want = orc.act_stats(Xf)
    assert rel_err(got, want).max() <= STATS_RTOL


@pytest.mark.parametrize("w", RAGGED, ids=[r.name for r in RAGGED])
def test_act_stats_ragged(awq, w):
    _, X, W, Xf, Wf = custom_cpu(w)
    got = awq.act_stats(X.cuda()).cpu().numpy()
    assert rel_err(got, orc.act_stats(Xf)).max() <= STATS_RTOL


def test_act_stats_strided(awq):
    """A leading dimension larger than D_in (a column slice of a wider matrix)."""
    import ctypes
    w = synth.custom("strided", 21, 130, 256, 256)
    _, X, _, Xf, _ = custom_cpu(w)
    wide = torch.zeros(130, 320, dtype=torch.bfloat16)
    wide[:, :256] = X
    wide[:, 256:] = 1000.0
    dev = wide.cuda()
    out = torch.empty(256, dtype=torch.float32, device="cuda")
    nb = awq.act_stats_workspace_size(130, 256)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    rc = awq.lib().awq_act_stats(ctypes.c_void_p(dev.data_ptr()), 130, 256, 320, ctypes.c_void_p(out.data_ptr()),
                                 ctypes.c_void_p(ws.data_ptr()), nb, None)
    assert rc == 0 and awq.workspace_status(ws) == 0
    assert rel_err(out.cpu().numpy(), orc.act_stats(Xf)).max() <= STATS_RTOL


# ---------------------------------------------------------------------------- step 4
def _pack_check(awq, Wb, Wf, s, g, sym):
    qw, sc, z = awq.quantize_pack(Wb.cuda(), torch.from_numpy(s).cuda(), group_size=g, symmetric=sym)
    oq, osc, oz = orc.pack(Wf, s, group_size=g, symmetric=sym)
    qw, sc, z = qw.cpu().numpy(), sc.cpu().numpy(), z.cpu().numpy()
    assert np.array_equal(sc.view(np.uint16), osc.view(np.uint16)), "scales differ"
    assert np.array_equal(z.view(np.uint16), oz.view(np.uint16)), "zeros differ"
    bad = np.count_nonzero(qw != oq)
    assert bad == 0, f"{bad} packed bytes differ"


@pytest.mark.parametrize("name", NAMES)
def test_pack_bit_exact(awq, name):
    w, X, W, Xf, Wf = workload_cpu(name)
    a = orc.act_stats(Xf)
    s = orc.scales(a, 0.5)
    _pack_check(awq, W, Wf, s, w.group_size, w.symmetric)


@pytest.mark.parametrize("w", RAGGED, ids=[r.name for r in RAGGED])
@pytest.mark.parametrize("alpha", [0.0, 0.35, 1.0])
def test_pack_bit_exact_ragged(awq, w, alpha):
    _, X, W, Xf, Wf = custom_cpu(w)
    s = orc.scales(orc.act_stats(Xf), alpha)
    _pack_check(awq, W, Wf, s, w.group_size, w.symmetric)


# ---------------------------------------------------------------------------- steps 2-3
def _search_full_check(awq, w, X, W, Xf, Wf):
    a_gpu = awq.act_stats(X.cuda())
    a = a_gpu.cpu().numpy()
    grid = orc.alpha_grid(21)
    assert list(grid) == awq.default_grid(21)
    res = awq.search(X.cuda(), W.cuda(), a_gpu, list(grid), group_size=w.group_size, symmetric=w.symmetric,
                     col_losses=True)
    ref = orc.search(Xf, Wf, a, grid, group_size=w.group_size, symmetric=w.symmetric)
    L = res.losses.cpu().numpy()
    assert rel_err(L, ref["losses"]).max() <= LOSS_RTOL, (L, ref["losses"])
    check_alpha_star(res.best, ref["losses"])
    s_star = res.s_star.cpu().numpy()
    assert np.array_equal(s_star, orc.scales(a, grid[res.best]))
    col = res.col_losses.cpu().numpy()
    check_column_losses(col, ref["col_losses"], label=w.name)
    np.testing.assert_allclose(col.sum(axis=1), L, rtol=1e-9)
    print(f"{w.name}: max per-alpha rel err {rel_err(L, ref['losses']).max():.3e}, best {res.best} / {ref['best']}")
    return res, ref


def test_search_tiny_full(awq):
    w, X, W, Xf, Wf = workload_cpu("tiny")
    res, ref = _search_full_check(awq, w, X, W, Xf, Wf)
    # the outlier channels make the scaled search beat plain RTN (alpha = 0)
    assert ref["losses"][0] / ref["losses"].min() > 1.0


@pytest.mark.parametrize("w", RAGGED, ids=[r.name for r in RAGGED])
def test_search_ragged_full(awq, w):
    _, X, W, Xf, Wf = custom_cpu(w)
    _search_full_check(awq, w, X, W, Xf, Wf)


@pytest.mark.parametrize("name", NAMES[1:])
def test_search_full_size_sampled_columns(awq, name):
    """Full-size launch; per-column losses of a seeded column sample against the
    oracle; totals checked through separability (L_k = sum of column losses)."""
    w, X, W, Xf, Wf = workload_cpu(name)
    a_gpu = awq.act_stats(X.cuda())
    a = a_gpu.cpu().numpy()
    grid = orc.alpha_grid(21)
    res = awq.search(X.cuda(), W.cuda(), a_gpu, list(grid), group_size=w.group_size, symmetric=w.symmetric,
                     col_losses=True)
    L = res.losses.cpu().numpy()
    col = res.col_losses.cpu().numpy()
    torch.cuda.empty_cache()
    cols = synth.sample_columns(w.D_out, PARITY_COLS, w.seed)
    ref = orc.search(Xf, Wf, a, grid, group_size=w.group_size, symmetric=w.symmetric, cols=cols)
    got = col[:, cols]
    err = rel_err(got.sum(axis=1), ref["losses"]).max()
    print(f"{name}: sampled per-alpha rel err {err:.3e}")
    assert err <= LOSS_RTOL
    check_column_losses(got, ref["col_losses"], label=f"{name} ({len(cols)} sampled columns)")
    np.testing.assert_allclose(col.sum(axis=1), L, rtol=1e-9)
    assert res.best == int(np.argmin(L))
    assert np.array_equal(res.s_star.cpu().numpy(), orc.scales(a, grid[res.best]))
    # the sample's own argmin agrees with the oracle's on that sample
    check_alpha_star(int(np.argmin(got.sum(axis=1))), ref["losses"])


# ---------------------------------------------------------------------------- step 4 after a search
def _searched_pack_check(awq, w, X, W, Xf, Wf):
    """awq_quantize_pack_searched equals the oracle's pack at the search's s*
    (and the standalone GPU pack) bit for bit."""
    Xd, Wd = X.cuda(), W.cuda()
    a = awq.act_stats(Xd)
    res = awq.search(Xd, Wd, a, group_size=w.group_size, symmetric=w.symmetric)
    qw, sc, z = awq.quantize_pack_searched(Wd, res, w.group_size, w.symmetric)
    s_star = res.s_star.cpu().numpy()
    torch.cuda.synchronize()
    oq, osc, oz = orc.pack(Wf, s_star, group_size=w.group_size, symmetric=w.symmetric)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16)), "scales differ"
    assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16)), "zeros differ"
    bad = np.count_nonzero(qw.cpu().numpy() != oq)
    assert bad == 0, f"{bad} packed bytes differ"
    q2, s2, z2 = awq.quantize_pack(Wd, res.s_star, w.group_size, w.symmetric)
    assert torch.equal(q2, qw) and torch.equal(s2, sc) and torch.equal(z2, z)


@pytest.mark.parametrize("name", NAMES)
def test_pack_searched_bit_exact(awq, name):
    w, X, W, Xf, Wf = workload_cpu(name)
    _searched_pack_check(awq, w, X, W, Xf, Wf)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", RAGGED, ids=[r.name for r in RAGGED])
def test_pack_searched_bit_exact_ragged(awq, w):
    _, X, W, Xf, Wf = custom_cpu(w)
    _searched_pack_check(awq, w, X, W, Xf, Wf)
