"""The W4A16 product on a packed layer, CUDA path against the CPU oracle.

Tolerance, from the arithmetic of the kernel: every weight enters the tensor
cores as bf16(RN(RN((code - zero) * scale) * RN(1/s_j))), where (code - zero)
* scale is exact, so its relative error is at most 2^-8 + 2^-22; the bf16 x
bf16 products are exact and K of them accumulate in fp32 (at most K * 2^-23
relative to sum |x w|); Y is rounded once to bf16 (2^-8 relative).  So
elementwise |Y - Y_ref| <= (2^-8 + 2^-22 + K 2^-23) A (1 + 2^-8) + 2^-8 |Y_ref|
with A = sum_j |x_j| |w_hat_j| / s_j.  That bound is loose (A is ~sqrt(K)
times |Y|), so the relative Frobenius error is also held to 2^-7, about five
times the expected size of the rounding noise: a systematic slip (a wrong
group's scale, a dropped zero) moves it by far more.

The decode form (M <= 4) stays well inside the same bound: its codes enter
the tensor cores as the exact bf16 values 128 + code, against x' = x / s split
into bf16 hi + lo parts (2^-16 of x'); the products are exact, the sums fp32,
and the 128 bias comes off with the group's fp32 row sum before the scale.

The oracle's packed inputs always come from the oracle's own pack; the GPU
runs on the GPU pack, which these tests first check to be bit-identical.
"""
import numpy as np
import pytest
import torch

from gpu_common import require_gpu
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import synth

pytestmark = pytest.mark.gpu

FRO_TOL = 2.0 ** -7


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


def _abs_dequant(qweight, scales, zeros, group_size):
    codes = orc.unpack_codes(qweight).astype(np.float64)
    g = np.arange(codes.shape[0]) // group_size
    return np.abs(codes - zeros.astype(np.float64)[g]) * scales.astype(np.float64)[g]


def check_close(Y, Y_ref, X, s, qweight, scales, zeros, group_size):
    K = X.shape[1]
    Xa = np.abs(X.astype(np.float64))
    if s is not None:
        Xa = Xa / s.astype(np.float64)[None, :]
    A = Xa @ _abs_dequant(qweight, scales, zeros, group_size)
    u = 2.0 ** -8 + 2.0 ** -22 + K * 2.0 ** -23
    bound = u * A * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(Y_ref)
    err = np.abs(Y - Y_ref)
    assert np.all(np.isfinite(Y))
    assert np.all(err <= bound), f"max err / bound {float((err / np.maximum(bound, 1e-300)).max()):.3g}"
    fro = np.linalg.norm(Y - Y_ref) / max(np.linalg.norm(Y_ref), 1e-300)
    assert fro <= FRO_TOL, f"relative Frobenius error {fro:.3g}"
    return fro


def _layer(seed, M, D_in, D_out, g, sym, alpha=0.5, w_sigma=0.02):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, D_in)).astype(np.float32)
    k = max(1, D_in // 100)
    ch = rng.choice(D_in, k, replace=False)
    X[:, ch] *= rng.uniform(10, 100, k).astype(np.float32)
    W = (rng.standard_normal((D_in, D_out)) * w_sigma).astype(np.float32)
    Xb, Wb = synth.to_bf16(X), synth.to_bf16(W)
    Xf, Wf = synth.bf16_to_f32(Xb), synth.bf16_to_f32(Wb)
    s = orc.scales(orc.act_stats(Xf), alpha)
    return Xb, Wb, Xf, Wf, s


CASES = [
    # M, D_in, D_out, group, symmetric: ragged rows (not a multiple of 512), ragged
    # columns (not a multiple of 256), several K steps per group, every group size;
    # M <= 4 takes the decode path: 64-row x 1024-column stages in contiguous runs per
    # CTA -- one stage per CTA, runs that cross column blocks, column blocks whose
    # segments need more than one batch of the final sum, a ragged last block
    (1, 256, 272, 128, False),
    (2, 320, 784, 64, True),
    (3, 768, 1040, 256, False),
    (1, 64, 8192, 64, True),
    (4, 1024, 28672, 128, False),
    (2, 8192, 2048, 256, True),
    (5, 1024, 528, 128, True),
    (8, 576, 4096, 64, False),
    (200, 384, 784, 64, True),
    (600, 512, 1040, 128, False),
    (513, 768, 528, 256, True),
    (1100, 1024, 256, 128, False),
]


@pytest.mark.parametrize("M,D_in,D_out,g,sym", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}_g{c[3]}_{'sym' if c[4] else 'asym'}"
                                                          for c in CASES])
@pytest.mark.parametrize("with_s", [True, False], ids=["s", "no_s"])
def test_w4a16_matches_oracle(awq, M, D_in, D_out, g, sym, with_s):
    Xb, Wb, Xf, Wf, s = _layer(M * 7 + D_out, M, D_in, D_out, g, sym)
    qw, sc, z = orc.pack(Wf, s, g, sym)
    sd = torch.from_numpy(s).cuda() if with_s else None
    Y = awq.w4a16_matmul(Xb.cuda(), torch.from_numpy(qw).cuda(), torch.from_numpy(sc).cuda(),
                         torch.from_numpy(z).cuda(), sd, group_size=g)
    Yh = Y.float().cpu().numpy().astype(np.float64)
    ref = orc.w4a16_matmul(Xf, qw, sc, z, s if with_s else None, group_size=g)
    check_close(Yh, ref, Xf, s if with_s else None, qw, sc, z, g)


def test_w4a16_round_trip_through_the_path(awq):
    """stats -> search -> searched pack -> W4A16 product: the product of the
    packed layer approximates X W no worse than the search's own loss says."""
    w = synth.custom("w4a16_path", 21, 512, 512, 784, symmetric=False, group_size=128)
    X, W = synth.generate(w)
    Xf, Wf = synth.bf16_to_f32(X), synth.bf16_to_f32(W)
    Xd, Wd = X.cuda(), W.cuda()
    a = awq.act_stats(Xd)
    res = awq.search(Xd, Wd, a, group_size=128, symmetric=False)
    qw, sc, z = awq.quantize_pack_searched(Wd, res, 128, False)
    s_star = res.s_star.cpu().numpy()
    oq, osc, oz = orc.pack(Wf, s_star, 128, False)
    assert np.array_equal(qw.cpu().numpy(), oq)
    Y = awq.w4a16_matmul(Xd, qw, sc, z, res.s_star, group_size=128).float().cpu().numpy().astype(np.float64)
    ref = orc.w4a16_matmul(Xf, oq, osc, oz, s_star, group_size=128)
    check_close(Y, ref, Xf, s_star, oq, osc, oz, 128)
    # the oracle's product error is the search's loss at alpha*
    E = ref - Xf.astype(np.float64) @ Wf.astype(np.float64)
    L = float((E * E).sum())
    L_star = float(res.losses.cpu().numpy()[res.best])
    assert abs(L - L_star) <= 1e-2 * L_star


def test_w4a16_zero_groups_and_single_row(awq):
    Xb, Wb, Xf, Wf, s = _layer(5, 1, 256, 256, 128, False)
    Wf = Wf.copy()
    Wf[0:128, 0:16] = 0.0     # zero groups: scale 0, every dequantised weight 0
    qw, sc, z = orc.pack(Wf, s, 128, False)
    Y = awq.w4a16_matmul(Xb.cuda(), torch.from_numpy(qw).cuda(), torch.from_numpy(sc).cuda(),
                         torch.from_numpy(z).cuda(), torch.from_numpy(s).cuda(), group_size=128)
    Yh = Y.float().cpu().numpy().astype(np.float64)
    ref = orc.w4a16_matmul(Xf, qw, sc, z, s, group_size=128)
    check_close(Yh, ref, Xf, s, qw, sc, z, 128)


@pytest.mark.parametrize("name", ["attn_proj", "mlp_down", "large_mlp"])
def test_w4a16_full_size_sampled(awq, name):
    """Full-size layers, the product launched exactly as for the whole layer;
    the oracle checks a seeded sample of 64 rows x 512 columns."""
    w = synth.WORKLOADS[name]
    X, W = synth.generate(w)
    Xf, Wf = synth.bf16_to_f32(X), synth.bf16_to_f32(W)
    s = orc.scales(orc.act_stats(Xf[:2048]), 0.5)
    Xd, Wd = X.cuda(), W.cuda()
    sd = torch.from_numpy(s).cuda()
    qw, sc, z = awq.quantize_pack(Wd, sd, w.group_size, w.symmetric)
    Y = awq.w4a16_matmul(Xd, qw, sc, z, sd, group_size=w.group_size)
    rng = np.random.default_rng(w.seed + 100)
    rows = np.sort(rng.choice(w.N, 64, replace=False))
    cols = synth.sample_columns(w.D_out, 512, w.seed)
    oq, osc, oz = orc.pack(Wf[:, cols], s, w.group_size, w.symmetric)
    assert np.array_equal(qw[:, cols].cpu().numpy(), oq)
    Ys = Y[rows][:, cols].float().cpu().numpy().astype(np.float64)
    ref = orc.w4a16_matmul(Xf[rows], oq, osc, oz, s, group_size=w.group_size)
    check_close(Ys, ref, Xf[rows], s, oq, osc, oz, w.group_size)
    del Xd, Wd, Y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [1, 4, 8])
def test_w4a16_decode_full_size_sampled(awq, M):
    """The large MLP layer's weights with a decode-sized X; the oracle checks
    512 sampled columns."""
    w = synth.WORKLOADS["large_mlp"]
    rng = np.random.default_rng(200 + M)
    Wf = (rng.standard_normal((w.D_in, w.D_out)) * 0.01).astype(np.float32)
    Xf = rng.standard_normal((M, w.D_in)).astype(np.float32)
    s = rng.uniform(0.5, 4.0, w.D_in).astype(np.float32)
    Wb, Xb = synth.to_bf16(Wf), synth.to_bf16(Xf)
    Wf, Xf = synth.bf16_to_f32(Wb), synth.bf16_to_f32(Xb)
    sd = torch.from_numpy(s).cuda()
    qw, sc, z = awq.quantize_pack(Wb.cuda(), sd, w.group_size, w.symmetric)
    Y = awq.w4a16_matmul(Xb.cuda(), qw, sc, z, sd, group_size=w.group_size)
    cols = synth.sample_columns(w.D_out, 512, w.seed)
    oq, osc, oz = orc.pack(Wf[:, cols], s, w.group_size, w.symmetric)
    assert np.array_equal(qw[:, cols].cpu().numpy(), oq)
    Ys = Y[:, cols].float().cpu().numpy().astype(np.float64)
    ref = orc.w4a16_matmul(Xf, oq, osc, oz, s, group_size=w.group_size)
    check_close(Ys, ref, Xf, s, oq, osc, oz, w.group_size)
