"""Edge cases of the CUDA path: degenerate groups, the activation floor,
non-finite inputs, fp16 range overflow, determinism, small shapes."""
import numpy as np
import pytest
import torch

from gpu_common import LOSS_RTOL, STATS_RTOL, check_alpha_star, custom_cpu, rel_err, require_gpu
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import AwqError, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


def _layer(seed, N=96, D_in=256, D_out=264, sym=False):
    w = synth.custom(f"edge{seed}", seed, N, D_in, D_out, symmetric=sym)
    return custom_cpu(w)


def test_degenerate_groups_pack_and_search(awq):
    """An all-zero group (zero step), one-signed groups and a zero activation
    channel (the floor) go through pack and search like the oracle."""
    w, X, W, Xf, Wf = _layer(31)
    Wf = Wf.copy()
    Wf[0:128, 0:8] = 0.0                       # zero group -> step 0
    Wf[128:256, 8:16] = np.abs(Wf[128:256, 8:16])      # positive group
    Wf[0:128, 16:24] = -np.abs(Wf[0:128, 16:24])       # negative group
    Xf = Xf.copy()
    Xf[:, 5] = 0.0                              # dead channel -> mean 0 -> floor
    Wb, Xb = synth.to_bf16(Wf), synth.to_bf16(Xf)
    Wf, Xf = synth.bf16_to_f32(Wb), synth.bf16_to_f32(Xb)
    a_gpu = awq.act_stats(Xb.cuda())
    a = a_gpu.cpu().numpy()
    assert a[5] == 0.0
    for sym in (False, True):
        s = orc.scales(a, 0.7)
        assert s[5] == np.float32(np.float32(1e-4).astype(np.float64) ** 0.7)
        qw, sc, z = awq.quantize_pack(Wb.cuda(), torch.from_numpy(s).cuda(), 128, sym)
        oq, osc, oz = orc.pack(Wf, s, 128, sym)
        assert np.array_equal(qw.cpu().numpy(), oq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
        assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))
        res = awq.search(Xb.cuda(), Wb.cuda(), a_gpu, symmetric=sym)
        ref = orc.search(Xf, Wf, a, orc.alpha_grid(21), symmetric=sym)
        assert rel_err(res.losses.cpu().numpy(), ref["losses"]).max() <= LOSS_RTOL
        check_alpha_star(res.best, ref["losses"])


def test_exact_ties_in_pack(awq):
    """Weights placed exactly on half steps exercise the tie path of the pack."""
    D_in, D_out = 128, 256
    rng = np.random.default_rng(5)
    half = np.where(rng.random((D_in, D_out)) < 0.5, 0.5, 0.0)
    s = np.ones(D_in, dtype=np.float32)
    for sym in (True, False):
        codes = rng.integers(-6, 7, size=(D_in, D_out)).astype(np.float64)
        Wf = ((codes + half) / 64.0).astype(np.float32)
        if sym:
            Wf[0, :] = 7.0 / 64.0      # max |w| = 7/64: step 1/64 in every column
        else:
            Wf[0, :] = 7.0 / 64.0      # range [-8/64, 7/64]: step 1/64, zero 8
            Wf[1, :] = -8.0 / 64.0
        Wb = synth.to_bf16(Wf)
        Wf = synth.bf16_to_f32(Wb)
        qw, sc, z = awq.quantize_pack(Wb.cuda(), torch.from_numpy(s).cuda(), 128, sym)
        oq, osc, oz = orc.pack(Wf, s, 128, sym)
        assert np.all(osc.astype(np.float32) == np.float32(1 / 64))
        assert np.array_equal(qw.cpu().numpy(), oq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
        assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))


def test_nonfinite_inputs_report_status(awq):
    w, X, W, Xf, Wf = _layer(32)
    Xn = X.clone()
    Xn[3, 7] = float("nan")
    with pytest.raises(AwqError) as e:
        awq.act_stats(Xn.cuda())
    assert e.value.name == "AWQ_ERR_NONFINITE"
    Wn = W.clone()
    Wn[10, 3] = float("inf")
    s = torch.ones(W.shape[0], dtype=torch.float32, device="cuda")
    with pytest.raises(AwqError) as e:
        awq.quantize_pack(Wn.cuda(), s, 128, False)
    assert e.value.name == "AWQ_ERR_NONFINITE"
    a = awq.act_stats(X.cuda())
    with pytest.raises(AwqError) as e:
        awq.search(X.cuda(), Wn.cuda(), a)
    assert e.value.name == "AWQ_ERR_NONFINITE"


def test_fp16_step_overflow_is_range_error(awq):
    W = torch.full((128, 16), 3.0e4, dtype=torch.bfloat16)
    W[1::2] = -3.0e4
    s = torch.full((128,), 50.0, dtype=torch.float32, device="cuda")
    with pytest.raises(AwqError) as e:
        awq.quantize_pack(W.cuda(), s, 128, False)
    assert e.value.name == "AWQ_ERR_RANGE"


def test_search_is_deterministic(awq):
    w, X, W, Xf, Wf = _layer(33, N=260, D_in=384, D_out=520)
    a = awq.act_stats(X.cuda())
    r1 = awq.search(X.cuda(), W.cuda(), a, col_losses=True)
    L1 = r1.losses.clone()
    c1 = r1.col_losses.clone()
    r2 = awq.search(X.cuda(), W.cuda(), a, col_losses=True)
    assert torch.equal(L1, r2.losses) and torch.equal(c1, r2.col_losses)
    a2 = awq.act_stats(X.cuda())
    assert torch.equal(a, a2)


def test_single_row_and_single_candidate(awq):
    w, X, W, Xf, Wf = _layer(34, N=1, D_in=128, D_out=8)
    a_gpu = awq.act_stats(X.cuda())
    a = a_gpu.cpu().numpy()
    assert rel_err(a, orc.act_stats(Xf)).max() <= STATS_RTOL
    res = awq.search(X.cuda(), W.cuda(), a_gpu, grid=[0.5], col_losses=True)
    ref = orc.search(Xf, Wf, a, np.array([0.5]))
    assert res.best == 0
    assert rel_err(res.losses.cpu().numpy(), ref["losses"]).max() <= LOSS_RTOL


def test_uniform_activations_flat_loss(awq):
    """With every channel equally active, s is uniform and the loss barely
    moves across alpha (scale invariance of the group quantiser)."""
    rng = np.random.default_rng(8)
    Xf = np.where(rng.random((128, 256)) < 0.5, -0.5, 0.5).astype(np.float32)
    Wf = (rng.standard_normal((256, 256)) * 0.02).astype(np.float32)
    Xb, Wb = synth.to_bf16(Xf), synth.to_bf16(Wf)
    a = awq.act_stats(Xb.cuda())
    assert torch.all(a == 0.5)
    L = awq.search(Xb.cuda(), Wb.cuda(), a).losses.cpu().numpy()
    assert L.max() / L.min() < 1.01


def test_rejects_wrong_dtype(awq):
    X = torch.zeros(8, 128, device="cuda", dtype=torch.float32)
    with pytest.raises(TypeError):
        awq.act_stats(X)


def test_pack_searched_degenerate_groups_and_ties(awq):
    """The searched pack on zero groups, one-signed groups and weights exactly
    on half steps (|x| = 1 everywhere, so s = 1 for every alpha)."""
    rng = np.random.default_rng(9)
    D_in, D_out = 256, 264
    for sym in (False, True):
        Xf = np.where(rng.random((64, D_in)) < 0.5, -1.0, 1.0).astype(np.float32)
        half = np.where(rng.random((D_in, D_out)) < 0.5, 0.5, 0.0)
        codes = rng.integers(-6, 7, size=(D_in, D_out)).astype(np.float64)
        Wf = ((codes + half) / 64.0).astype(np.float32)
        Wf[0, :] = 7.0 / 64.0
        if not sym:
            Wf[1, :] = -8.0 / 64.0
        Wf[128:256, 0:8] = 0.0                             # zero group
        Wf[128:256, 8:16] = np.abs(Wf[128:256, 8:16])      # one-signed groups
        Xb, Wb = synth.to_bf16(Xf), synth.to_bf16(Wf)
        Wf = synth.bf16_to_f32(Wb)
        a = awq.act_stats(Xb.cuda())
        assert torch.all(a == 1.0)
        res = awq.search(Xb.cuda(), Wb.cuda(), a, symmetric=sym)
        qw, sc, z = awq.quantize_pack_searched(Wb.cuda(), res, 128, sym)
        s_star = res.s_star.cpu().numpy()
        assert np.all(s_star == 1.0)
        oq, osc, oz = orc.pack(Wf, s_star, 128, sym)
        assert np.array_equal(qw.cpu().numpy(), oq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
        assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))


def _subnormal_step_groups(rng, D_out, sym):
    """Two groups of 128 rows: the first with so small a range that the fp16
    step is subnormal and rounds far down (raw step 1.4 * 2^-24 -> 2^-24), the
    second ordinary.  Asymmetric: the first group is negative, so -min/step =
    21 and the zero is clamped to 15, leaving the minimum's rint(w/step) + 15
    below 0 unless the code is clamped; symmetric: max|w|/step = 9.8, so the
    largest codes need the clamp at 7."""
    Wf = (rng.standard_normal((256, D_out)) * 0.02).astype(np.float32)
    m = np.float32((21.0 if not sym else 9.8) * 2.0 ** -24)
    frac = rng.random((128, D_out)).astype(np.float32)
    Wf[:128] = -frac * m if not sym else (frac * 2 - 1) * m
    Wf[0] = -m
    return Wf


def test_pack_zero_clamped_by_a_subnormal_step(awq):
    """Codes on the group minimum where the zero is clamped at 15 (and, for
    symmetric codes, where the largest |w|/step exceeds 7.5): both packs
    bit-exact against the oracle, which clamps every code to [0, 15]."""
    rng = np.random.default_rng(21)
    D_out = 64
    for sym in (False, True):
        Wb = synth.to_bf16(_subnormal_step_groups(rng, D_out, sym))
        Wf = synth.bf16_to_f32(Wb)
        s = np.ones(256, dtype=np.float32)
        oq, osc, oz = orc.pack(Wf, s, 128, sym)
        if not sym:
            assert np.all(oz.astype(np.float32)[0] == 15.0)
        qw, sc, z = awq.quantize_pack(Wb.cuda(), torch.from_numpy(s).cuda(), 128, sym)
        assert np.array_equal(qw.cpu().numpy(), oq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
        assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))
        # the searched pack at s* = 1 (|x| = 1 everywhere, so s = 1 for every alpha)
        Xb = synth.to_bf16(np.where(rng.random((64, 256)) < 0.5, -1.0, 1.0).astype(np.float32))
        a = awq.act_stats(Xb.cuda())
        res = awq.search(Xb.cuda(), Wb.cuda(), a, symmetric=sym)
        assert np.all(res.s_star.cpu().numpy() == 1.0)
        qw, sc, z = awq.quantize_pack_searched(Wb.cuda(), res, 128, sym)
        assert np.array_equal(qw.cpu().numpy(), oq)
        assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))


def test_pack_takes_s_at_a_4_byte_offset(awq):
    """awq_quantize_pack reads s with plain loads: any 4-byte aligned s works
    (here a view one float into a buffer), with results equal to the oracle's."""
    w, X, W, Xf, Wf = _layer(34, D_in=256, D_out=136)
    rng = np.random.default_rng(34)
    s = (rng.random(256) * 3 + 0.25).astype(np.float32)
    buf = torch.zeros(257, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(s).cuda()
    sv = buf[1:]
    assert sv.data_ptr() % 16 == 4
    for sym in (False, True):
        qw, sc, z = awq.quantize_pack(W.cuda(), sv, 128, sym)
        oq, osc, oz = orc.pack(Wf, s, 128, sym)
        assert np.array_equal(qw.cpu().numpy(), oq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
        assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))
