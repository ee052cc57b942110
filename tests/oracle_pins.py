"""Checks that pin the CPU oracle to things other than itself.

Each check takes the oracle module as an argument so the same checks can be
run against deliberately broken copies (``test_oracle_mutants.py``): every
plausible slip in the oracle (a dropped term, a wrong sign, a transposed
operand, a wrong rounding rule) must make at least one check fail.

What each check stands on:
  worked_sym / worked_asym  hand-worked values in tests/golden (symmetric: the
                            aiqz article's worked absmax formula; asymmetric:
                            the reading written in the fixture)
  brute_force_codes         nearest grid point by enumerating all 16 codes
  loss_triple_loop          L written as ||X S^-1 W'hat - X W||^2 with explicit
                            Python loops (not the difference form, no BLAS)
  alpha_zero_is_rtn         alpha = 0 gives s = 1: plain RTN group quantisation,
                            built here by brute force
  error_bound               |w'hat - w'| <= step * (1/2 + 2^-6)
  scale_invariance          s -> 2^k s leaves codes and the loss unchanged
  separability              loss over all columns = sum over a column split
  act_stats_closed_forms    mean|x| on inputs with a known answer
  argmin_first / L(a*)<=L(0)
"""
from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_round(a):
    """Round float32 values to bf16 precision (round to nearest even), as float32."""
    a = np.asarray(a, dtype=F32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(F32)


def small_layer(seed, N=16, D_in=16, D_out=16, outliers=(3,), factor=40.0, sigma=0.02):
    rng = _rng(seed)
    X = rng.standard_normal((N, D_in)).astype(F32)
    for j in outliers:
        X[:, j] *= F32(factor)
    W = (rng.standard_normal((D_in, D_out)) * sigma).astype(F32)
    return _bf16_round(X), _bf16_round(W)


# ---------------------------------------------------------------------------
def check_worked_sym(orc):
    g = read_golden("sym_worked_example.txt")
    w = np.array([float(v) for v in g["w_s"]], dtype=F32).reshape(-1, 1)
    codes, step, zero = orc.quantize_groups(w, int(g["group_size"][0]), True)
    assert float(step[0, 0]) == float(g["delta"][0]), (step, g["delta"])
    assert [int(c) for c in codes[:, 0]] == [int(v) for v in g["nibble"]], codes[:, 0]
    assert float(zero[0, 0]) == 8.0
    deq = orc.dequantize(codes, step, zero, int(g["group_size"][0]))[:, 0]
    assert np.array_equal(deq, np.array([float(v) for v in g["dequant"]], dtype=F32)), deq


def check_worked_asym(orc):
    g = read_golden("asym_worked_example.txt")
    w = np.array([float(v) for v in g["w"]], dtype=F32).reshape(-1, 1)
    codes, step, zero = orc.quantize_groups(w, int(g["group_size"][0]), False)
    assert float(step[0, 0]) == float(g["step"][0]), step
    assert float(zero[0, 0]) == float(g["zero"][0]), zero
    assert [int(c) for c in codes[:, 0]] == [int(v) for v in g["code"]], codes[:, 0]
    deq = orc.dequantize(codes, step, zero, int(g["group_size"][0]))[:, 0]
    assert np.array_equal(deq, np.array([float(v) for v in g["dequant"]], dtype=F32)), deq


def _nearest_code(x, step, zero, lo, hi):
    """Code c in [lo, hi] whose dequant (c - zero)*step is nearest x; ties -> even (c - zero)."""
    best, bestd = None, None
    for c in range(lo, hi + 1):
        d = abs(float(x) / float(step) - (c - float(zero)))
        if bestd is None or d < bestd - 1e-12 or (abs(d - bestd) <= 1e-12 and (c - int(zero)) % 2 == 0):
            best, bestd = c, d
    return best


def check_brute_force_codes(orc, seed=0):
    for sym, g in itertools.product((False, True), (8, 16)):
        rng = _rng(seed + 7 * g + sym)
        Wp = (rng.standard_normal((32, 12)) * 0.3).astype(F32)
        Wp[0:g, 0] = np.abs(Wp[0:g, 0])          # a one-signed group
        Wp[g:2 * g, 1] = -np.abs(Wp[g:2 * g, 1])  # a negative one-signed group
        codes, step, zero = orc.quantize_groups(Wp, g, sym)
        lo, hi = (1, 15) if sym else (0, 15)
        for j in range(Wp.shape[0]):
            for n in range(Wp.shape[1]):
                t = j // g
                st, z = step[t, n], zero[t, n]
                assert st > 0
                want = _nearest_code(Wp[j, n], st, z, lo, hi)
                assert int(codes[j, n]) == want, (sym, g, j, n, codes[j, n], want)
        # the zero point dequantises to exactly 0
        assert np.all((zero - zero.astype(np.int64)) == 0)
        # step is the smallest fp16 value covering the range: range/15 or max/7 rounded
        Wg = Wp.reshape(-1, g, Wp.shape[1])
        if sym:
            want_step = (np.abs(Wg).max(axis=1) / F32(7)).astype(np.float16).astype(F32)
        else:
            rngw = np.maximum(Wg.max(axis=1), 0) - np.minimum(Wg.min(axis=1), 0)
            want_step = (rngw / F32(15)).astype(np.float16).astype(F32)
        assert np.array_equal(step, want_step)


def _scaled_quant_dequant_bruteforce(W, s, g, sym, orc):
    """S^-1 W'hat built element by element from nearest codes (float64)."""
    Wp = (W * s[:, None]).astype(F32)
    _, step, zero = orc.quantize_groups(Wp, g, sym)
    lo, hi = (1, 15) if sym else (0, 15)
    out = np.zeros(W.shape, dtype=np.float64)
    for j in range(W.shape[0]):
        for n in range(W.shape[1]):
            t = j // g
            c = _nearest_code(Wp[j, n], step[t, n], zero[t, n], lo, hi)
            out[j, n] = (c - float(zero[t, n])) * float(step[t, n]) / float(s[j])
    return out


def check_loss_triple_loop(orc, seed=1):
    for sym, g in ((False, 8), (True, 16), (False, 16)):
        X, W = small_layer(seed + g)
        a = orc.act_stats(X)
        grid = orc.alpha_grid(5)
        res = orc.search(X, W, a, grid, group_size=g, symmetric=sym)
        for k, alpha in enumerate(grid):
            s = orc.scales(a, alpha)
            Wh = _scaled_quant_dequant_bruteforce(W, s, g, sym, orc)
            N, D_in = X.shape
            D_out = W.shape[1]
            L = 0.0
            for r in range(N):
                for n in range(D_out):
                    yq = 0.0
                    y = 0.0
                    for j in range(D_in):
                        yq += float(X[r, j]) * Wh[j, n]
                        y += float(X[r, j]) * float(W[j, n])
                    L += (yq - y) ** 2
            got = res["losses"][k]
            assert abs(got - L) <= 1e-9 * max(L, 1e-30), (sym, g, k, got, L)


def check_alpha_zero_is_rtn(orc, seed=2):
    X, W = small_layer(seed)
    a = orc.act_stats(X)
    res = orc.search(X, W, a, orc.alpha_grid(3), group_size=8, symmetric=False)
    ones = np.ones(W.shape[0], dtype=F32)
    assert np.array_equal(orc.scales(a, 0.0), ones)
    Wh = _scaled_quant_dequant_bruteforce(W, ones, 8, False, orc)
    E = X.astype(np.float64) @ (Wh - W.astype(np.float64))
    assert abs(res["losses"][0] - float((E * E).sum())) <= 1e-9 * float((E * E).sum())


def check_error_bound(orc, seed=3):
    rng = _rng(seed)
    for sym in (False, True):
        W = (rng.standard_normal((256, 64)) * 0.02).astype(F32)
        s = (rng.uniform(0.5, 30.0, 256)).astype(F32)
        Wp = (W * s[:, None]).astype(F32)
        codes, step, zero = orc.quantize_groups(Wp, 128, sym)
        deq = orc.dequantize(codes, step, zero, 128)
        err = np.abs(deq - Wp).reshape(2, 128, 64)
        assert np.all(err <= step[:, None, :] * (0.5 + 2.0 ** -6)), float((err / step[:, None, :]).max())


def check_scale_invariance(orc, seed=4):
    X, W = small_layer(seed, N=24, D_in=32, D_out=8)
    a = orc.act_stats(X)
    for sym in (False, True):
        for alpha in (0.35, 0.8):
            s = orc.scales(a, alpha)
            c1, st1, z1 = orc.quantize_groups((W * s[:, None]).astype(F32), 16, sym)
            s2 = (s * F32(4.0)).astype(F32)
            c2, st2, z2 = orc.quantize_groups((W * s2[:, None]).astype(F32), 16, sym)
            assert np.array_equal(c1, c2) and np.array_equal(z1, z2)
            assert np.array_equal(st2, st1 * F32(4.0))
            d1 = orc.candidate_delta(W, s, 16, sym)
            d2 = orc.candidate_delta(W, s2, 16, sym)
            assert np.array_equal(d1, d2)


def check_separability(orc, seed=5):
    X, W = small_layer(seed, N=20, D_in=32, D_out=24)
    a = orc.act_stats(X)
    grid = orc.alpha_grid(6)
    full = orc.search(X, W, a, grid, group_size=16)
    left = orc.search(X, W, a, grid, group_size=16, cols=np.arange(0, 10))
    right = orc.search(X, W, a, grid, group_size=16, cols=np.arange(10, 24))
    np.testing.assert_allclose(left["losses"] + right["losses"], full["losses"], rtol=1e-12)
    np.testing.assert_allclose(full["col_losses"][:, 3:5], left["col_losses"][:, 3:5], rtol=1e-12)


def check_act_stats_closed_forms(orc):
    X = np.full((5, 4), -0.75, dtype=F32)
    assert np.array_equal(orc.act_stats(X), np.full(4, 0.75, dtype=F32))
    X = np.zeros((8, 3), dtype=F32)
    X[2] = [4.0, -8.0, 0.5]
    assert np.array_equal(orc.act_stats(X), np.array([0.5, 1.0, 0.0625], dtype=F32))
    rng = _rng(6)
    X = rng.standard_normal((7, 5)).astype(F32)
    want = []
    for j in range(5):
        acc = 0.0
        for r in range(7):
            acc += abs(float(X[r, j]))
        want.append(acc / 7)
    np.testing.assert_allclose(orc.act_stats(X), np.array(want), rtol=1e-7)


def check_argmin_and_improvement(orc, seed=7):
    X, W = small_layer(seed, N=32, D_in=32, D_out=16, outliers=(1, 9), factor=60.0)
    a = orc.act_stats(X)
    res = orc.search(X, W, a, orc.alpha_grid(21), group_size=16)
    L = res["losses"]
    assert res["best"] == min(range(len(L)), key=lambda k: (L[k], k))
    assert L[res["best"]] <= L[0]
    # with strong outlier channels the scaled search beats plain RTN
    assert L[0] / L[res["best"]] > 1.0
    assert np.array_equal(res["s_star"], orc.scales(a, orc.alpha_grid(21)[res["best"]]))


def check_pack_layout(orc):
    W = np.array([[0.875], [-0.4375], [0.0625], [0.1625], [0.225], [-0.875], [0.3125], [0.1875]], dtype=F32)
    s = np.ones(8, dtype=F32)
    qw, sc, z = orc.pack(W, s, group_size=8, symmetric=True)
    # nibbles 15 4 | 8 9 | 10 1 | 10 10 (even row low)
    assert [int(b) for b in qw[:, 0]] == [0x4F, 0x98, 0x1A, 0xAA], qw[:, 0]
    assert float(sc[0, 0]) == 0.125 and float(z[0, 0]) == 8.0
    assert np.array_equal(orc.unpack_codes(qw)[:, 0], np.array([15, 4, 8, 9, 10, 1, 10, 10]))


ALL_CHECKS = [
    check_worked_sym, check_worked_asym, check_brute_force_codes, check_loss_triple_loop,
    check_alpha_zero_is_rtn, check_error_bound, check_scale_invariance, check_separability,
    check_act_stats_closed_forms, check_argmin_and_improvement, check_pack_layout,
]


def check_scales_closed_forms(orc):
    a = np.array([4.0, 0.25, 9.0, 1e-6, 0.0, 2.0], dtype=F32)
    # alpha = 1 returns the (floored) statistic itself, alpha = 0 returns 1
    assert np.array_equal(orc.scales(a, 1.0), np.array([4.0, 0.25, 9.0, 1e-4, 1e-4, 2.0], dtype=F32))
    assert np.array_equal(orc.scales(a, 0.0), np.ones(6, dtype=F32))
    # alpha = 1/2 is the square root (exact for these values)
    assert np.array_equal(orc.scales(a[:3], 0.5), np.array([2.0, 0.5, 3.0], dtype=F32))
    # pow(2, 0.25) rounded to float32
    assert orc.scales(a[5:], 0.25)[0] == F32(2.0 ** 0.25)


ALL_CHECKS.append(check_scales_closed_forms)


def check_zero_point_is_canonical(orc):
    """A zero point is an integer code: a group whose minimum is 0 stores +0, not -0."""
    W = np.abs(np.linspace(0.1, 1.0, 16, dtype=F32)).reshape(16, 1)
    _, qs, qz = orc.pack(W, np.ones(16, dtype=F32), group_size=16, symmetric=False)
    assert qz.view(np.uint16)[0, 0] == 0


ALL_CHECKS.append(check_zero_point_is_canonical)


# ---------------------------------------------------------------- W4A16 product
def check_w4a16_hand_bytes(orc):
    """Two groups of two rows, two columns: every code, zero, scale and 1/s
    worked by hand from (code - zero) * scale / s_j."""
    qweight = np.array([[0x3A, 0x0F], [0x81, 0x77]], dtype=np.uint8)
    scales = np.array([[0.5, 1.0], [0.25, 2.0]], dtype=np.float16)
    zeros = np.array([[8, 0], [8, 5]], dtype=np.float16)
    s = np.array([1.0, 2.0, 4.0, 0.5], dtype=F32)
    X = np.vstack([np.eye(4), np.ones((1, 4))]).astype(F32)
    # column 0: codes 10, 3, 1, 8 -> 1.0, -2.5, -1.75, 0 -> / s -> 1.0, -1.25, -0.4375, 0
    # column 1: codes 15, 0, 7, 7 -> 15, 0, 4, 4      -> / s -> 15, 0, 1, 8
    want = np.array([[1.0, 15.0], [-1.25, 0.0], [-0.4375, 1.0], [0.0, 8.0], [-0.6875, 24.0]])
    Y = orc.w4a16_matmul(X, qweight, scales, zeros, s, group_size=2)
    assert np.array_equal(Y, want), Y
    # without s the dequantised weights themselves
    Y = orc.w4a16_matmul(np.eye(4, dtype=F32), qweight, scales, zeros, None, group_size=2)
    assert np.array_equal(Y, np.array([[1.0, 15.0], [-2.5, 0.0], [-1.75, 4.0], [0.0, 4.0]]))


def _grid_layer(rng, D_in, D_out, g, sym):
    """W = (q - z) * step / s with power-of-two steps and scales: weights that
    the quantiser reproduces exactly (each group-column holds both ends of its
    code range, so the range gives back the same step and zero)."""
    T = D_in // g
    e = rng.integers(-9, -3, size=(T, D_out))
    step = np.ldexp(1.0, e)
    if sym:
        q = rng.integers(-7, 8, size=(T, g, D_out)).astype(np.float64)
        q[:, 0, :] = np.where(rng.random((T, D_out)) < 0.5, 7.0, -7.0)
        z = np.zeros((T, D_out))
    else:
        z = rng.integers(0, 16, size=(T, D_out)).astype(np.float64)
        q = rng.integers(0, 16, size=(T, g, D_out)).astype(np.float64)
        q[:, 0, :] = 0.0
        q[:, 1, :] = 15.0
        q = q - z[:, None, :]
    s = np.ldexp(1.0, rng.integers(-3, 4, size=D_in))
    Wp = (q * step[:, None, :]).reshape(D_in, D_out)
    return (Wp / s[:, None]).astype(F32), s.astype(F32)


def check_w4a16_grid_roundtrip(orc, seed=8):
    """On weights the quantiser reproduces exactly, pack followed by the
    W4A16 product is the plain product X W."""
    rng = _rng(seed)
    for sym in (False, True):
        W, s = _grid_layer(rng, 64, 24, 16, sym)
        X = rng.standard_normal((9, 64)).astype(F32)
        qw, sc, z = orc.pack(W, s, group_size=16, symmetric=sym)
        Y = orc.w4a16_matmul(X, qw, sc, z, s, group_size=16)
        ref = X.astype(np.float64) @ W.astype(np.float64)
        np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def check_w4a16_error_bound(orc, seed=9):
    """Off the grid: |Y - X W| <= sum_j |x_j| / s_j * step_jn * (1/2 + 2^-6)."""
    rng = _rng(seed)
    for sym in (False, True):
        W = (rng.standard_normal((128, 40)) * 0.02).astype(F32)
        s = rng.uniform(0.5, 20.0, 128).astype(F32)
        X = rng.standard_normal((6, 128)).astype(F32)
        qw, sc, z = orc.pack(W, s, group_size=32, symmetric=sym)
        Y = orc.w4a16_matmul(X, qw, sc, z, s, group_size=32)
        ref = X.astype(np.float64) @ W.astype(np.float64)
        step_rows = np.repeat(sc.astype(np.float64), 32, axis=0)           # [D_in, D_out]
        bound = (np.abs(X.astype(np.float64)) / s.astype(np.float64)[None, :]) @ (step_rows * (0.5 + 2.0 ** -6))
        assert np.all(np.abs(Y - ref) <= bound * (1 + 1e-9) + 1e-12)


ALL_CHECKS += [check_w4a16_hand_bytes, check_w4a16_grid_roundtrip, check_w4a16_error_bound]


# ---------------------------------------------------------------- streaming statistic and max variant
def check_act_stats_max_closed_forms(orc):
    X = np.array([[1.0, -2.0, 0.0], [-3.5, 0.5, 0.0], [2.0, -0.25, 0.0]], dtype=F32)
    assert np.array_equal(orc.act_stats_max(X), np.array([3.5, 2.0, 0.0], dtype=F32))
    # one row: |x| itself; max >= mean everywhere
    rng = _rng(10)
    X = rng.standard_normal((9, 7)).astype(F32)
    assert np.array_equal(orc.act_stats_max(X[:1]), np.abs(X[0]))
    assert np.all(orc.act_stats_max(X) >= orc.act_stats(X))


def check_act_stats_stream_matches_single_shot(orc):
    """On dyadic inputs every float64 sum is exact, so the batch-by-batch mean
    equals the one-shot mean bit for bit whatever the split; and a batch of
    constant |x| = c gives c."""
    rng = _rng(11)
    X = (rng.integers(-64, 65, size=(37, 6)) / 8.0).astype(F32)
    one = orc.act_stats(X)
    for cuts in ([37], [5, 32], [1, 1, 35], [12, 12, 13]):
        parts = np.split(X, np.cumsum(cuts)[:-1])
        assert np.array_equal(orc.act_stats_stream(parts), one)
    c = np.full((4, 3), -0.375, dtype=F32)
    assert np.array_equal(orc.act_stats_stream([c, c[:1]]), np.full(3, 0.375, dtype=F32))
    # the running total is divided by the rows of all batches, not averaged per batch
    a = np.ones((1, 2), dtype=F32)
    b = np.zeros((3, 2), dtype=F32)
    assert np.array_equal(orc.act_stats_stream([a, b]), np.full(2, 0.25, dtype=F32))


ALL_CHECKS += [check_act_stats_max_closed_forms, check_act_stats_stream_matches_single_shot]


# ---------------------------------------------------------------- the ADR's greedy search
def check_greedy_group_error_bruteforce(orc, seed=12):
    """The greedy's objective written out element by element with the
    nearest-code quantiser: sum_j a_j sum_n (w'hat_jn / s_j - w_jn)^2."""
    rng = _rng(seed)
    for sym in (False, True):
        Wg = (rng.standard_normal((8, 5)) * 0.02).astype(F32)
        s = np.array([1, 2, 0.5, 1, 4, 1, 0.25, 1], dtype=F32)
        a = rng.uniform(0.1, 3.0, 8)
        Wh = _scaled_quant_dequant_bruteforce(Wg, s, 8, sym, orc)
        want = 0.0
        for j in range(8):
            for n in range(5):
                d = Wh[j, n] - float(Wg[j, n])
                want += float(a[j]) * d * d
        got = orc.group_error(Wg, s, a, sym)
        assert abs(got - want) <= 1e-12 * want, (got, want)


def check_greedy_decisions(orc, seed=13):
    """Every decision is the argmin of the group error over the candidates
    (recomputed here independently), never worse than keeping the current
    scale; grid = powers of two around 1; a salient channel ends above 1."""
    rng = _rng(seed)
    cand = orc.greedy_candidates()
    assert len(cand) == 20 and cand[10] == 1.0 and np.all(cand[1:] == 2 * cand[:-1])
    W = (rng.standard_normal((16, 12)) * 0.02).astype(F32)
    a = rng.uniform(0.5, 1.5, 16)
    a[5] = 60.0                     # salient channel ...
    W[5] *= 0.1                     # ... whose weights sit far below the group max
    W[2] = 0.0                      # every candidate gives the same error: the scale stays 1
    for sym in (False, True):
        s, trace, errors = orc.greedy_search(W, a, group_size=8, symmetric=sym, passes=2)
        # replay: each decision against errors recomputed from the running s
        cur = np.ones(16, dtype=F32)
        for p in range(2):
            for j in range(16):
                t = j // 8
                rows = slice(8 * t, 8 * t + 8)
                e = []
                for c in cand:
                    trial = cur[rows].copy()
                    trial[j - 8 * t] = c
                    e.append(orc.group_error(W[rows], trial, a[rows], sym))
                e = np.array(e)
                np.testing.assert_allclose(errors[p, j], e, rtol=1e-12)
                k = int(trace[p, j])
                prev = int(np.flatnonzero(cand == cur[j])[0])
                assert e[k] == e.min() and e[k] <= e[prev]
                assert k == prev or e[k] < e[prev]
                cur[j] = cand[k]
        assert np.array_equal(cur, s)
        assert s[5] > 1.0 and s[2] == 1.0
        assert orc.group_error(W[:8], s[:8], a[:8], sym) < orc.group_error(W[:8], np.ones(8, F32), a[:8], sym)


ALL_CHECKS += [check_greedy_group_error_bruteforce, check_greedy_decisions]


# ---------------------------------------------------------------- closed-form scale
def check_closed_form_scales(orc):
    """Rows of constant magnitude c give mean |W_i| = c; alpha = 0 gives 1/c;
    alpha = 1/2 the square root over c; a zero row gets 1; the floor applies
    to the statistic."""
    W = np.array([[0.5, -0.5, 0.5, -0.5], [2.0, 2.0, -2.0, 2.0], [0.0, 0.0, 0.0, 0.0],
                  [0.25, -0.75, 0.0, 0.5]], dtype=F32)
    a = np.array([4.0, 9.0, 3.0, 0.0], dtype=F32)
    assert np.array_equal(orc.closed_form_scales(W, a, 0.0), np.array([2.0, 0.5, 1.0, F32(1 / 0.375)], dtype=F32))
    floored = np.sqrt(np.float64(F32(1e-4)))  # the statistic's floor is the fp32 value of 1e-4
    assert np.array_equal(orc.closed_form_scales(W, a, 0.5), np.array([4.0, 1.5, 1.0, F32(floored / 0.375)], dtype=F32))
    assert np.array_equal(orc.closed_form_scales(W, a, 1.0)[:2], np.array([8.0, 4.5], dtype=F32))


ALL_CHECKS.append(check_closed_form_scales)


# ---------------------------------------------------------------- subnormal fp16 steps
def check_subnormal_step_codes(orc, seed=14):
    """Groups so small that the fp16 step is subnormal and rounds far below
    the raw step (1.4 * 2^-24 -> 2^-24): a negative asymmetric group then has
    -min/step = 21 and zero 15, a symmetric one max|w|/step = 9.8.  Every
    code is still the nearest of the 16 (brute force), so the group minimum
    takes the lowest code and the symmetric extremes +-7."""
    rng = _rng(seed)
    for sym in (False, True):
        m = F32((9.8 if sym else 21.0) * 2.0 ** -24)
        frac = rng.random((16, 6)).astype(F32)
        Wp = (frac * 2 - 1) * m if sym else -frac * m
        Wp[0] = -m
        Wp = _bf16_round(Wp)
        codes, step, zero = orc.quantize_groups(Wp, 16, sym)
        assert np.all(step == F32(2.0 ** -24)), step
        if not sym:
            assert np.all(zero == 15.0) and np.all(-Wp[0] / step[0] > 15.5)
        lo, hi = (1, 15) if sym else (0, 15)
        for j in range(Wp.shape[0]):
            for n in range(Wp.shape[1]):
                assert int(codes[j, n]) == _nearest_code(Wp[j, n], step[0, n], zero[0, n], lo, hi), (sym, j, n)
        assert np.all(codes[0] == lo)


ALL_CHECKS.append(check_subnormal_step_codes)


# ---------------------------------------------------------------- relative error (aiqz section 5)
def check_relative_error_hand(orc):
    """epsilon = ||X (W - W_hat)||^2 / ||X W||^2 on a 2 x 2 case worked by
    hand: X W = [[3, 2], [7, 4]], whose squares sum to 9 + 4 + 49 + 16 = 78, so
    a loss of 39 is epsilon = 1/2 and a loss of 78 is 1.  The loss itself is
    the search's, and a quantised layer's epsilon is its loss over the same
    energy (checked against a product formed element by element)."""
    X = np.array([[1.0, 2.0], [3.0, 4.0]], dtype=F32)
    W = np.array([[1.0, 0.0], [1.0, 1.0]], dtype=F32)
    assert orc.relative_error(X, W, 39.0) == 0.5
    assert orc.relative_error(X, W, 78.0) == 1.0
    Xs, Ws = small_layer(21, N=8, D_in=16, D_out=4)
    res = orc.search(Xs, Ws, orc.act_stats(Xs), orc.alpha_grid(3), group_size=8, symmetric=True)
    energy = 0.0
    for r in range(Xs.shape[0]):
        for n in range(Ws.shape[1]):
            y = sum(float(Xs[r, j]) * float(Ws[j, n]) for j in range(Xs.shape[1]))
            energy += y * y
    for L in res["losses"]:
        assert abs(orc.relative_error(Xs, Ws, float(L)) - float(L) / energy) <= 1e-12 * float(L) / energy


ALL_CHECKS.append(check_relative_error_hand)
