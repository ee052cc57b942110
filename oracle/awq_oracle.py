"""Plain CPU oracle of the AWQ calibration hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module: only
the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference arm
of ``bench.py`` may call it.  It shares no code, constants or helpers with the
CUDA path; it is a slow, literal restatement of what the pages define, step by
step, in numpy.  Quantisation is done in float32 (one IEEE round-to-nearest
operation per step), losses in float64.

Sources (page title, then section):
  [concept]  "AWQ (Activation-aware Weight Quantization)" (compassingai concept page)
  [aiqz]     aiqz.cc article "awq-activation-aware-quantization", sections 1-5
  [adr]      "009. AWQ Integration" (ADR), Decision / 关键设计
  [glossary] "量化推理算法 GPTQ / AWQ" (slowleelab), L4 section 4.1 / 4.3

Readings where the pages are silent or disagree:
  R1 statistic is mean|X_j| (the concept page also mentions max; the aiqz
     article and the ADR use the mean of absolute values).
  R2 the scale exponent grid is alpha_k = k/(G-1), computed in float64, and the
     scale is s_j = fp32(pow(fp64(max(a_j, act_floor)), alpha_k)); no
     normalisation of s (it cannot change the result, see the scale-invariance
     pin in the tests).
  R3 asymmetric quantiser (never printed on the pages): range [min(w,0),
     max(w,0)], step = fp16(range/15), zero = clamp(rint(-min/step), 0, 15),
     code = clamp(rint(w/step) + zero, 0, 15).
  R4 symmetric quantiser ([concept] 量化数学基础, [aiqz] section 4):
     step = fp16(max|w| / 7), code = clamp(rint(w/step), -7, 7), stored as
     nibble code+8 with zero 8.
  R5 both quantisers use the fp16-rounded step for the codes, so the stored
     scale reproduces them ([adr] 关键设计 3: search and pack share one
     quantiser).
  R6 a step of 0 gives codes 0 (zero point 0) and dequantised value 0; a step
     that overflows fp16 is an error.  A subnormal fp16 step can round well
     below range/15 (or max/7); the codes of R3 / R4 are then decided by
     their clamps (a zero clamped at 15, symmetric codes at +-7).
  R7 loss is the plain sum of squares ||X S^-1 W'hat - X W||^2 (no mean),
     evaluated in the equivalent difference form X (S^-1 W'hat - W).
  R8 argmin takes the first index on ties.
  R9 packing: two codes per byte, the even input row in the low nibble.

Parity unpinned: the exact constants of the asymmetric quantiser (R3) are not
printed on any page; they are pinned only by the brute-force nearest-code
check and the error-bound / invariance tests, not by a worked example.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


class OracleRangeError(ArithmeticError):
    """A quantisation step does not fit in fp16."""


class OracleNonFiniteError(ArithmeticError):
    """An input holds NaN or infinity."""


# ---------------------------------------------------------------------------
# Step 1: per-input-channel activation statistic
# [concept] 技术原理 - 重要通道识别的统计依据 (activation_scale = mean |X[:, j]|);
# [aiqz] section 1, importance I_i = E[|X_i|].
# ---------------------------------------------------------------------------
def act_stats(X: np.ndarray) -> np.ndarray:
    """a_j = (1/N) * sum_r |x_rj|, summed in float64, returned as float32."""
    X = np.asarray(X)
    N = X.shape[0]
    if N == 0:
        raise ValueError("act_stats needs at least one calibration row")
    X64 = X.astype(np.float64)
    if not np.all(np.isfinite(X64)):
        raise OracleNonFiniteError("X holds non-finite values")
    total = np.abs(X64).sum(axis=0)
    return (total / N).astype(F32)


def act_stats_max(X: np.ndarray) -> np.ndarray:
    """The alternative statistic a_j = max_r |x_rj| ([concept] 二、缩放因子的搜索:
    s_j = (max |X_j|)^alpha; 重要通道识别的统计依据: "或 max").  Exact."""
    X = np.asarray(X)
    if X.shape[0] == 0:
        raise ValueError("act_stats_max needs at least one calibration row")
    X64 = X.astype(np.float64)
    if not np.all(np.isfinite(X64)):
        raise OracleNonFiniteError("X holds non-finite values")
    return np.abs(X64).max(axis=0).astype(F32)


def act_stats_stream(batches) -> np.ndarray:
    """The mean |x| accumulated batch by batch ([adr] Decision, Layer 2:
    AWQQuantizer.add_batch accumulates the per-channel mean-abs activation):
    each batch's column sums of |x| in float64 are added to a running float64
    total in batch order, and the total is divided once by the number of rows
    seen."""
    total = None
    rows = 0
    for X in batches:
        X64 = np.asarray(X).astype(np.float64)
        if not np.all(np.isfinite(X64)):
            raise OracleNonFiniteError("X holds non-finite values")
        part = np.abs(X64).sum(axis=0)
        total = part if total is None else total + part
        rows += X64.shape[0]
    if rows == 0:
        raise ValueError("act_stats_stream needs at least one calibration row")
    return (total / rows).astype(F32)


# ---------------------------------------------------------------------------
# Step 2a: candidate scale family
# [concept] 缩放因子优化的完整流程 step 3: s_j(alpha) = activation_scale[j]^alpha,
# alpha in {0, 0.05, ..., 1.0}.
# ---------------------------------------------------------------------------
def alpha_grid(G: int = 21) -> np.ndarray:
    """alpha_k = k / (G - 1) for k = 0..G-1 (float64)."""
    if G == 1:
        return np.zeros(1, dtype=np.float64)
    return np.array([k / (G - 1) for k in range(G)], dtype=np.float64)


def scales(mean_abs: np.ndarray, alpha: float, act_floor: float = 1e-4) -> np.ndarray:
    """s_j = fp32(pow(fp64(max(a_j, floor)), alpha))."""
    a = np.maximum(np.asarray(mean_abs, dtype=F32), F32(act_floor))
    return np.power(a.astype(np.float64), np.float64(alpha)).astype(F32)


def closed_form_scales(W: np.ndarray, mean_abs: np.ndarray, alpha: float = 0.5,
                       act_floor: float = 1e-4) -> np.ndarray:
    """The closed-form scale of [aiqz] section 3: s_i = (E|X_i|)^alpha / mean_j |W_ij|,
    one value per input channel i (row i of W [D_in, D_out]), alpha = 0.5 by
    default.  Readings: E|X_i| is the floored statistic as for the grid
    search; mean_j |W_ij| is summed in float64; the quotient is formed in
    float64 and rounded once to float32; a row of zeros gets s = 1 (its
    weights quantise to zero whatever s is)."""
    W64 = np.asarray(W, dtype=F32).astype(np.float64)
    den = np.abs(W64).sum(axis=1) / W64.shape[1]
    stat = np.maximum(np.asarray(mean_abs, dtype=np.float32), np.float32(act_floor))   # floored as in scales()
    num = np.power(stat.astype(np.float64), np.float64(alpha))
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.where(den > 0, num / np.where(den > 0, den, 1.0), 1.0)
    return s.astype(F32)


# ---------------------------------------------------------------------------
# Step 2b: per-group b-bit quantisation of W' = diag(s) W
# [concept] 技术原理 - 量化数学基础 (absmax step, round, clamp, dequant);
# [aiqz] section 4 (Delta = max|w_s| / (2^(N-1) - 1), round, clamp);
# asymmetric with zero point: reading R3 above.
# ---------------------------------------------------------------------------
def _f16_step(x: np.ndarray) -> np.ndarray:
    """Round a float32 step to fp16 (nearest even) and widen it back."""
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    if not np.all(np.isfinite(h)):
        raise OracleRangeError("quantisation step overflows fp16")
    return h.astype(F32)


def quantize_groups(Wp: np.ndarray, group_size: int, symmetric: bool, bits: int = 4):
    """Quantise W' [D_in, D_out] (float32) in groups of `group_size` rows.

    Returns (codes, step, zero):
      codes uint8 [D_in, D_out]   stored nibble (symmetric: q + 2^(b-1))
      step  float32 [T, D_out]    fp16-representable step per (group, column)
      zero  float32 [T, D_out]    zero point per (group, column)
    Dequantisation is (code - zero) * step for both quantisers.
    """
    Wp = np.asarray(Wp, dtype=F32)
    D_in, D_out = Wp.shape
    g = group_size
    if D_in % g:
        raise ValueError("D_in must be a multiple of group_size")
    if not np.all(np.isfinite(Wp)):
        raise OracleNonFiniteError("scaled weights hold non-finite values")
    Wg = Wp.reshape(D_in // g, g, D_out)
    if symmetric:
        qmax = 2 ** (bits - 1) - 1
        amax = np.abs(Wg).max(axis=1)                       # [T, D_out]
        step = _f16_step(amax / F32(qmax))
        zero = np.zeros_like(step)
        ok = step > 0
        stepb = np.where(ok, step, F32(1))[:, None, :]
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.rint(Wg / stepb)
        q = np.clip(q, -qmax, qmax)
        q = np.where(ok[:, None, :], q, F32(0))
        codes = (q + 2 ** (bits - 1)).astype(np.uint8)
        zero = np.full_like(step, F32(2 ** (bits - 1)))
    else:
        qmax = 2 ** bits - 1
        mn = np.minimum(Wg.min(axis=1), F32(0))
        mx = np.maximum(Wg.max(axis=1), F32(0))
        step = _f16_step((mx - mn) / F32(qmax))
        ok = step > 0
        stepb = np.where(ok, step, F32(1))
        zero = np.clip(np.rint(-mn / stepb), 0, qmax).astype(F32)
        zero = np.where(ok, zero, F32(0)) + F32(0)   # an integer code: -0 becomes +0
        q = np.rint(Wg / stepb[:, None, :]) + zero[:, None, :]
        q = np.clip(q, 0, qmax)
        q = np.where(ok[:, None, :], q, F32(0))
        codes = q.astype(np.uint8)
    return codes.reshape(D_in, D_out), step, zero


def dequantize(codes: np.ndarray, step: np.ndarray, zero: np.ndarray, group_size: int) -> np.ndarray:
    """W'hat = (code - zero) * step, float32 (exact: small integer times fp16 value)."""
    D_in, D_out = codes.shape
    c = codes.astype(F32).reshape(D_in // group_size, group_size, D_out)
    return ((c - zero[:, None, :]) * step[:, None, :]).reshape(D_in, D_out)


# ---------------------------------------------------------------------------
# Step 2c: loss L(alpha) = ||X S^-1 W'hat - X W||^2
# [concept] 缩放因子优化的完整流程 step 4c; 技术原理 (Delta Y = X S^-1 eps_SW).
# ---------------------------------------------------------------------------
def candidate_delta(W: np.ndarray, s: np.ndarray, group_size: int, symmetric: bool,
                    bits: int = 4) -> np.ndarray:
    """S^-1 W'hat - W in float64 for one scale vector s [D_in]."""
    W = np.asarray(W, dtype=F32)
    Wp = W * s[:, None]                                  # W' = diag(s) W, fp32
    codes, step, zero = quantize_groups(Wp, group_size, symmetric, bits)
    What = dequantize(codes, step, zero, group_size)     # W'hat, fp32
    return What.astype(np.float64) / s.astype(np.float64)[:, None] - W.astype(np.float64)


def column_losses(X: np.ndarray, delta: np.ndarray) -> np.ndarray:
    """Per output column n: sum_r (sum_j x_rj delta_jn)^2, float64."""
    E = np.asarray(X, dtype=np.float64) @ delta
    return (E * E).sum(axis=0)


def search(X, W, mean_abs, grid=None, group_size=128, symmetric=False, bits=4,
           act_floor=1e-4, cols=None):
    """The alpha-grid scale search.

    [concept] 缩放因子优化的完整流程 steps 3-6; [glossary] 4.3 grid-search
    pseudocode.  `cols` restricts the loss to a subset of output columns (the
    loss is a sum over columns, so a subset gives that subset's share).

    Returns dict with losses [G] (float64), best (first argmin), alpha_star,
    s_star (float32 [D_in]) and col_losses [G, len(cols)] (float64).
    """
    W = np.asarray(W, dtype=F32)
    if grid is None:
        grid = alpha_grid(21)
    grid = np.asarray(grid, dtype=np.float64)
    if cols is not None:
        W = W[:, np.asarray(cols)]
    X64 = np.asarray(X, dtype=np.float64)
    G = len(grid)
    col = np.zeros((G, W.shape[1]), dtype=np.float64)
    svecs = []
    for k in range(G):
        s = scales(mean_abs, grid[k], act_floor)
        svecs.append(s)
        col[k] = column_losses(X64, candidate_delta(W, s, group_size, symmetric, bits))
    losses = col.sum(axis=1)
    best = int(np.argmin(losses))              # first index on ties
    return {"losses": losses, "best": best, "alpha_star": float(grid[best]),
            "s_star": svecs[best], "col_losses": col}


# ---------------------------------------------------------------------------
# The ADR's second search: per-group coordinate greedy over power-of-two
# channel scales.  [adr] 关键设计 1: groups are independent along the input
# dimension; within a group, each input channel in turn tries every grid
# candidate (20 powers of two centred on 1), the whole group's
# activation-weighted reconstruction error is evaluated with the pack's own
# quantiser, and the best candidate is kept; 3 passes let a channel react to
# a group maximum that a later channel enlarged.  [adr] 关键设计 2-3: the
# error is measured in the original space (w'hat / s - w), with the exact
# quantiser of the pack.
# Readings (the ADR gives no formula): candidates 2^k, k = -10 .. 9; initial
# s = 1; weight of channel j = its mean |x| (a_j, not squared); a candidate
# replaces the current value only when strictly better, and among equally
# good candidates the first in k order wins; channels in index order.
# ---------------------------------------------------------------------------
def greedy_candidates(count: int = 20, k_min: int = -10) -> np.ndarray:
    """The power-of-two grid 2^k, k = k_min .. k_min + count - 1 (float32, exact)."""
    return np.array([2.0 ** k for k in range(k_min, k_min + count)], dtype=F32)


def group_error(Wg: np.ndarray, s: np.ndarray, a: np.ndarray, symmetric: bool, bits: int = 4) -> float:
    """sum_j a_j sum_n (w'hat_jn / s_j - w_jn)^2 for one group Wg [g, D_out] (float64 sum)."""
    Wg = np.asarray(Wg, dtype=F32)
    s = np.asarray(s, dtype=F32)
    g = Wg.shape[0]
    codes, step, zero = quantize_groups(Wg * s[:, None], g, symmetric, bits)
    What = dequantize(codes, step, zero, g)
    D = What.astype(np.float64) / s.astype(np.float64)[:, None] - Wg.astype(np.float64)
    return float((np.asarray(a, dtype=np.float64)[:, None] * D * D).sum())


def greedy_search(W, mean_abs, group_size=128, symmetric=False, passes=3, candidates=None, follow=None):
    """Per-group coordinate greedy of [adr] 关键设计 1.

    Returns (s float32 [D_in], trace int [passes, D_in] of chosen candidate
    indices, errors float64 [passes, D_in, len(candidates)] of every
    evaluated candidate).  `follow`, if given ([passes, D_in] candidate
    indices), replaces each decision by the given one (used to replay another
    implementation's choices and weigh each against these errors).
    """
    W = np.asarray(W, dtype=F32)
    a = np.asarray(mean_abs, dtype=np.float64)
    if candidates is None:
        candidates = greedy_candidates()
    cand = np.asarray(candidates, dtype=F32)
    D_in = W.shape[0]
    s = np.ones(D_in, dtype=F32)
    one = int(np.flatnonzero(cand == F32(1.0))[0])
    cur = np.full(D_in, one, dtype=np.int64)
    trace = np.zeros((passes, D_in), dtype=np.int64)
    errors = np.zeros((passes, D_in, len(cand)), dtype=np.float64)
    for t in range(D_in // group_size):
        rows = slice(t * group_size, (t + 1) * group_size)
        Wg, ag = W[rows], a[rows]
        for p in range(passes):
            for jj in range(group_size):
                j = t * group_size + jj
                sg = s[rows].copy()
                for c in range(len(cand)):
                    sg[jj] = cand[c]
                    errors[p, j, c] = group_error(Wg, sg, ag, symmetric)
                e = errors[p, j]
                best = cur[j]
                for c in range(len(cand)):           # strictly better; the first in k order among equals
                    if e[c] < e[best]:
                        best = c
                if follow is not None:
                    best = int(follow[p, j])
                trace[p, j] = best
                cur[j] = best
                s[j] = cand[best]
    return s, trace, errors


# ---------------------------------------------------------------------------
# Step 4: offline pack of Quantize(diag(s*) W)
# [concept] 推理时的等效实现 (W_quantized = Quantize(diag(s*) W), s* kept as
# metadata); [adr] Consequences (two 4-bit weights per byte).
# ---------------------------------------------------------------------------
def pack(W, s, group_size=128, symmetric=False, bits=4):
    """Return (qweight uint8 [D_in/2, D_out], scales fp16 [T, D_out], zeros fp16 [T, D_out])."""
    if bits != 4:
        raise ValueError("only 4-bit packing is defined")
    W = np.asarray(W, dtype=F32)
    s = np.asarray(s, dtype=F32)
    codes, step, zero = quantize_groups(W * s[:, None], group_size, symmetric, bits)
    lo = codes[0::2].astype(np.uint8)
    hi = codes[1::2].astype(np.uint8)
    qweight = (lo | (hi << 4)).astype(np.uint8)
    return qweight, step.astype(np.float16), zero.astype(np.float16)


def unpack_codes(qweight: np.ndarray) -> np.ndarray:
    """Inverse of the nibble layout of `pack`: codes [D_in, D_out]."""
    q = np.asarray(qweight, dtype=np.uint8)
    out = np.empty((q.shape[0] * 2, q.shape[1]), dtype=np.uint8)
    out[0::2] = q & 0xF
    out[1::2] = q >> 4
    return out


# ---------------------------------------------------------------------------
# After the path: the W4A16 inference product on the packed layer.
# [concept] 推理时的等效实现: offline W_quantized = Quantize(diag(s*) W) with
# s* kept as metadata; online Y = (X diag(1/s*)) Dequant(W_quantized), the
# 1/s* scaling optionally folded into the kernel's dequantisation
# (ASCII 架构图: "Dequant + MatMul (融合 s* 缩放)").  Dequant is the
# quantiser's inverse, (code - zero) * scale per group (量化数学基础 step 3).
# ---------------------------------------------------------------------------
def w4a16_matmul(X, qweight, scales, zeros, s, group_size=128):
    """Y = (X diag(1/s)) Dequant(qweight) in float64.

    X [M, D_in] (any float type, taken exactly), qweight uint8 [D_in/2, D_out]
    in the pack layout, scales / zeros fp16 [D_in/group_size, D_out], s fp32
    [D_in] (None: no scaling).  Returns float64 [M, D_out].
    """
    codes = unpack_codes(qweight).astype(np.float64)             # [D_in, D_out]
    D_in, D_out = codes.shape
    g = np.arange(D_in) // group_size                            # group of each input row
    Wq = (codes - np.asarray(zeros, dtype=np.float64)[g, :]) * np.asarray(scales, dtype=np.float64)[g, :]
    X64 = np.asarray(X, dtype=np.float64)
    if s is not None:
        X64 = X64 / np.asarray(s, dtype=np.float64)[None, :]     # X diag(1/s), elementwise
    return X64 @ Wq


# ---------------------------------------------------------------------------
# Diagnostic: relative activation-weighted error, [aiqz] section 5
# epsilon = E||X (W - W_hat)||^2 / E||X W||^2.
# ---------------------------------------------------------------------------
def relative_error(X, W, loss: float) -> float:
    Y = np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64)
    return float(loss / (Y * Y).sum())
