"""Plant plausible mistakes in copies of the oracle (CPU only) and check that
the pins catch every one of them."""
import importlib.util
import os

import pytest

import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "awq_oracle.py")

# (name, exact source text, replacement).  Clamping symmetric codes to [-8, 7]
# instead of [-7, 7] is not listed: with step = max|w|/7 the code -8 is never
# reached (|w|/step <= 7 * (1 + 2^-11) < 7.5), so that change is equivalent.
MUTANTS = [
    ("stat_max_not_mean", "total = np.abs(X64).sum(axis=0)\n    return (total / N)",
     "total = np.abs(X64).max(axis=0)\n    return (total / 1)"),
    ("stat_divides_by_N_minus_1", "return (total / N)", "return (total / max(N - 1, 1))"),
    ("stat_no_abs", "total = np.abs(X64).sum(axis=0)", "total = X64.sum(axis=0)"),
    ("floor_ignored", "a = np.maximum(np.asarray(mean_abs, dtype=F32), F32(act_floor))",
     "a = np.asarray(mean_abs, dtype=F32)"),
    ("sym_divides_by_8", "qmax = 2 ** (bits - 1) - 1", "qmax = 2 ** (bits - 1)"),
    ("asym_divides_by_16", "qmax = 2 ** bits - 1", "qmax = 2 ** bits"),
    ("zero_sign_flipped", "zero = np.clip(np.rint(-mn / stepb), 0, qmax)", "zero = np.clip(np.rint(mn / stepb), 0, qmax)"),
    ("floor_rounding_sym", "q = np.rint(Wg / stepb)", "q = np.floor(Wg / stepb)"),
    ("half_away_rounding_asym", "q = np.rint(Wg / stepb[:, None, :]) + zero[:, None, :]",
     "q = np.sign(Wg / stepb[:, None, :]) * np.floor(np.abs(Wg / stepb[:, None, :]) + 0.5) + zero[:, None, :]"),
    ("step_not_fp16", "h = x.astype(np.float16)", "h = x.astype(np.float32)"),
    ("range_excludes_zero", "mn = np.minimum(Wg.min(axis=1), F32(0))", "mn = Wg.min(axis=1)"),
    ("dequant_drops_zero", "return ((c - zero[:, None, :]) * step[:, None, :])", "return ((c) * step[:, None, :])"),
    ("loss_forgets_inverse_scale", "return What.astype(np.float64) / s.astype(np.float64)[:, None] - W.astype(np.float64)",
     "return What.astype(np.float64) - W.astype(np.float64)"),
    ("scales_columns_not_rows", "Wp = W * s[:, None]                                  # W' = diag(s) W, fp32",
     "Wp = W * s[None, :]"),
    ("loss_abs_not_square", "return (E * E).sum(axis=0)", "return np.abs(E).sum(axis=0)"),
    ("argmax_not_argmin", "best = int(np.argmin(losses))", "best = int(np.argmax(losses))"),
    ("nibbles_swapped", "qweight = (lo | (hi << 4)).astype(np.uint8)", "qweight = (hi | (lo << 4)).astype(np.uint8)"),
    ("w4a16_nibbles_swapped", "codes = unpack_codes(qweight).astype(np.float64)             # [D_in, D_out]",
     "codes = unpack_codes(((qweight >> 4) | (qweight << 4)).astype(np.uint8)).astype(np.float64)"),
    ("w4a16_drops_zero", "Wq = (codes - np.asarray(zeros, dtype=np.float64)[g, :])", "Wq = (codes - 0 * np.asarray(zeros, dtype=np.float64)[g, :])"),
    ("w4a16_scales_not_divides", "X64 = X64 / np.asarray(s, dtype=np.float64)[None, :]", "X64 = X64 * np.asarray(s, dtype=np.float64)[None, :]"),
    ("w4a16_group_index_mod", "g = np.arange(D_in) // group_size", "g = np.arange(D_in) % (D_in // group_size)"),
    ("w4a16_group_of_pairs", "g = np.arange(D_in) // group_size", "g = (np.arange(D_in) // 2) // group_size"),
    ("max_stat_no_abs", "return np.abs(X64).max(axis=0).astype(F32)", "return X64.max(axis=0).astype(F32)"),
    ("stream_mean_of_batch_means", "total = part if total is None else total + part\n        rows += X64.shape[0]",
     "part = part / X64.shape[0]\n        total = part if total is None else total + part\n        rows += 1"),
    ("greedy_weight_squared", "return float((np.asarray(a, dtype=np.float64)[:, None] * D * D).sum())",
     "return float((np.asarray(a, dtype=np.float64)[:, None] ** 2 * D * D).sum())"),
    ("greedy_error_in_scaled_space", "D = What.astype(np.float64) / s.astype(np.float64)[:, None] - Wg.astype(np.float64)",
     "D = What.astype(np.float64) - (Wg * s[:, None]).astype(np.float64)"),
    ("greedy_keeps_last_of_equals", "if e[c] < e[best]:", "if e[c] <= e[best]:"),
    ("greedy_grid_off_by_one", "return np.array([2.0 ** k for k in range(k_min, k_min + count)], dtype=F32)",
     "return np.array([2.0 ** k for k in range(k_min + 1, k_min + count + 1)], dtype=F32)"),
    ("closed_form_mean_over_rows", "den = np.abs(W64).sum(axis=1) / W64.shape[1]",
     "den = np.abs(W64).sum(axis=0)[: W64.shape[0]] / W64.shape[0]"),
    ("closed_form_no_abs", "den = np.abs(W64).sum(axis=1) / W64.shape[1]", "den = np.abs(W64.sum(axis=1)) / W64.shape[1]"),
    ("closed_form_alpha_on_both", "s = np.where(den > 0, num / np.where(den > 0, den, 1.0), 1.0)",
     "s = np.where(den > 0, num / np.power(np.where(den > 0, den, 1.0), alpha), 1.0)"),
    ("asym_no_lower_clamp", "q = np.clip(q, 0, qmax)", "q = np.minimum(q, qmax)"),
    ("sym_no_clamp", "q = np.clip(q, -qmax, qmax)", "q = q"),
    ("alpha_scaled_twice", "return np.power(a.astype(np.float64), np.float64(alpha)).astype(F32)",
     "return np.power(a.astype(np.float64), np.float64(2 * alpha)).astype(F32)"),
    ("epsilon_over_weight_energy", "return float(loss / (Y * Y).sum())",
     "return float(loss / (np.asarray(W, dtype=np.float64) ** 2).sum())"),
    ("epsilon_transposed_weight", "Y = np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64)",
     "Y = np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T"),
    ("epsilon_not_squared", "return float(loss / (Y * Y).sum())", "return float(loss / np.abs(Y).sum())"),
]


def _load_mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = src.replace(old, new)
    spec = importlib.util.spec_from_loader(f"awq_oracle_{name}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    mod = _load_mutant(name, old, new)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception:   # an assertion or a crash both count as caught
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {name}"
