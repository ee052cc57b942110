"""B300 (sm_103a) AWQ calibration hot path: a thin ctypes binding over
``libawq_b300.so``.

The functions here only marshal torch tensors into the C ABI declared in
``include/awq.h`` (pointers, sizes, the current CUDA stream); every step of
the path runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing or the device is not sm_103 the calls raise.

    a = act_stats(X)                                  # mean |X[:, j]|
    r = search(X, W, a)                               # alpha grid search
    qweight, scales, zeros = quantize_pack(W, r.s_star)
    qweight, scales, zeros = quantize_pack_searched(W, r)   # same, reusing the search's parameters
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libawq_b300.so")

AWQ_STATUS = {
    0: "AWQ_OK", 1: "AWQ_ERR_INVALID_ARG", 2: "AWQ_ERR_SHAPE", 3: "AWQ_ERR_ALIGNMENT",
    4: "AWQ_ERR_WORKSPACE", 5: "AWQ_ERR_UNSUPPORTED_DEVICE", 6: "AWQ_ERR_CUDA",
    7: "AWQ_ERR_RANGE", 8: "AWQ_ERR_NONFINITE", 9: "AWQ_ERR_TIMEOUT",
}


class AwqError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = AWQ_STATUS.get(code, f"status {code}")
        super().__init__(f"{where}: {self.name}")


class awq_cfg(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("symmetric", ctypes.c_int32), ("act_floor", ctypes.c_float)]


class awq_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


_c_i64, _c_i32, _c_sz, _vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p

_SIGS = {
    "awq_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "awq_workspace_status": ([_vp, _vp], ctypes.c_int),
    "awq_act_stats_workspace_size": ([_c_i64, _c_i64, ctypes.POINTER(_c_sz)], ctypes.c_int),
    "awq_act_stats": ([_vp, _c_i64, _c_i64, _c_i64, _vp, _vp, _c_sz, _vp], ctypes.c_int),
    "awq_act_stats_accumulate": ([_vp, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp, _c_sz, _vp], ctypes.c_int),
    "awq_act_stats_finalize": ([_vp, _c_i64, _c_i64, _vp, _vp], ctypes.c_int),
    "awq_search_workspace_size": ([_c_i64, _c_i64, _c_i64, _c_i32, ctypes.POINTER(awq_cfg),
                                   ctypes.POINTER(_c_sz)], ctypes.c_int),
    "awq_search": ([_vp, _vp, _c_i64, _c_i64, _c_i64, _vp, ctypes.POINTER(ctypes.c_double), _c_i32,
                    ctypes.POINTER(awq_cfg), _vp, _vp, _vp, _vp, _vp, _c_sz, _vp], ctypes.c_int),
    "awq_search_gram_workspace_size": ([_c_i64, _c_i64, _c_i64, _c_i32, ctypes.POINTER(awq_cfg),
                                        ctypes.POINTER(_c_sz)], ctypes.c_int),
    "awq_search_gram": ([_vp, _vp, _c_i64, _c_i64, _c_i64, _vp, ctypes.POINTER(ctypes.c_double), _c_i32,
                         ctypes.POINTER(awq_cfg), _vp, _vp, _vp, _vp, _vp, _c_sz, _vp], ctypes.c_int),
    "awq_pack_workspace_size": ([_c_i64, _c_i64, ctypes.POINTER(awq_cfg), ctypes.POINTER(_c_sz)], ctypes.c_int),
    "awq_quantize_pack": ([_vp, _vp, _c_i64, _c_i64, ctypes.POINTER(awq_cfg), _vp, _vp, _vp, _vp, _c_sz, _vp],
                          ctypes.c_int),
    "awq_quantize_pack_searched": ([_vp, _c_i64, _c_i64, _c_i32, ctypes.POINTER(awq_cfg), _vp, _c_sz, _vp, _vp,
                                    _vp, _vp, _vp, _vp], ctypes.c_int),
    "awq_closed_form_scales": ([_vp, _c_i64, _c_i64, _vp, ctypes.c_double, ctypes.POINTER(awq_cfg), _vp, _vp],
                               ctypes.c_int),
    "awq_greedy_workspace_size": ([_c_i64, _c_i64, ctypes.POINTER(awq_cfg), ctypes.POINTER(_c_sz)], ctypes.c_int),
    "awq_greedy_search": ([_vp, _vp, _c_i64, _c_i64, ctypes.POINTER(awq_cfg), _c_i32, _c_i32, _c_i32, _vp, _vp, _vp,
                           _vp, _c_sz, _vp], ctypes.c_int),
    "awq_w4a16_workspace_size": ([_c_i64, _c_i64, _c_i64, ctypes.POINTER(_c_sz)], ctypes.c_int),
    "awq_w4a16_matmul": ([_vp, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp, _vp, ctypes.POINTER(awq_cfg), _vp, _vp, _c_sz,
                          _vp], ctypes.c_int),
    "awq_search_block_losses": ([_vp, _c_sz, _c_i64, _c_i64, _c_i64, _c_i32, ctypes.POINTER(awq_cfg), _vp, _vp],
                                ctypes.c_int),
    "awq_search_select": ([_vp, _c_i64, _c_i32, _vp, _c_sz, _c_i64, _c_i64, _c_i64, ctypes.POINTER(awq_cfg), _vp,
                          _vp, _vp, _vp], ctypes.c_int),
    "awq_selftest_gemm_bf16": ([_vp, _vp, _c_i32, _c_i64, _c_i64, _c_i64, _vp, _vp, _c_sz, _vp], ctypes.c_int),
    "awq_selftest_wait_timeout": ([ctypes.c_uint64, _c_i32, _vp, _vp, _c_sz, _vp], ctypes.c_int),
    "awq_profile_enable": ([_c_i32], ctypes.c_int),
    "awq_profile_collect": ([ctypes.POINTER(awq_kernel_time), _c_i32, ctypes.POINTER(_c_i32)], ctypes.c_int),
}

_lib = None


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m post_weight_quantization_column_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise AwqError(code, where)


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_cfg(group_size=128, symmetric=False, bits=4, act_floor=1e-4) -> awq_cfg:
    return awq_cfg(int(bits), int(group_size), 1 if symmetric else 0, float(act_floor))


def default_grid(G: int = 21):
    """alpha_k = k / (G - 1), the pages' {0, 0.05, ..., 1.0} for G = 21."""
    if G == 1:
        return [0.0]
    return [k / (G - 1) for k in range(G)]


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device status word of `ws`."""
    return lib().awq_workspace_status(_ptr(ws), _stream_handle(stream))


def _alloc_ws(nbytes: int, device) -> torch.Tensor:
    # 256-byte aligned by the caching allocator
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def check_workspace(ws: torch.Tensor, where: str, stream=None):
    _check(workspace_status(ws, stream), where)


# ---------------------------------------------------------------------- step 1
def act_stats_workspace_size(N: int, D_in: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().awq_act_stats_workspace_size(N, D_in, ctypes.byref(n)), "awq_act_stats_workspace_size")
    return n.value


def act_stats(X: torch.Tensor, out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
              stream=None, check: bool = True) -> torch.Tensor:
    """mean_r |X[r, j]| for X bf16 [N, D_in] on the GPU -> fp32 [D_in]."""
    _need(X, torch.bfloat16, "X")
    N, D = X.shape
    if out is None:
        out = torch.empty(D, dtype=torch.float32, device=X.device)
    if ws is None:
        ws = _alloc_ws(act_stats_workspace_size(N, D), X.device)
    st = _stream_handle(stream)
    _check(lib().awq_act_stats(_ptr(X), N, D, D, _ptr(out), _ptr(ws), ws.numel(), st), "awq_act_stats")
    if check:
        check_workspace(ws, "awq_act_stats (device)", stream)
    return out


class StatsAccumulator:
    """The statistic over a stream of calibration batches (the ADR's add_batch):
    float64 running column sums of |x| and, optionally, the running max |x|."""

    def __init__(self, D_in: int, device, track_max: bool = False):
        self.D_in = D_in
        self.rows = 0
        self.sum_abs = torch.zeros(D_in, dtype=torch.float64, device=device)
        self.max_abs = torch.zeros(D_in, dtype=torch.float32, device=device) if track_max else None
        self._ws = None

    def add_batch(self, X: torch.Tensor, stream=None, check: bool = True):
        _need(X, torch.bfloat16, "X")
        N, D = X.shape
        if D != self.D_in:
            raise ValueError("batch has the wrong number of channels")
        need = act_stats_workspace_size(N, D)
        if self._ws is None or self._ws.numel() < need:
            self._ws = _alloc_ws(need, X.device)
        _check(lib().awq_act_stats_accumulate(_ptr(X), N, D, D, _ptr(self.sum_abs), _ptr(self.max_abs),
                                              _ptr(self._ws), self._ws.numel(), _stream_handle(stream)),
               "awq_act_stats_accumulate")
        if check:
            check_workspace(self._ws, "awq_act_stats_accumulate (device)", stream)
        self.rows += N
        return self

    def mean(self, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(self.D_in, dtype=torch.float32, device=self.sum_abs.device)
        _check(lib().awq_act_stats_finalize(_ptr(self.sum_abs), self.rows, self.D_in, _ptr(out),
                                            _stream_handle(stream)), "awq_act_stats_finalize")
        return out


def act_stats_max(X: torch.Tensor, stream=None) -> torch.Tensor:
    """max_r |X[r, j]| for X bf16 [N, D_in] on the GPU -> fp32 [D_in] (exact)."""
    acc = StatsAccumulator(X.shape[1], X.device, track_max=True)
    acc.add_batch(X, stream=stream)
    return acc.max_abs


# ---------------------------------------------------------------------- steps 2-3
@dataclass
class SearchResult:
    losses: torch.Tensor        # fp64 [G]
    best_idx: torch.Tensor      # int32 [1]
    s_star: torch.Tensor        # fp32 [D_in]
    col_losses: Optional[torch.Tensor]  # fp64 [G, D_out] or None
    grid: list
    workspace: torch.Tensor
    # the call that filled it (set by search(); used by the column-sharded form)
    shape: tuple = ()           # (N, D_in, D_out)
    cfg: tuple = ()             # (group_size, symmetric, act_floor)
    gram: bool = False

    @property
    def best(self) -> int:
        return int(self.best_idx.item())

    @property
    def alpha_star(self) -> float:
        return float(self.grid[self.best])


def search_workspace_size(N, D_in, D_out, G=21, group_size=128, symmetric=False, act_floor=1e-4) -> int:
    cfg = make_cfg(group_size, symmetric, 4, act_floor)
    n = ctypes.c_size_t(0)
    _check(lib().awq_search_workspace_size(N, D_in, D_out, G, ctypes.byref(cfg), ctypes.byref(n)),
           "awq_search_workspace_size")
    return n.value


def search_gram_workspace_size(N, D_in, D_out, G=21, group_size=128, symmetric=False, act_floor=1e-4) -> int:
    cfg = make_cfg(group_size, symmetric, 4, act_floor)
    n = ctypes.c_size_t(0)
    _check(lib().awq_search_gram_workspace_size(N, D_in, D_out, G, ctypes.byref(cfg), ctypes.byref(n)),
           "awq_search_gram_workspace_size")
    return n.value


def search(X: torch.Tensor, W: torch.Tensor, mean_abs: torch.Tensor, grid=None, group_size: int = 128,
           symmetric: bool = False, act_floor: float = 1e-4, col_losses: bool = False,
           ws: Optional[torch.Tensor] = None, out: Optional[SearchResult] = None, stream=None,
           check: bool = True, gram: bool = False) -> SearchResult:
    """The alpha-grid scale search over X bf16 [N, D_in], W bf16 [D_in, D_out].

    gram=True evaluates the same losses through the Gram factor of X (N >= D_in): cheaper when N > D_in."""
    _need(X, torch.bfloat16, "X")
    _need(W, torch.bfloat16, "W")
    _need(mean_abs, torch.float32, "mean_abs")
    N, D_in = X.shape
    D_in2, D_out = W.shape
    if D_in2 != D_in or mean_abs.numel() != D_in:
        raise ValueError("shape mismatch between X, W and mean_abs")
    grid = list(default_grid() if grid is None else grid)
    G = len(grid)
    cfg = make_cfg(group_size, symmetric, 4, act_floor)
    dev = X.device
    if ws is None:
        size_fn = search_gram_workspace_size if gram else search_workspace_size
        ws = _alloc_ws(size_fn(N, D_in, D_out, G, group_size, symmetric, act_floor), dev)
    if out is None:
        out = SearchResult(torch.empty(G, dtype=torch.float64, device=dev),
                           torch.empty(1, dtype=torch.int32, device=dev),
                           torch.empty(D_in, dtype=torch.float32, device=dev),
                           torch.empty(G, D_out, dtype=torch.float64, device=dev) if col_losses else None,
                           grid, ws)
    garr = (ctypes.c_double * G)(*grid)
    fn = lib().awq_search_gram if gram else lib().awq_search
    name = "awq_search_gram" if gram else "awq_search"
    _check(fn(_ptr(X), _ptr(W), N, D_in, D_out, _ptr(mean_abs), garr, G, ctypes.byref(cfg), _ptr(out.losses),
              _ptr(out.best_idx), _ptr(out.s_star), _ptr(out.col_losses), _ptr(ws), ws.numel(),
              _stream_handle(stream)), name)
    if check:
        check_workspace(ws, f"{name} (device)", stream)
    out.workspace, out.shape, out.cfg, out.gram = ws, (N, D_in, D_out), (group_size, symmetric, act_floor), gram
    return out


def search_block_losses(res: SearchResult, stream=None) -> torch.Tensor:
    """The fp64 block partials [G, ceil(D_out / 256)] of a finished search
    (each the candidate's loss over 256 consecutive output columns)."""
    if res.gram or len(res.shape) != 3:
        raise ValueError("block partials are available from a direct search() result")
    N, D_in, D_out = res.shape
    G = len(res.grid)
    cfg = make_cfg(res.cfg[0], res.cfg[1], 4, res.cfg[2])
    blk = torch.empty(G, (D_out + 255) // 256, dtype=torch.float64, device=res.workspace.device)
    _check(lib().awq_search_block_losses(_ptr(res.workspace), res.workspace.numel(), N, D_in, D_out, G,
                                         ctypes.byref(cfg), _ptr(blk), _stream_handle(stream)),
           "awq_search_block_losses")
    return blk


def search_select(res: SearchResult, blk: torch.Tensor, stream=None, check: bool = True) -> SearchResult:
    """Overwrite res.losses / best_idx / s_star from block partials [G, nb] of
    all column slices (slice order): the global alpha* of a column-sharded
    search, written where awq_quantize_pack_searched reads it."""
    _need(blk, torch.float64, "blk")
    N, D_in, D_out = res.shape
    G = len(res.grid)
    if blk.dim() != 2 or blk.shape[0] != G:
        raise ValueError("blk must be [G, nb]")
    blk = blk.contiguous()
    cfg = make_cfg(res.cfg[0], res.cfg[1], 4, res.cfg[2])
    _check(lib().awq_search_select(_ptr(blk), blk.shape[1], G, _ptr(res.workspace), res.workspace.numel(), N, D_in,
                                   D_out, ctypes.byref(cfg), _ptr(res.losses), _ptr(res.best_idx), _ptr(res.s_star),
                                   _stream_handle(stream)), "awq_search_select")
    if check:
        check_workspace(res.workspace, "awq_search_select (device)", stream)
    return res


# ---------------------------------------------------------------------- step 4
def quantize_pack(W: torch.Tensor, s: torch.Tensor, group_size: int = 128, symmetric: bool = False,
                  out=None, ws: Optional[torch.Tensor] = None, stream=None, check: bool = True):
    """Quantize(diag(s) W) -> (qweight u8 [D_in/2, D_out], scales fp16 [T, D_out], zeros fp16 [T, D_out])."""
    _need(W, torch.bfloat16, "W")
    _need(s, torch.float32, "s")
    D_in, D_out = W.shape
    dev = W.device
    if D_in % group_size:
        raise ValueError("D_in must be a multiple of group_size")
    T = D_in // group_size
    if out is None:
        out = (torch.empty(D_in // 2, D_out, dtype=torch.uint8, device=dev),
               torch.empty(T, D_out, dtype=torch.float16, device=dev),
               torch.empty(T, D_out, dtype=torch.float16, device=dev))
    qweight, scales, zeros = out
    cfg = make_cfg(group_size, symmetric)
    if ws is None:
        n = ctypes.c_size_t(0)
        _check(lib().awq_pack_workspace_size(D_in, D_out, ctypes.byref(cfg), ctypes.byref(n)),
               "awq_pack_workspace_size")
        ws = _alloc_ws(n.value, dev)
    _check(lib().awq_quantize_pack(_ptr(W), _ptr(s), D_in, D_out, ctypes.byref(cfg), _ptr(qweight),
                                   _ptr(scales), _ptr(zeros), _ptr(ws), ws.numel(), _stream_handle(stream)),
           "awq_quantize_pack")
    if check:
        check_workspace(ws, "awq_quantize_pack (device)", stream)
    return qweight, scales, zeros


def quantize_pack_searched(W: torch.Tensor, result: SearchResult, group_size: int = 128, symmetric: bool = False,
                           out=None, stream=None):
    """The pack right after `search`: same outputs as quantize_pack(W, result.s_star), using the group
    parameters the search computed for its best candidate (one streaming pass over W)."""
    _need(W, torch.bfloat16, "W")
    D_in, D_out = W.shape
    dev = W.device
    if D_in % group_size:
        raise ValueError("D_in must be a multiple of group_size")
    T = D_in // group_size
    if out is None:
        out = (torch.empty(D_in // 2, D_out, dtype=torch.uint8, device=dev),
               torch.empty(T, D_out, dtype=torch.float16, device=dev),
               torch.empty(T, D_out, dtype=torch.float16, device=dev))
    qweight, scales, zeros = out
    cfg = make_cfg(group_size, symmetric)
    ws = result.workspace
    _check(lib().awq_quantize_pack_searched(_ptr(W), D_in, D_out, len(result.grid), ctypes.byref(cfg), _ptr(ws),
                                            ws.numel(), _ptr(result.best_idx), _ptr(result.s_star), _ptr(qweight),
                                            _ptr(scales), _ptr(zeros), _stream_handle(stream)),
           "awq_quantize_pack_searched")
    return qweight, scales, zeros


# ---------------------------------------------------------------------- closed-form scale
def closed_form_scales(W: torch.Tensor, mean_abs: torch.Tensor, alpha: float = 0.5, act_floor: float = 1e-4,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """s_i = (max(E|X_i|, floor))^alpha / mean_j |W_ij| -> fp32 [D_in] (a zero row gets 1)."""
    _need(W, torch.bfloat16, "W")
    _need(mean_abs, torch.float32, "mean_abs")
    D_in, D_out = W.shape
    if out is None:
        out = torch.empty(D_in, dtype=torch.float32, device=W.device)
    cfg = make_cfg(act_floor=act_floor)
    _check(lib().awq_closed_form_scales(_ptr(W), D_in, D_out, _ptr(mean_abs), float(alpha), ctypes.byref(cfg),
                                        _ptr(out), _stream_handle(stream)), "awq_closed_form_scales")
    return out


# ---------------------------------------------------------------------- the ADR's greedy search
def greedy_search(W: torch.Tensor, mean_abs: torch.Tensor, group_size: int = 128, symmetric: bool = False,
                  passes: int = 3, k_min: int = -10, n_cand: int = 20, trace: bool = False, errors: bool = False,
                  stream=None, check: bool = True):
    """Per-group coordinate greedy over 2^k channel scales -> s fp32 [D_in] (and, when asked,
    the chosen candidate per step [passes, D_in] and every evaluated error [passes, D_in, n_cand])."""
    _need(W, torch.bfloat16, "W")
    _need(mean_abs, torch.float32, "mean_abs")
    D_in, D_out = W.shape
    dev = W.device
    cfg = make_cfg(group_size, symmetric)
    n = ctypes.c_size_t(0)
    _check(lib().awq_greedy_workspace_size(D_in, D_out, ctypes.byref(cfg), ctypes.byref(n)),
           "awq_greedy_workspace_size")
    ws = _alloc_ws(n.value, dev)
    s = torch.empty(D_in, dtype=torch.float32, device=dev)
    tr = torch.empty(passes, D_in, dtype=torch.int32, device=dev) if trace else None
    er = torch.empty(passes, D_in, n_cand, dtype=torch.float64, device=dev) if errors else None
    _check(lib().awq_greedy_search(_ptr(W), _ptr(mean_abs), D_in, D_out, ctypes.byref(cfg), passes, k_min, n_cand,
                                   _ptr(s), _ptr(tr), _ptr(er), _ptr(ws), ws.numel(), _stream_handle(stream)),
           "awq_greedy_search")
    if check:
        check_workspace(ws, "awq_greedy_search (device)", stream)
    return s, tr, er


# ---------------------------------------------------------------------- after the path
def w4a16_workspace_size(M: int, D_in: int, D_out: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().awq_w4a16_workspace_size(M, D_in, D_out, ctypes.byref(n)), "awq_w4a16_workspace_size")
    return max(n.value, 256)


def w4a16_matmul(X: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                 s: Optional[torch.Tensor] = None, group_size: int = 128, out: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None, stream=None, check: bool = True) -> torch.Tensor:
    """Y = (X diag(1/s)) Dequant(qweight), bf16 [M, D_out]: the inference product on a packed layer."""
    _need(X, torch.bfloat16, "X")
    _need(qweight, torch.uint8, "qweight")
    _need(scales, torch.float16, "scales")
    _need(zeros, torch.float16, "zeros")
    if s is not None:
        _need(s, torch.float32, "s")
    M, D_in = X.shape
    D_out = qweight.shape[1]
    if qweight.shape[0] * 2 != D_in:
        raise ValueError("qweight must be [D_in/2, D_out]")
    if out is None:
        out = torch.empty(M, D_out, dtype=torch.bfloat16, device=X.device)
    if ws is None:
        ws = _alloc_ws(w4a16_workspace_size(M, D_in, D_out), X.device)
    cfg = make_cfg(group_size)
    _check(lib().awq_w4a16_matmul(_ptr(X), M, D_in, D_out, _ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(s),
                                  ctypes.byref(cfg), _ptr(out), _ptr(ws), ws.numel(), _stream_handle(stream)),
           "awq_w4a16_matmul")
    if check:
        check_workspace(ws, "awq_w4a16_matmul (device)", stream)
    return out


# ---------------------------------------------------------------------- self-test
def selftest_gemm(A: torch.Tensor, B: torch.Tensor, b_mn_major: bool = True, stream=None) -> torch.Tensor:
    """C = A @ B through the library's tensor-core main loop (test helper).

    A bf16 [M, K]; B bf16 [K, N] if b_mn_major else [N, K] (then C = A @ B.T)."""
    _need(A, torch.bfloat16, "A")
    _need(B, torch.bfloat16, "B")
    M, K = A.shape
    N = B.shape[1] if b_mn_major else B.shape[0]
    C = torch.empty(M, N, dtype=torch.float32, device=A.device)
    ws = _alloc_ws(256, A.device)
    _check(lib().awq_selftest_gemm_bf16(_ptr(A), _ptr(B), 1 if b_mn_major else 0, M, N, K, _ptr(C), _ptr(ws),
                                        ws.numel(), _stream_handle(stream)), "awq_selftest_gemm_bf16")
    check_workspace(ws, "awq_selftest_gemm_bf16 (device)", stream)
    return C


def selftest_wait_timeout(limit_ns: int, pairs: int, ws: torch.Tensor, stream=None) -> list:
    """Run the CTA-pair kernels' abort path on waits that never complete
    (test helper).  Returns the kernel's record [CTAs finished, CTAs whose
    wait expired, longest CTA run time in microseconds, CTAs whose bulk copy
    landed intact]; the status word of ws is left at AWQ_ERR_TIMEOUT."""
    record = torch.zeros(4, dtype=torch.int32, device=ws.device)
    _check(lib().awq_selftest_wait_timeout(int(limit_ns), int(pairs), _ptr(record), _ptr(ws), ws.numel(),
                                           _stream_handle(stream)), "awq_selftest_wait_timeout")
    return [int(v) for v in record.cpu().tolist()]


# ---------------------------------------------------------------------- profiling aid
def profile_enable(on: bool = True):
    """Bracket every library launch with CUDA events on its stream (process-wide)."""
    _check(lib().awq_profile_enable(1 if on else 0), "awq_profile_enable")


def profile_collect() -> dict:
    """{launcher name: (launches, total_ms)} since the last collect (synchronises the events)."""
    buf = (awq_kernel_time * 32)()
    n = ctypes.c_int32(0)
    _check(lib().awq_profile_collect(buf, 32, ctypes.byref(n)), "awq_profile_collect")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n.value)}
