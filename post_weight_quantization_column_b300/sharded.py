"""The search sharded over output columns: one process per GPU.

"AWQ (Activation-aware Weight Quantization)", 缩放因子优化的完整流程 step 4c:
the loss L = ||X S^-1 W'hat - X W||^2 is a sum over output columns, so every
candidate's loss of the whole layer is the sum of its losses over disjoint
column slices.  Each rank searches X against its own slice W[:, c0:c1]; the
only exchange is one all-gather of the G x ceil(slice / 256) fp64 block
partials, after which every rank sums the blocks in slice order on its GPU
(awq_search_select), so all ranks hold the same losses, alpha* and s*, and
each packs its own slice at that alpha*.

When every slice but the last spans a multiple of 256 columns, the blocks are
exactly those one search of the whole layer forms, and the losses are the
same to the last bit.  This module only moves data; the sums run in the
library's kernels.
"""
from __future__ import annotations

import torch

from . import SearchResult, search, search_block_losses, search_select

BLOCK_COLS = 256


def gather_block_losses(blk: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather each rank's [G, nb_r] block partials; returns [G, sum nb_r]
    with the ranks' blocks in rank order (identical on every rank).  Works
    with the gloo backend on CPU tensors and with NCCL on CUDA tensors."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    G, nb = blk.shape
    sizes = [torch.zeros(1, dtype=torch.int64, device=blk.device) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([nb], dtype=torch.int64, device=blk.device), group=group)
    sizes = [int(t.item()) for t in sizes]
    width = max(sizes)
    padded = torch.zeros(G, width, dtype=blk.dtype, device=blk.device)
    padded[:, :nb] = blk
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded.contiguous(), group=group)
    return torch.cat([p[:, :n] for p, n in zip(parts, sizes)], dim=1).contiguous()


def check_slices(widths) -> None:
    """Every slice but the last must span whole 256-column blocks, so that the
    gathered blocks are the whole layer's blocks."""
    for w in list(widths)[:-1]:
        if w % BLOCK_COLS:
            raise ValueError(f"a column slice of {w} columns: every slice but the last must span a multiple of "
                             f"{BLOCK_COLS} columns")


def search_column_sharded(X: torch.Tensor, W_slice: torch.Tensor, mean_abs: torch.Tensor, grid=None,
                          group_size: int = 128, symmetric: bool = False, act_floor: float = 1e-4, group=None,
                          stream=None) -> SearchResult:
    """This rank's part of the column-sharded search.  X and mean_abs are the
    whole layer's; W_slice is this rank's columns (ranks in column order).
    Returns this rank's search result with losses / best_idx / s_star of the
    whole layer; awq_quantize_pack_searched on it packs this rank's slice."""
    import torch.distributed as dist
    res = search(X, W_slice, mean_abs, grid, group_size, symmetric, act_floor, stream=stream)
    blk = search_block_losses(res, stream)
    backend = dist.get_backend(group)
    host = backend == "gloo"
    local = blk.cpu() if host else blk
    widths = [torch.zeros(1, dtype=torch.int64, device=local.device) for _ in range(dist.get_world_size(group))]
    dist.all_gather(widths, torch.tensor([W_slice.shape[1]], dtype=torch.int64, device=local.device), group=group)
    check_slices([int(w.item()) for w in widths])
    full = gather_block_losses(local, group)
    return search_select(res, full.to(blk.device) if host else full, stream)


def concat_block_losses(blks) -> torch.Tensor:
    """The slices' block partials side by side, in slice order (one process
    holding several slices' results)."""
    return torch.cat(list(blks), dim=1).contiguous()


__all__ = ["gather_block_losses", "check_slices", "search_column_sharded", "concat_block_losses", "BLOCK_COLS"]
