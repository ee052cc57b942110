"""The column-sharded search on one GPU: the layer's columns split into
slices, each slice searched on its own, their block partials gathered in
slice order and the global alpha* selected in every slice's workspace.  The
losses, alpha* and s* must equal one search of the whole layer bit for bit,
and the slices' searched packs must be the whole layer's pack, column by
column.  (The multi-process exchange itself is tested with gloo ranks on the
CPU.)"""
import numpy as np
import pytest
import torch

from gpu_common import require_gpu
from post_weight_quantization_column_b300 import sharded, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


@pytest.mark.parametrize("widths,sym", [((768, 200), False), ((256, 512, 256), True)])
def test_sharded_search_equals_whole_layer(awq, widths, sym):
    w = synth.custom("sharded_gpu", 41, 300, 512, sum(widths), symmetric=sym, group_size=128)
    X, W = synth.generate(w)
    Xd, Wd = X.cuda(), W.cuda()
    a = awq.act_stats(Xd)
    full = awq.search(Xd, Wd, a, group_size=128, symmetric=sym)
    qf, sf, zf = awq.quantize_pack_searched(Wd, full, 128, sym)

    sharded.check_slices(widths)
    c0, parts = 0, []
    for width in widths:
        Ws = Wd[:, c0:c0 + width].contiguous()
        parts.append((c0, Ws, awq.search(Xd, Ws, a, group_size=128, symmetric=sym)))
        c0 += width
    blk = sharded.concat_block_losses([awq.search_block_losses(r) for _, _, r in parts])
    assert blk.shape == (21, (sum(widths) + 255) // 256)
    for c0, Ws, r in parts:
        awq.search_select(r, blk)
        torch.cuda.synchronize()
        assert torch.equal(r.losses, full.losses)
        assert r.best == full.best
        assert torch.equal(r.s_star, full.s_star)
        q, s_, z = awq.quantize_pack_searched(Ws, r, 128, sym)
        n = Ws.shape[1]
        assert torch.equal(q, qf[:, c0:c0 + n]) and torch.equal(s_, sf[:, c0:c0 + n]) and torch.equal(z, zf[:, c0:c0 + n])
