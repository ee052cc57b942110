"""bench.py's multi-rank plumbing with two gloo ranks on the CPU: the
rendezvous, the max over ranks of the step time, the barrier, and the
reference arm, which rank 0 alone runs and prints."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import contextlib
    import io

    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup()
    got = bench.max_over_ranks(1.5 * (r + 1), w)
    bench.barrier(w)
    args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0",
                             "--gpus", str(w)])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(args, w, r)
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "max": got, "rc": rc, "stdout": buf.getvalue()}, f)


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["world"] == r1["world"] == 2
    assert r0["max"] == r1["max"] == 3.0          # the larger of the two ranks' times
    assert r0["rc"] == r1["rc"] == 0
    assert r1["stdout"] == ""                     # the other ranks do no work
    line = json.loads(r0["stdout"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


# ---------------------------------------------------------------------------- column-sharded search, the exchange
def _block_tree(col):
    """fp64 block partials [G, nb] of per-column losses [G, D_out] in the
    search's order: each 256-column block (zero-padded) summed by halving,
    element t taking t + w for w = 128, 64, ..., 1."""
    import numpy as np
    G, D = col.shape
    nb = (D + 255) // 256
    sh = np.zeros((G, nb, 256), dtype=np.float64)
    sh.reshape(G, -1)[:, :D] = col
    w = 128
    while w >= 1:
        sh[:, :, :w] = sh[:, :, :w] + sh[:, :, w:2 * w]
        w //= 2
    return sh[:, :, 0].copy()


def _in_order(blk):
    L = [0.0] * blk.shape[0]
    for k in range(blk.shape[0]):
        acc = 0.0
        for b in range(blk.shape[1]):
            acc += float(blk[k, b])
        L[k] = acc
    return L


def _sharded_rank(rank, world, port, outdir, widths):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist

    from oracle import awq_oracle as orc
    from post_weight_quantization_column_b300 import sharded, synth
    from test_multirank_cpu import _block_tree
    dist.init_process_group("gloo")
    w = synth.custom("sharded", 31, 48, 256, sum(widths), symmetric=False, group_size=128)
    X, W = synth.generate(w)
    Xf, Wf = synth.bf16_to_f32(X), synth.bf16_to_f32(W)
    a = orc.act_stats(Xf)
    grid = orc.alpha_grid(21)
    c0 = sum(widths[:rank])
    cols = np.arange(c0, c0 + widths[rank])
    local = orc.search(Xf, Wf, a, grid, group_size=128, symmetric=False, cols=cols)["col_losses"]
    blk = torch.from_numpy(_block_tree(local))
    full = sharded.gather_block_losses(blk)
    err = ""
    try:
        sharded.check_slices([13 * 8] + list(widths))
    except ValueError as e:
        err = str(e)
    dist.destroy_process_group()
    np.save(os.path.join(outdir, f"blk{rank}.npy"), full.numpy())
    with open(os.path.join(outdir, f"err{rank}.txt"), "w") as f:
        f.write(err)


@pytest.mark.parametrize("widths", [(512, 256), (768, 200), (256, 256, 512)])
def test_column_sharded_exchange_is_bit_identical(tmp_path, widths):
    """Each rank holds the block partials of its own column slice (from the
    oracle's per-column losses, summed in the search's block order); after the
    all-gather every rank holds exactly the whole layer's block partials, so
    the in-order sums (the losses) and their argmin are the single-rank ones
    bit for bit."""
    import numpy as np

    from oracle import awq_oracle as orc
    from post_weight_quantization_column_b300 import synth
    world = len(widths)
    port = _free_port()
    mp.start_processes(_sharded_rank, args=(world, port, str(tmp_path), list(widths)), nprocs=world, join=True,
                       start_method="spawn")
    w = synth.custom("sharded", 31, 48, 256, sum(widths), symmetric=False, group_size=128)
    X, W = synth.generate(w)
    Xf, Wf = synth.bf16_to_f32(X), synth.bf16_to_f32(W)
    ref = orc.search(Xf, Wf, orc.act_stats(Xf), orc.alpha_grid(21), group_size=128, symmetric=False)
    single = _block_tree(ref["col_losses"])
    L_single = _in_order(single)
    for r in range(world):
        got = np.load(tmp_path / f"blk{r}.npy")
        assert got.shape == single.shape
        assert np.array_equal(got.view(np.uint64), single.view(np.uint64)), r
        L = _in_order(got)
        assert L == L_single
        assert int(np.argmin(L)) == int(np.argmin(L_single))
        # the oracle's own sum over all columns agrees to rounding
        np.testing.assert_allclose(L, ref["losses"], rtol=1e-12)
        assert "multiple of 256" in open(tmp_path / f"err{r}.txt").read()
