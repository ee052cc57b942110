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
