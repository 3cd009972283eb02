"""bench.py's multi-process host logic (replicas, one process per GPU) on
CPU with the gloo backend and two ranks: the barrier, the max over ranks of
the step time, the whole-job aggregate, and the reference arm running on
rank 0 only.  No GPU is involved."""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist

    w, r, local = bench._dist()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench._barrier(w)
    # each rank's step time; the job takes the slowest
    t = bench._max_over_ranks(1.0 + rank, w)
    # whole-job value: units all ranks processed / the slowest rank's time
    kv_step = 1e9
    value = w * kv_step / (t * 1e-3) / 1e9
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max_ms": t, "value": value}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(x["max_ms"] == 2.0 for x in res)  # both ranks see the slower rank's time
    assert all(x["value"] == pytest.approx(world * 1e9 / 2e-3 / 1e9) for x in res)


def _ref_main(rank, world, port, out_dir):
    import contextlib
    import io
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    buf = io.StringIO()
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(world), "--steps", "1",
                "--warmup", "3"]
    with contextlib.redirect_stdout(buf):
        bench.main()
    with open(os.path.join(out_dir, f"ref{rank}.txt"), "w") as f:
        f.write(buf.getvalue())


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_ref_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text().strip()
    assert out1 == ""
    line = json.loads(out0[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == world
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
