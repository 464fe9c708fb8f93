"""The replica path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The hot path shards with no exchange, so N GPUs run N independent replicas;
what crosses ranks is host logic only: a barrier, the max of the timings
over ranks, and the whole-job value (all ranks' units / the slowest rank's
time).  The reference arm prints from rank 0 alone.
"""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, what):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    if what == "aggregate":
        r, w, dist = bench.dist_setup(world)
        assert (r, w) == (rank, world)
        ms_local = [2.0, 5.0][rank]
        value, ms = bench.whole_job_gbs(dist, w, 10 ** 9, ms_local)
        bench.barrier(dist)
        with open(os.path.join(out_dir, "agg%d.json" % rank), "w") as f:
            json.dump({"value": value, "ms": ms}, f)
        dist.destroy_process_group()
    else:
        import argparse
        import contextlib
        import io
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(argparse.Namespace(gpus=world, steps=1, warmup=0))
        with open(os.path.join(out_dir, "ref%d.txt" % rank), "w") as f:
            f.write(buf.getvalue())


def _spawn(world, what, out_dir):
    mp.start_processes(_rank_main, args=(world, _free_port(), str(out_dir), what), nprocs=world,
                       start_method="spawn", join=True)


def test_whole_job_value_takes_the_slowest_rank(tmp_path):
    _spawn(2, "aggregate", tmp_path)
    for r in range(2):
        d = json.load(open(tmp_path / ("agg%d.json" % r)))
        assert d["ms"] == 5.0                      # max over ranks, seen by every rank
        assert d["value"] == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    _spawn(2, "reference", tmp_path)
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text().strip()
    assert out1 == ""
    assert len(out0) == 1
    line = json.loads(out0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
