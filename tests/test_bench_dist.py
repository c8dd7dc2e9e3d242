"""bench.py's multi-process plumbing on CPU (gloo, world size 2): the
max/sum reductions over ranks, and a torchrun launch of the reference arm
in which rank 0 alone prints the JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    results[rank] = (d.max(float(rank + 1)), d.sum(float(10 * (rank + 1))))
    d.close()


def test_dist_reductions_gloo_two_ranks():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
        assert dict(results) == {0: (2.0, 30.0), 1: (2.0, 30.0)}


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert "whole steps" in line["cpu_baseline"]["sample"] and "rank 0 of 2" in line["cpu_baseline"]["sample"]
    cfg = line["config"]
    assert set(cfg) == {"workload", "tokens_per_step_per_gpu", "parts_tokens", "algorithmic_bytes_per_step", "l2",
                        "parallelism"}
    assert cfg["tokens_per_step_per_gpu"] == sum(cfg["parts_tokens"].values())
    assert cfg["parallelism"].startswith("replicas x2")


def test_algorithmic_bytes_per_part():
    """The byte counts both arms put in ``config``, on hand-sized parts."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench

    # a [2, 3] map with 4 segments: read 24 bytes, write 5 boundaries
    assert bench.part_bytes("map_small", np.zeros((2, 3), np.int32), 4, 6) == 24 + 20
    # ids/labels/one position plane, 3 kept sequences, T = 10, a [2, 2] length table
    thd = {"seq_lens": np.zeros((2, 2), np.int64)}
    assert bench.part_bytes("thd_small", thd, 3, 10) == 3 * 2 * 10 * 8 + 10 + 8 * 4 + 2 * 8 * 4
    # mRoPE counts three planes of positions
    assert bench.part_bytes("thd_ids", thd, 3, 10) == 5 * 2 * 10 * 8 + 10 + 8 * 4 + 2 * 8 * 4
    # bf16 rows of 6: two copies of T rows of 12 bytes
    emb = {"seq_lens": np.zeros((2, 2), np.int64), "hidden": np.zeros((2, 5, 6), np.int16)}
    assert bench.part_bytes("thd_emb", emb, 3, 10) == 2 * 10 * 6 * 2 + 10 + 8 * 4 + 2 * 8 * 4
    # two bins of width 8, members of 3 and 5 real tokens: read the real tokens,
    # write every slot (8 bytes) and its mask byte, and both cu arrays
    sq = {"bin_offsets": np.array([0, 1, 2]), "real_lens": np.array([3, 5]), "width": 8}
    assert bench.part_bytes("squeeze", sq, 2, 0) == 8 * 8 + 9 * 2 * 8 + 8 * 4


def test_native_arm_refuses_multi_gpu_without_torchrun():
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2"], cwd=ROOT, capture_output=True, text=True,
                       timeout=120, env={**os.environ, "WORLD_SIZE": "1"})
    assert r.returncode != 0 and "torchrun" in r.stderr
