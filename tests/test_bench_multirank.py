"""The bench's multi-rank host path on the CPU: two gloo ranks stand in for two
GPUs (one process per GPU, each a seeded replica of the workload; the step
time is the max over ranks; rank 0 alone prints the JSON line)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local_ms = [12.5, 30.25][rank]                 # rank 1 is the slow one
        ms = b.reduce_max(local_ms, world)
        dist.barrier()
        n_tok = 131072
        value = b.job_throughput(world, n_tok, ms / 4)  # 4 steps in the timed region
        line = b.emit({"rank_seen": rank, "ms": ms, "value": value}, rank)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value, "line": line,
                       "seed_offset": b.replica_seed_offset(rank)}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_rank0_output(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    # both ranks agree on the slowest rank's time
    assert r[0]["ms"] == r[1]["ms"] == 30.25
    # whole-job throughput: 2 replicas x 131072 tokens per (30.25 / 4) ms
    assert r[0]["value"] == pytest.approx(2 * 131072 / (30.25 / 4 / 1e3))
    # rank 0 prints one JSON line, the others print nothing
    assert r[0]["line"] is not None and json.loads(r[0]["line"])["rank_seen"] == 0
    assert r[1]["line"] is None
    # each rank draws its own seeded replica
    assert r[0]["seed_offset"] != r[1]["seed_offset"]


def test_single_rank_helpers():
    assert bench.reduce_max(7.0, 1) == 7.0
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(500000.0)
    assert bench.replica_seed_offset(0) == 0


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun the reference arm runs on rank 0 only: rank 1 exits 0 and
    prints nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_reports_the_device_arms_config(monkeypatch):
    """The reference arm's config is the one the device arm prints for rank 0
    (the cold long prompt's sizes come from its host-side segment lengths); the
    device draws are replaced by their offsets alone."""
    import types
    import numpy as np
    from linear_attn_state_gb300 import synth
    lengths = synth.cold_long_lengths()
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    fake = types.SimpleNamespace(offsets=off, n_seg=len(lengths), n_streams=480)
    monkeypatch.setattr(synth, "cold_long_device", lambda dev, n_layers=None, seed=None: fake)
    w = bench.ColdLong("cpu", 0, 30)
    assert dict(w.config, parallelism="replicas1") == bench.workload_config("cold_long", 30, 1)
    assert w.config["n_streams"] == 480 and w.config["n_tok"] == 131072
    lay = bench.workload_config("layer_reuse", 30, 2)
    assert lay["n_tok"] == 65536 and lay["parallelism"] == "replicas2"
