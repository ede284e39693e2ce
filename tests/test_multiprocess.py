"""The multi-rank path of bench.py on CPU (gloo, world size 2): the path is
replicas only (no collective on the data path), so what is tested is the
timing protocol around it: barriers, the max of the per-rank times, the
whole-job value = all ranks' tokens / that time, and the reference arm
running on rank 0 alone."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_info()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        ms = 2.0 + rank  # rank 1 is the slower replica
        ms_max = bench.reduce_max(ms, ws)
        T = 32768
        value = ws * T / (ms_max * 1e-3)  # whole-job tokens over the slowest rank's time
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms_max} {value}\n")
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_protocol(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for ms_max, value in rows:
        assert float(ms_max) == 3.0  # every rank sees the slowest rank's time
        assert float(value) == pytest.approx(2 * 32768 / 3e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""  # rank 1 prints nothing and does no work


def test_reduce_max_is_identity_at_world_size_one():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.25, 1) == 1.25
    bench.barrier(1)


def test_both_arms_share_the_headline_config():
    """The headline line and the reference arm name the same workload; the
    whole-job parallelism follows the world size."""
    sys.path.insert(0, ROOT)
    import bench
    from kda_gated_delta_02_gb300 import synth
    c1, c4 = bench.prefill_config(1), bench.prefill_config(4)
    assert c1["workload"] == synth.PREFILL_32K.name and c1["T"] == 32768 and c1["H"] == 96
    assert c1["parallelism"] == "replicas x1" and c4["parallelism"] == "replicas x4"
    assert {k: v for k, v in c1.items() if k != "parallelism"} == {k: v for k, v in c4.items() if k != "parallelism"}


def test_traffic_of_a_changed_kernel_is_not_reported(tmp_path, monkeypatch):
    """`traffic` comes from the committed ncu summary only while the kernel's
    source is the one captured; it scales with the tokens of a launch."""
    import json
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    root = tmp_path / "r"
    (root / "profiles").mkdir(parents=True)
    (root / "k.cu").write_text("kernel source\n")
    import hashlib
    sha = hashlib.sha256(b"kernel source\n").hexdigest()[:16]
    rec = {"k": {"source": "k.cu", "source_sha256_16": sha, "captured_T": 1000, "traffic_bytes_captured": 5e6}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.kernel_traffic("k", 4000) == 2e7
    assert bench.kernel_traffic("missing", 4000) is None
    (root / "k.cu").write_text("kernel source, changed\n")
    assert bench.kernel_traffic("k", 4000) is None
    shutil.rmtree(root)
