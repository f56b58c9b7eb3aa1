"""The multi-process path of bench.py, on the host with gloo (no GPU).

Under torchrun every rank runs an independent replica of the workload; the
only cross-rank steps are the barrier around each timed region and the max of
the per-rank times, from which the whole-job rate follows.  The reference arm
runs on rank 0 only.  Two gloo ranks check exactly those pieces."""
import argparse
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    D = bench.Dist("gloo")
    D.barrier()
    ms = 10.0 + 5.0 * rank  # the slower rank bounds the job
    slowest = D.max(ms)
    rate = bench.job_rate(1000, slowest, D.world)
    D.barrier()
    queue.put((rank, D.world, slowest, rate))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in results] == [2, 2]
    assert [r[2] for r in results] == [15.0, 15.0]
    assert results[0][3] == results[1][3] == pytest.approx(2 * 1000 / 0.015)


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    D = bench.Dist("gloo")
    assert D.world == 1 and D.pg is None
    D.barrier()
    assert D.max(3.5) == 3.5
    assert bench.job_rate(64, 2.0, 1) == pytest.approx(32000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_measured_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """The DRAM traffic bench.py reports comes from a committed ncu record and
    is scaled by the units a launch processes; it is withdrawn (None) as soon as
    one of the kernel sources the record names differs from the captured ones."""
    import hashlib
    root = tmp_path
    (root / "profiles").mkdir()
    csrc = root / "rnn_sequence_mixer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("kernel a\n")
    (csrc / "b.cuh").write_text("header b\n")
    h = hashlib.sha256(b"kernel a\n" + b"header b\n").hexdigest()
    (root / "profiles" / "rec.md").write_text(
        f"# record\n\nbytes_per_token_head: 1277.50\nsource_sha256: {h}\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.measured_traffic("rec.md", ("a.cu", "b.cuh"), 1000) == pytest.approx(1277500.0)
    assert bench.measured_traffic("missing.md", ("a.cu", "b.cuh"), 1000) is None
    (csrc / "b.cuh").write_text("header b, changed\n")
    assert bench.measured_traffic("rec.md", ("a.cu", "b.cuh"), 1000) is None
