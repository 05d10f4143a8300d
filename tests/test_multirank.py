"""The multi-rank bench path on CPU: world_size-2 gloo ranks check the
max-over-ranks timing and the whole-job throughput, and a torchrun launch of
the reference arm prints exactly one line (rank 0) while rank 1 exits 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = [3.0, 5.0][rank]
        m = bench.max_over_ranks(ms, world, "cpu")
        dist.barrier()
        out.put((rank, m, bench.job_throughput(1000, m, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    for rank, m, value in got:
        assert m == 5.0                      # the slowest rank's time
        assert value == pytest.approx(2 * 1000 / 5e-3)   # both ranks' units / that time


def test_single_rank_helpers_need_no_process_group():
    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.job_throughput(10, 2.0, 1) == pytest.approx(5000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2",
           "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2 and line["steps"] == 2 and line["warmup"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0


def test_reference_arm_sample_shrinks_to_the_host_budget(monkeypatch, capsys):
    # With a budget far below one full step, each step times fewer samples.
    monkeypatch.setattr(bench, "REF_BUDGET_S", 1e-6)
    bench.main(["--impl", "reference", "--workload", "char_asr", "--steps", "2", "--warmup", "1",
                "--ref-samples", "8"])
    line = json.loads([l for l in capsys.readouterr().out.splitlines() if l.startswith("{")][-1])
    assert line["cpu_baseline"]["sample"].startswith("first 1 of 32 samples")
    assert line["value"] > 0
