"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the max-over-ranks timing,
the whole-job value, and the reference arm's rank handling (rank 0 alone runs and prints). The
path shards into independent replicas, so there is no data-path collective to test."""
import importlib.util
import io
import os
import socket
import contextlib

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        b = _bench()
        step_ms = 2.0 + rank * 1.5          # rank 1 is the slower one
        mx = b.max_over_ranks(step_ms, world, "cpu")
        value = b.whole_job_gbs(world, 1e9, mx)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{mx!r} {value!r}\n")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for mx, value in got:
        assert float(mx) == 3.5                                # every rank sees the slowest rank's time
        assert float(value) == pytest.approx(2 * 1e9 / 3.5e-3 / 1e9)


def test_single_rank_helpers_need_no_process_group():
    b = _bench()
    assert b.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert b.whole_job_gbs(1, 2e9, 1.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    b = _bench()
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 0, 2

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = b.run_reference(Args(), b.synth.WORKLOADS[b.DEFAULT_WORKLOAD])
    assert rc == 0 and buf.getvalue() == ""
