"""bench.py's multi-rank host logic on CPU: two gloo ranks.

With N processes (one per GPU under torchrun) the bench reports whole-job
figures: the slowest rank's time and the units summed over ranks.  These
tests run that reduction with two CPU ranks over gloo on 127.0.0.1 (no GPU),
check the numbers rank 0 would print, and check that the reference arm does
its work on rank 0 only.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r: train 100 + 50 r ms for 4,096 merges, encode 10 + r ms of 2^30 bytes
        times, units = bench.reduce_ranks([100.0 + 50 * rank, 10.0 + rank], [4096, 1 << 30], world, "cpu")
        value = bench.throughput(units[0], times[0])
        gbs = bench.throughput(units[1], times[1]) / 1e9
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{times[0]} {times[1]} {units[0]} {units[1]} {value} {gbs}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_whole_job_figures(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    assert rows[0] == rows[1]                        # every rank holds the same whole-job figures
    t_train, t_enc, merges, nbytes, value, gbs = map(float, rows[0])
    assert t_train == 150.0 and t_enc == 11.0        # the slowest rank's times
    assert merges == 2 * 4096 and nbytes == 2 * (1 << 30)
    assert value == pytest.approx(8192 / 0.150)      # total merges / max time ("weak" scaling)
    assert gbs == pytest.approx(2 * (1 << 30) / 0.011 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    times, units = bench.reduce_ranks([3.0, 4.0], [7, 8], 1, "cpu")
    assert times == [3.0, 4.0] and units == [7.0, 8.0]
    assert bench.throughput(5, 0.0) == 0.0 and bench.throughput(5, 1000.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only():
    import bench
    import argparse
    ns = argparse.Namespace(train="tiny", encode="none", steps=1, warmup=0, gpus=2, impl="reference")
    assert bench.run_reference(ns, 1, 2) is None      # other ranks exit without work
    out = bench.run_reference(ns, 0, 2)
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["cpu_baseline"]["cores"] == 1
    # the JSON line's contract: the bench line's keys, with this run's own
    # figures in cpu_baseline and e2e
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in out, key
    assert out["steps"] == 1 and out["warmup"] == 0 and out["higher_is_better"] is True
    assert out["vs_baseline"] is None and out["config"]["workload"]
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["sample"] and cb["value"] == out["value"] and cb["unit"] == out["unit"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"] and e2e["d2h_bytes_per_step"] == 0
