"""bench.py's multi-process host logic with two gloo ranks on CPU: process
group set-up from the launcher's environment, barrier, max-over-ranks time
and the whole-job aggregate (every rank's work over the slowest rank's time)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.dist_barrier()
    t = 1.0 + rank                        # rank 1 is the slow one
    t_max = bench.dist_max(t)
    value = bench.aggregate(1e12, 10, w, t_max)
    out.put((rank, t_max, value))
    bench.dist_barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, value in res:
        assert t_max == pytest.approx(2.0)
        # 2 ranks x 10 steps x 1 TFLOP over the slowest rank's 2 s
        assert value == pytest.approx(10.0)


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_max(3.5) == 3.5
    assert bench.aggregate(2e12, 5, 1, 2.0) == pytest.approx(5.0)


def test_kernel_hash_ignores_comments_only():
    """The traffic figures stay tied to the kernel code: a comment edit keeps
    the hash, a code edit changes it."""
    import bench
    src = "int a = 1; // one\n/* block\n comment */\nint b = 2;\n"
    assert bench.code_of(src) == bench.code_of("int a = 1;   // other words\n\nint b = 2;\n")
    assert bench.code_of(src) != bench.code_of("int a = 1;\nint b = 3;\n")
    assert len(bench.kernel_hash()) == 16


def test_sweep_best_names_the_fastest_point_per_op():
    import bench
    pts = [
        {"op": "ag", "N": 4, "chunks": 1, "ring": "uni", "ms": 2.2, "frac_of_peak": 0.90},
        {"op": "rs", "N": 4, "chunks": 1, "ring": "uni", "ms": 2.3, "frac_of_peak": 0.88},
        {"op": "ag", "N": 8, "chunks": 2, "ring": "bidi", "ms": 2.1, "frac_of_peak": 0.95},
        {"op": "rs", "N": 16, "chunks": 4, "ring": "pipelined", "ms": 3.0, "frac_of_peak": 0.6},
        {"op": "ag", "N": 16, "chunks": 4, "ring": "uni", "ms": 2.15, "frac_of_peak": 0.93},
    ]
    best = {b["sweep_best"]: b for b in bench.sweep_best(pts)}
    assert list(best) == ["ag", "rs"]
    assert (best["ag"]["N"], best["ag"]["chunks"], best["ag"]["ring"], best["ag"]["ms"]) == (8, 2, "bidi", 2.1)
    assert (best["rs"]["N"], best["rs"]["ring"], best["rs"]["ms"]) == (4, "uni", 2.3)
    assert bench.sweep_best([]) == []


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the reference arm's other ranks join the process group
    and leave at once, without work and without a line of output."""
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    joined = []
    monkeypatch.setattr(bench, "dist_init", lambda backend: joined.append(backend) or (1, 2))

    def no_work(*a, **k):
        raise AssertionError("rank 1 must not build inputs or time the oracle")

    monkeypatch.setattr(bench, "make_step_inputs", no_work)
    monkeypatch.setattr(bench, "oracle_sample", no_work)
    args = argparse.Namespace(gpus=2, steps=2, warmup=3, ref_seconds=1.0)
    assert bench.run_reference(args) == 0
    assert joined == ["gloo"]
    assert capsys.readouterr().out == ""
