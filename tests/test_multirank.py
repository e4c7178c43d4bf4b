"""Replicas over ranks, on CPU (gloo, world size 2).

The indexer has no exchange step, so N GPUs run N independent replicas:
bench.py takes each timing's maximum over the ranks (a MAX all-reduce) and
reports every rank's pairs over that time. These tests run the same
functions with two gloo ranks on the host, and check that the reference arm
does no work on a rank other than 0.
"""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step time 10 + r ms, end-to-end time 30 - r ms
        mx = bench.max_over_ranks([10.0 + rank, 30.0 - rank], world, "cpu")
        q.put((rank, mx, bench.whole_job_value(1000, world, 5, mx[0])))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_replicas_report_the_slowest_rank():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value in got:
        assert mx == [11.0, 30.0]                      # element-wise max over the two ranks
        assert value == pytest.approx(1000 * 2 * 5 / 11e-3)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert bench.whole_job_value(10, 1, 4, 2.0) == pytest.approx(20000.0)


def test_reference_arm_works_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""                      # no line, no work


def test_bench_command_line_parses():
    """bench.py imports and lists every mode without a GPU (its timed paths run
    on the GPU; this catches a broken edit before that)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--help"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    for opt in ("--gpus", "--steps", "--warmup", "--workload", "--impl", "--ln-append", "--project",
                "--mla", "--fused-only", "--record-traffic"):
        assert opt in r.stdout, opt
