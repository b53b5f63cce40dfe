"""The N > 1 path of bench.py on CPU: two ranks over gloo (the GPU runs use
NCCL and one GPU per rank; each rank is an independent replica, so the only
cross-rank steps are the barrier and the max over ranks of the step time).
Also: under torchrun only rank 0 runs the reference arm; the others exit 0
without work."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = [2.5, 3.75][rank]             # the second rank is slower
        dist.barrier()
        ms = bench.max_over_ranks(local_ms, ws)
        value = bench.job_tflops(ws, 3, 2.0 * 4096 ** 3, ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {value!r}\n")
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    ws, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    sys.path.insert(0, ROOT)
    import bench
    want_value = bench.job_tflops(2, 3, 2.0 * 4096 ** 3, 3.75)
    for r in range(ws):
        ms, value = map(float, open(tmp_path / f"rank{r}.txt").read().split())
        assert ms == 3.75
        assert value == pytest.approx(want_value, rel=1e-12)
    # replicas: two ranks doing the same work in the same time double the job rate
    assert bench.job_tflops(2, 3, 1e12, 1.0) == pytest.approx(2 * bench.job_tflops(1, 3, 1e12, 1.0))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
