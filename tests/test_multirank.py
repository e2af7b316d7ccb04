"""The bench's multi-process path, on CPU with the gloo backend (two ranks).

The GEMM path does not shard (each GPU runs an independent replica), so the
only cross-rank steps are the bench's: every rank reads its rank from the
launcher's environment, the job's time is the slowest rank's, and only rank 0
prints.  These run here without a GPU."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        world, r, local = bench.dist_env()
        # rank 1 is the slow one: both ranks must report its time
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world, device="cpu")
        q.put((rank, world, r, local, got))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    out = sorted(q.get(timeout=5) for _ in range(2))
    assert out == [(0, 2, 0, 0, 15.0), (1, 2, 1, 1, 15.0)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_nonzero_rank_of_reference_arm_exits_quietly():
    """Under torchrun the reference arm runs on rank 0 alone; other ranks exit
    0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
