"""The bench's multi-rank logic on CPU with two gloo ranks: max-over-ranks timing, barriers,
and rank-0-only output of the reference arm.  No GPU and no data-path collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    got = bench.reduce_max(10.0 + 5.0 * rank, w)
    args = type("A", (), {"ref_tokens": 1, "warmup": 0, "steps": 1})()
    line = bench.reference_arm(args, w, r) if rank == 1 else None
    q.put((rank, got, line))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0], "max over ranks"
    assert res[1][2] is None, "only rank 0 runs and prints the reference arm"


@pytest.mark.slow
def test_reference_arm_line_shape():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), {"ref_tokens": 2, "warmup": 0, "steps": 1})()
    line = bench.reference_arm(args, 1, 0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
