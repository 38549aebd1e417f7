"""bench.py's multi-rank path on CPU with gloo, world_size 2 (no GPU): the timing
reduction takes the maximum over ranks, both ranks pass the barriers, and the reference
arm prints its single JSON line on rank 0 only."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, mode):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if mode == "max":
            w, r, _ = bench.dist_env()
            bench.barrier(w)
            t = bench.max_over_ranks(0.25 + rank, w)
            bench.barrier(w)
            q.put(("max", r, w, t))
        else:
            import contextlib
            import io
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                bench.main(["--impl", "reference", "--workload", "caseA", "--steps", "1", "--warmup", "3"])
            q.put(("ref", rank, world, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def _run(mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q, mode)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda x: x[1])


def test_time_is_the_maximum_over_ranks():
    out = _run("max")
    assert [o[2] for o in out] == [2, 2]
    assert all(o[3] == pytest.approx(1.25) for o in out)


def test_reference_arm_prints_once_on_rank0():
    out = _run("ref")
    line0, line1 = out[0][3].strip(), out[1][3].strip()
    assert line1 == ""
    d = json.loads(line0)
    assert d["impl"] == "reference" and d["unit"] == "TFLOPS" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
