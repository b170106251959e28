"""The N > 1 path of bench.py on CPU, two ranks over gloo (127.0.0.1): the
rendezvous, the barrier and the max-over-ranks reduction that turns per-rank
times into the whole-job figure, and a two-process launch of the reference
arm (rank 0 alone prints its JSON line; the other ranks exit 0).  The
operator shards as replicas (independent heads), so these are the only
cross-rank steps."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, ws, r, local = bench._dist()
    try:
        bench._barrier(dist)
        mx = bench._max_over_ranks(dist, 1.5 + rank)      # per-rank "times" 1.5 and 2.5
        out.put((r, ws, local, mx, dist.get_backend()))
    finally:
        dist.destroy_process_group()


def _build_worker(rank, port, out, fail):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from bidirectional_masked_linear_gb300 import build

    def fake_build():
        if fail:
            raise RuntimeError("nvcc failed: planted error")
        return build.LIB

    build.build = fake_build
    dist, ws, r, local = bench._dist()
    try:
        bench._build_once(dist, r)
        out.put((r, "ok"))
    except (RuntimeError, SystemExit) as e:
        out.put((r, str(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fail", (False, True))
def test_build_outcome_reaches_every_rank(fail):
    """Rank 0 builds; a failed build ends the other rank with the same error
    (through the process group's store) instead of leaving it in a barrier."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_build_worker, args=(r, port, q, fail)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    if fail:
        assert "planted error" in res[0] and "planted error" in res[1] and "rank 1" in res[1]
    else:
        assert res == {0: "ok", 1: "ok"}


def test_two_rank_helpers_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1]
    for rank, ws, local, mx, backend in res:
        assert ws == 2 and local == rank and backend == "gloo"
        assert mx == 2.5                                     # the slower rank sets the job time


def test_reference_arm_under_torchrun_two_ranks():
    pytest.importorskip("torch.distributed.run")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_d_fp32", "--mask", "d",
           "--chunk", "16"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                                  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
