"""The multi-process path of bench.py on CPU with the gloo backend (world size 2): the timing
reduction takes the maximum over ranks, the barrier returns on every rank, and under torchrun
only rank 0 prints its JSON line.  The forward itself shards over (batch, head) pairs with no
data-path collective, so these host-side pieces are all there is to the N > 1 path."""
import json
import os
import socket
import subprocess
import sys
import time

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, local, w = bench.dist_setup()
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(w)
    got = bench.max_over_ranks(1.0 + 2.0 * rank, w)  # rank 0: 1.0, rank 1: 3.0
    out[rank] = got
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 3.0, 1: 3.0}


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def _worker_dead_peer(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_setup(timeout_s=15)
    if rank == 1:
        return  # this rank leaves before the barrier: it never joins the collective
    t0 = time.time()
    try:
        bench.barrier(world)
        bench.max_over_ranks(1.0, world)
        out[rank] = ("no error", time.time() - t0)
    except Exception as e:  # the surviving rank must learn of the missing peer
        out[rank] = (type(e).__name__, time.time() - t0)


def test_dead_rank_is_detected_not_waited_for():
    """A rank that exits between steps: the other rank's next collective fails within the
    process-group timeout (15 s here) instead of waiting for it."""
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker_dead_peer, args=(2, port, out), nprocs=2, join=True)
        kind, waited = out[0]
        assert kind != "no error"
        assert waited < 60, waited

