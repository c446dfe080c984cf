"""bench.py's multi-rank plumbing on two gloo ranks on the CPU.  The decode path
does not shard (each GPU runs an independent replica, no collective on the data
path); what spans ranks is the timing: the rendezvous, the barrier around the
timed region, the maximum of the per-rank step times, and the reference arm,
which rank 0 alone runs and prints."""
import json
import os
import socket
import sys
import types

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    # CPU ranks (gloo) even where GPUs are present: the GPUs stay hidden from them
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    try:
        w, r, _ = bench.dist_init(types.SimpleNamespace(impl="tfl"))
        backend = dist.get_backend()
        bench.barrier(w)
        worst = bench.max_over_ranks(1.5 + 2.0 * r, w)  # rank 1's step time is the larger
        bench.barrier(w)
        q.put((r, w, backend, worst))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_of_step_times():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    # both ranks see the slower rank's time: the whole-job rate divides the units
    # of all ranks by it
    assert got == [(0, 2, "gloo", 3.5), (1, 2, "gloo", 3.5)]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(context=8192, gpus=2, steps=1, warmup=3)
    bench.run_reference(args, 2, 1)  # rank 1: no work, no line
    assert capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1) == 4.25
    bench.barrier(1)  # no process group: a no-op
    assert json.dumps({"ok": True})
