"""bench.py's multi-process plumbing on CPU: two gloo ranks rendezvous on
127.0.0.1, the timing reduction returns the maximum over ranks on every rank,
and the reference arm does its work on rank 0 only (the other ranks return at
once). The path itself runs as independent replicas (no data-path
collective), so this is all the N > 1 logic there is."""
import multiprocessing as mp
import os
import socket
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                          MASTER_PORT=str(port), EPILORA_BENCH_BACKEND="gloo")
        import torch.distributed as dist

        import bench
        r, w, local = bench.dist_setup()
        mx = bench.max_over_ranks(1.5 * (rank + 1), w, "cpu")
        bench.barrier(w)
        args = types.SimpleNamespace(workload="8b_m1_fp8", steps=3, warmup=3)
        ref = bench.run_reference(args, r, w) if r != 0 else "skipped"
        dist.destroy_process_group()
        q.put((rank, r, w, local, mx, ref))
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks_reduce_max_and_reference_runs_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(i, 2, port, q)) for i in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, *rest in res:
        assert rest[0] != "error", rest
        r, w, local, mx, ref = rest
        assert (r, w, local) == (rank, 2, rank)
        assert mx == 3.0
        assert ref == ("skipped" if rank == 0 else None)
