"""bench.py's host logic on CPU: the multi-process plumbing (world size 2,
gloo) and the source hash that keys the committed ncu traffic.

The scan has no collective (one process per GPU runs an independent replica),
so what bench.py adds for N > 1 is host logic: process-group setup from the
torchrun environment, the barrier around the timed region, the max (and sum)
of a timing over ranks, and a reference arm that only rank 0 runs.  These
tests run that logic as two spawned CPU processes on the gloo backend.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), SSD_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    bench.dist_barrier()
    mx = bench.dist_reduce(10.0 + rank, "max")
    sm = bench.dist_reduce(1.5, "sum")
    # the reference arm: rank 0 alone works, the others return nothing
    ref = bench.run_reference(types.SimpleNamespace(workload="tiny", steps=1, warmup=0), rank, world) \
        if rank != 0 else "skipped"
    bench.dist_barrier()
    dist.destroy_process_group()
    out.put((rank, r, w, local, mx, sm, ref))


def test_two_gloo_ranks_reduce_and_barrier():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=10) for _ in range(2))
    for rank, (r, r2, w, local, mx, sm, ref) in enumerate(got):
        assert (r, r2, w, local) == (rank, rank, 2, rank)
        assert mx == 11.0          # the slowest rank's time is the job's
        assert sm == 3.0
        if rank != 0:
            assert ref is None     # only rank 0 runs and prints the reference arm


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_reduce(4.25, "max") == 4.25
    assert bench.dist_reduce(4.25, "sum") == 4.25
    bench.dist_barrier()   # no process group: a no-op


def test_kernel_hash_ignores_comments_only():
    """The source hash that keys the committed ncu traffic tracks code, not
    comments or layout."""
    sys.path.insert(0, ROOT)
    import bench
    a = 'int f(int x) { // one\n  return x + 1; /* two\n lines */ }\nconst char *s = "// kept";\n'
    b = 'int f(int x) {\n    return x + 1;\n}\nconst char *s = "// kept";  // note\n'
    c = 'int f(int x) { return x + 2; }\nconst char *s = "// kept";\n'
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens(a) != bench.code_tokens(c)
    assert '"// kept"' in bench.code_tokens(a)
    h = bench.kernel_source_hash("chunk_scan")
    assert len(h) == 16 and h == bench.kernel_source_hash("chunk_scan")
