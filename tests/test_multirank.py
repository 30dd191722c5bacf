"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The copy itself shards into independent replicas (no data-path collective);
what crosses ranks is the barrier around the timed region and the
max-over-ranks of the elapsed time.  The reference arm runs on rank 0 only.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        got = bench.max_over_ranks(10.0 * (rank + 1))
        info = bench.rank_info()
        # the reference arm: ranks other than 0 return at once without work
        args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
        rc = bench.run_reference(args) if rank != 0 else 0
        out.put((rank, got, info, rc))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, got, info, rc in res:
        assert got == 20.0                      # max over ranks, seen by every rank
        assert info == (rank, world, rank)
        assert rc == 0


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5     # not distributed: identity
    bench.barrier()                             # no-op
    cfg = {"n_tiles": 8, "src": {"shape": (4, 4), "stride": (4, 1), "offset": 0, "tile_stride": 0},
           "dst": {"shape": (4, 4), "stride": (1, 4), "offset": 0, "tile_stride": 0}, "elem_bytes": 2}
    assert bench.workload_bytes(cfg) == 2 * 8 * 16 * 2
    half = bench.sampled(cfg, 0.5)
    assert half["n_tiles"] == 4 and cfg["n_tiles"] == 8
    one = dict(cfg, n_tiles=1)
    s = bench.sampled(one, 0.5)
    assert s["src"]["shape"] == (2, 4) and s["dst"]["shape"] == (2, 4)


def test_bench_flag_combinations():
    """Mode flags that name no workload are refused before any GPU work."""
    import bench
    for argv in (["--in-place", "--workload", "5"], ["--unit-run", "--in-place"], ["--loop", "[(1, 1, 0)]"],
                 ["--unit-run", "--workload", "8"]):
        with pytest.raises(SystemExit):
            bench.check_args(bench.parse_args(argv))
    for argv in ([], ["--in-place"], ["--unit-run"], ["--workload", "8", "--loop", "[(4, 1, 0)]"]):
        bench.check_args(bench.parse_args(argv))


def test_kernel_hash_ignores_comments_but_not_code():
    """Profiles record a hash of their kernel's code; comment and spacing
    edits must leave it alone, code edits must not."""
    import bench
    a = bench._code_only(b"int a;  // one\n/* two\n three */ int b;\n\n#define X 1\n")
    b = bench._code_only(b"int a; /* other */\n   int b; // note\n#define X 1\n")
    c = bench._code_only(b"int a;\nint c;\n#define X 1\n")
    d = bench._code_only(b"int a;\nint b;\n#define X 2\n")
    assert a == b and a != c and a != d
    assert len(bench.kernel_sources_sha("warp_permute")) == 16
