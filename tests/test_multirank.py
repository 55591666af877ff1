"""Two ranks on CPU (gloo): the benchmark's cross-rank timing reductions.

The library shards only as independent replicas (no data-path collective):
each rank times its own GEMM, rank 0 reports the FLOPs of all ranks over the
slowest rank's time.  These are the host-side pieces that combine ranks."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        ms = [3.0, 5.0][rank]            # rank 1 is the slow one
        flops = [1e12, 2e12][rank]
        bench.barrier(w)
        mx = bench.reduce_max(ms, w, device="cpu")
        tot = bench.reduce_sum(flops, w, device="cpu")
        out_q.put((rank, mx, tot))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    results = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, tot in results:
        assert mx == 5.0                 # max over ranks
        assert tot == 3e12               # sum over ranks
    # whole-job value as bench computes it: total FLOPs / slowest time
    assert tot / (mx / 1e3) / 1e12 == pytest.approx(600.0)


def test_single_rank_reductions_are_identity():
    import bench
    assert bench.reduce_max(2.5, 1) == 2.5
    assert bench.reduce_sum(7.0, 1) == 7.0
    bench.barrier(1)


def test_paper_figures_pin_the_flop_and_traffic_counts():
    """The pages print 137 GFLOP and 548 GB (naive reads) for 4092^3 and a
    block intensity of 32 FLOP/B for a 128 x 128 tile; the benchmark's
    counting functions must reproduce them (tests/golden/napkin_4092.txt)."""
    import bench
    rows = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "napkin_4092.txt")):
        if line.strip() and not line.startswith("#"):
            key, val = line.split()[:2]
            rows[key] = float(val)
    assert round(bench.gemm_flops(4092, 4092, 4092) / 1e9) == rows["gemm_flops_4092"]
    assert round(bench.naive_read_bytes(4092, 4092, 4092) / 1e9) == rows["naive_read_bytes_4092"]
    for bm, key in ((128, "block_ai_128x128"), (32, "block_ai_32x32")):
        # per k step: 2*BM*BN flops over 4*(BM+BN) bytes moved into shared memory
        assert bench.gemm_flops(bm, bm, 1) / (4 * (bm + bm)) == rows[key]
    # compulsory traffic: A, B read once, C written once (beta = 0)
    assert bench.compulsory_bytes(4092, 4092, 4092) == 3 * 4 * 4092 * 4092
