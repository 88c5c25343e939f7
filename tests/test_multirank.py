"""The benchmark's multi-rank host logic on CPU: two gloo ranks, launched the
way torchrun launches them (WORLD_SIZE / RANK / LOCAL_RANK in the environment,
rendezvous on 127.0.0.1).  Replicas exchange no data; the only collective is the
MAX over the ranks' step times, and the job's value is all ranks' work over the
slowest rank's time.  The reference arm runs on rank 0 alone."""
import contextlib
import io
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    from context_ra_forward_gb300 import inputs

    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
        w_, r_, lr_ = bench.rank_env()
        assert (w_, r_, lr_) == (world, rank, rank)
        # each rank's own step time; the job takes the slowest
        ms = [12.5, 40.0][rank]
        slowest = bench.max_over_ranks(ms, world)
        bench.barrier(world)
        value = bench.whole_job_tflops(world, 3.0e15, slowest)
        # every rank draws its own batch (small shape of the same generator)
        w = inputs.Workload("mr", 1, 1, 64, 64, "bf16", True, False, 2, "zigzag", False, 11)
        x = inputs.make_inputs(w, seed=bench.rank_seed(w, rank))["q"].float()
        gathered = [torch.zeros_like(x) for _ in range(world)]
        dist.all_gather(gathered, x)
        distinct = not torch.equal(gathered[0], gathered[1])
        # the reference arm: rank 0 alone prints; rank 1 returns at once without work
        out = io.StringIO()
        if rank == 1:
            with contextlib.redirect_stdout(out):
                bench.run_reference(None, w)
        dist.destroy_process_group()
        q.put((rank, slowest, value, distinct, out.getvalue()))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, "error", repr(e), None, None))


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r = q.get(timeout=240)
        res[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert res[r][1] != "error", res[r][2]
        _, slowest, value, distinct, out = res[r]
        assert slowest == 40.0                       # MAX over ranks, the same on both
        assert abs(value - 2 * 3.0e15 / 40e-3 / 1e12) < 1e-9
        assert distinct                               # no two replicas time the same batch
    assert res[1][4] == ""                            # reference arm: rank 1 printed nothing


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)
    assert abs(bench.whole_job_tflops(1, 1.0e12, 1.0) - 1000.0) < 1e-9
