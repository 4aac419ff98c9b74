"""The replicas path of bench.py (no data-path collective: each rank drafts its
own blocks) on CPU: two gloo ranks through the same rendezvous, barrier and
max-over-ranks timing the GPU run uses, and the whole-job figures and config the
JSON line reports for N ranks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench as b
    try:
        w, r, loc = b.dist_setup()
        b.barrier(w)
        # rank r's step took (r + 1) ms; every rank must see the slowest one
        ms = b.max_over_ranks(float(r + 1), w)
        e2e = b.max_over_ranks(float(r + 1) * 1.25, w)
        b.barrier(w)
        q.put((r, w, loc, ms, e2e, b.job_figures(ms, e2e, w, 1, 7)))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_replica():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for r, (rank, w, loc, ms, e2e, jf) in enumerate(res):
        assert (rank, w, loc) == (r, world, r)
        assert ms == 2.0 and e2e == 2.5  # the maximum over ranks, on every rank
        # whole job: two replicas each draft one block per 2 ms step
        assert jf["us_per_block"] == pytest.approx(1000.0)
        assert jf["e2e_us_per_block"] == pytest.approx(1250.0)
        assert jf["drafted_tokens_per_s"] == pytest.approx(7 * 2 / 2e-3)


def test_single_process_needs_no_process_group():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_setup() == (1, 0, 0)
    bench.barrier(1)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_config_counts_every_replica():
    from synthetic.configs import FULL_STEP
    from synthetic import generate as gen
    ctx = gen.context_lengths(FULL_STEP)
    c1 = bench.run_config(FULL_STEP, ctx, 1, 0, 0, 1.0, 0.95, "bf16", 7 * 10**9)
    c4 = bench.run_config(FULL_STEP, ctx, 4, 0, 0, 1.0, 0.95, "bf16", 7 * 10**9)
    assert c1["parallelism"] == "replicas1" and c4["parallelism"] == "replicas4"
    assert c4["global_batch"] == 4 * c1["global_batch"] == 4 * FULL_STEP.bs
    assert c4["blocks_per_step"] == 4 * FULL_STEP.bs
    assert c1["temperature"] is None and c1["draft"] == "greedy"
