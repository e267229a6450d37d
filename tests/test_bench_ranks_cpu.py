"""The N > 1 host logic of bench.py on CPU, with two gloo ranks: each rank
takes its own contiguous batch of tokens, the timed region's times reduce
to the slowest rank's, the whole-job rate counts every rank's tokens, and
the reference arm runs on rank 0 only."""
import multiprocessing as mp
import os
import socket
import sys
from pathlib import Path
from types import SimpleNamespace

import pytest

ROOT = Path(__file__).resolve().parent.parent


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    sys.path.insert(0, str(ROOT))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank times: (step ms, end-to-end ms, GEMM ms), different on each rank
        local = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        reduced = bench.max_over_ranks(local, world, "cpu")
        dist.barrier()
        q.put((rank, reduced, bench.rank_token_range(rank, 8)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_split_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for _, reduced, _ in results:
        assert reduced == [2.0, 5.0, 0.5]  # element-wise maximum over the ranks
    (r0, _, t0), (r1, _, t1) = results
    assert (r0, r1) == (0, 1)
    assert t0 == (0, 8) and t1 == (8, 16)  # disjoint, contiguous token batches


def test_whole_job_rate_and_one_rank():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.whole_job_rate(8, 2, 4.0) == pytest.approx(8 * 2 / 4e-3)
    assert bench.max_over_ranks([3.0, 1.5], 1, "cpu") == [3.0, 1.5]
    assert bench.rank_token_range(0, 4096) == (0, 4096)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, str(ROOT))
    import bench
    args = SimpleNamespace(config="tiny", steps=1, warmup=3, w8a8=False, emulate=False)
    assert bench.reference_arm(args, None, 1, 2) is None
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes_match_the_per_expert_figures():
    """The roofline's byte counts: one touched expert with no routes is its
    weights (MXFP4 23,396,352 B and NVFP4 24,772,608 B at H=7168, I=2048;
    E4M3 plus fp32 row scales; BF16), one route of one token with no weights
    is the activation traffic of each GEMM plus the token's fp32 output row,
    further routes of that token add their activation rows only; the Kimi
    decode line (44 touched experts, 64 routes) is the 686,606,336 B of the
    committed profile."""
    sys.path.insert(0, str(ROOT))
    import bench
    H, I = 7168, 2048
    assert sum(bench.algorithmic_bytes(H, I, "mxfp4", "a4w4", 1, 0, 0)) == 23_396_352
    assert sum(bench.algorithmic_bytes(H, I, "nvfp4", "a4w4", 1, 0, 0)) == 24_772_608
    assert sum(bench.algorithmic_bytes(H, I, "mxfp4", "w8a8", 1, 0, 0)) == 3 * H * I + 4 * (2 * I + H)
    assert sum(bench.algorithmic_bytes(H, I, "nvfp4", "emulate", 1, 0, 0)) == 3 * H * I * 2
    gu, dn = bench.algorithmic_bytes(H, I, "mxfp4", "a4w4", 0, 1, 1)
    assert gu == (H + I) * 17 / 32 and dn == I * 17 / 32 + 4 * H
    gu8, dn8 = bench.algorithmic_bytes(H, I, "mxfp4", "a4w4", 0, 8, 1)
    assert gu8 == 8 * gu and dn8 == 8 * I * 17 / 32 + 4 * H
    assert bench.algorithmic_bytes(H, I, "mxfp4", "a4w4", 44, 64, 8)[0] == 686_606_336
    with pytest.raises(ValueError):
        bench.algorithmic_bytes(H, I, "mxfp4", "w4a16", 1, 1, 1)
