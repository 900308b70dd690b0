"""The N > 1 host path of bench.py on CPU: two gloo ranks (127.0.0.1).

bench.py runs one independent replica per GPU (slots shard by conversation,
no collective on the data path); across ranks it only needs the rendezvous,
a barrier around the timed region, the slowest rank's time, the whole-job
rate and rank-0-only reporting.  The reference arm does its work on rank 0
alone.  Each is checked here with real processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(world)
    try:
        bench.barrier()
        slowest = bench.max_over_ranks(10.0 * (rank + 1))
        rate = bench.whole_job_rate(w, 254, 4, slowest)

        class Args:
            steps, warmup, cpu_rows = 1, 0, 4
        ref_line = bench.run_reference(Args, r, w)[0]   # rank 0: 4 suffix rows of one layer
        q.put((r, w, dist.get_backend(), slowest, rate, ref_line))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank_and_only_rank0_reports():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[:3] for r in results] == [(0, 2, "gloo"), (1, 2, "gloo")]
    for r in results:
        assert r[3] == pytest.approx(20.0)                       # max over ranks of 10, 20 ms
        assert r[4] == pytest.approx(2 * 254 * 4 / 0.020)        # whole-job rows/s
    assert results[1][5] is None                                 # rank 1 of the reference arm: no work, no line
    # rank 0's reference line: the contract's keys, the GPU arm's config and metric, e2e without copies
    line = results[0][5]
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    sys.path.insert(0, ROOT)
    import bench
    assert line["impl"] == "reference" and line["metric"] == "suffix-prefill rows/s" and line["unit"] == "rows/s"
    assert line["config"] == bench.turn9_config(2) and line["n_gpus"] == 2
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and "4 suffix rows" in cb["sample"]
