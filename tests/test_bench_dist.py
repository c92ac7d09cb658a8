"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2).

The layer runs as independent replicas on several GPUs; the benchmark only sums the
routed rows of all ranks and divides by the slowest rank's time.
"""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.Dist(backend="gloo")
    d.barrier()
    value, t = bench.aggregate(100.0 * (rank + 1), 1.0 + rank, d)
    q.put((rank, value, t))
    d.close()


def test_aggregate_sums_units_over_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, t in res:
        assert t == 2.0 and value == 150.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    d = bench.Dist(init=False)
    args = bench.main.__globals__["argparse"].Namespace(workload="tiny", steps=1, warmup=3,
                                                        ref_budget_s=1.0)
    assert bench.run_reference(args, d) is None


def test_work_model_counts_valid_rows_only():
    from combine_persistent_warp_gb300.workloads import make_inputs
    inp = make_inputs("tiny")
    inp.topk_idx[0, 0] = -1
    m = bench.work_model(inp)
    assert m["M"] == 64 * 2 - 1
    assert m["flops"] == 6 * m["M"] * 256 * 128
