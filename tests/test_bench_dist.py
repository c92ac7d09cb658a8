"""The benchmark's bookkeeping on CPU: multi-rank aggregation (gloo, world size 2), the
reference arm's rank, the work model and the recorded DRAM-traffic lookup.

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


def test_recorded_traffic_is_used_only_for_the_sources_it_was_taken_on(monkeypatch):
    """A recorded DRAM-traffic figure enters the roofline line only while the kernel's
    sources hash to the state it was captured on; block-scaled workloads look up the
    block-scaled kernel's sources."""
    from combine_persistent_warp_gb300.workloads import make_inputs
    m = bench.work_model(make_inputs("tiny"))
    cur = bench.kernel_sources_sha("expert_ffn")
    cur_bs = bench.kernel_sources_sha("expert_ffn_bs")
    assert cur != cur_bs
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {
        ("tiny", "expert_ffn"): {"bytes": 1234, "src_sha": cur},
        ("tiny-pow2", "expert_ffn"): {"bytes": 5678, "src_sha": cur_bs},
        ("tiny-mxfp4", "expert_ffn"): {"bytes": 999, "src_sha": cur},   # the other kernel's state
    })
    assert bench.roofline_for("expert_ffn", 1e-5, m, "tiny", None)["traffic"] == 1234
    assert bench.roofline_for("expert_ffn", 1e-5, m, "tiny-pow2", None)["traffic"] == 5678
    assert bench.roofline_for("expert_ffn", 1e-5, m, "tiny-mxfp4", None)["traffic"] is None
    assert bench.roofline_for("expert_ffn", 1e-5, m, "decode", None)["traffic"] is None
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {("tiny", "expert_ffn"): {"bytes": 1234, "src_sha": "0" * 16}})
    assert bench.roofline_for("expert_ffn", 1e-5, m, "tiny", None)["traffic"] is None
