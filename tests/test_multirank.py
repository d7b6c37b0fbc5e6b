"""The host logic of bench.py on CPU: with two gloo ranks (replicas
only, so the only exchange is the max-over-ranks of the timed region), the
job's value counts every replica, and the reference arm runs on rank 0
alone (the other ranks exit without work); in one process, the reference
arm's line carries the same workload config as the GPU arm's."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [12.5, 20.0][rank]
        out[rank] = {"max": bench.max_over_ranks(elapsed, dist, "cpu"),
                     "value": bench.job_tokens_per_s(world, 256, 10,
                                                     bench.max_over_ranks(elapsed, dist, "cpu"))}
        args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "3",
                                 "--warmup", "3"])
        res = bench.run_reference(args, rank, world)
        out[rank] = dict(out[rank], ref=None if res is None else res["impl"])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_aggregate_value():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        assert res[r]["max"] == 20.0                    # the slowest replica's time
        assert res[r]["value"] == pytest.approx(2 * 256 * 10 / 0.020)
        assert res[r]["ref"] == ("reference" if r == 0 else None)   # rank 0 alone


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tokens_per_s(1, 256, 100, 10.0) == pytest.approx(256 * 100 / 0.010)


def test_bench_path_rules_follow_the_library(monkeypatch):
    """bench.py names the kernels lora_linear takes (and counts its launches
    from them): the cooperative kernel on the tiny batch, the rank-128
    tensor-core kernel on the large one (72 or more tokens per SM) unless
    LORA_PUNICA_LINEAR_TC=0, three kernels on the rank-64 prefill."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    from dataclasses import replace
    for k in ("LORA_PUNICA_COOP", "LORA_PUNICA_FUSED", "LORA_PUNICA_LINEAR_TC",
              "LORA_PUNICA_LINEAR_TC_MIN_TOKENS"):
        monkeypatch.delenv(k, raising=False)
    assert bench.coop_path(W.WORKLOADS["tiny"]) and not bench.linear_tc_path(W.WORKLOADS["tiny"])
    assert bench.linear_tc_path(W.WORKLOADS["large"], 152)
    # below 72 tokens per SM: the separate kernels
    assert not bench.linear_tc_path(replace(W.WORKLOADS["large"], num_tokens=8192), 152)
    assert bench.linear_tc_path(replace(W.WORKLOADS["large"], num_tokens=8192), 100)
    assert not bench.linear_tc_path(W.WORKLOADS["prefill"])          # rank 64
    assert not bench.linear_tc_path(W.WORKLOADS["embedding"])
    monkeypatch.setenv("LORA_PUNICA_LINEAR_TC", "0")
    assert not bench.linear_tc_path(W.WORKLOADS["large"])


def test_reference_line_matches_the_contract():
    """The reference arm times the oracle on the host on the same workload
    config as the GPU arm, with zero host-device bytes in its e2e."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "3",
                             "--warmup", "3"])
    res = bench.run_reference(args, 0, 1)
    assert res["impl"] == "reference" and res["metric"] == bench.METRIC
    assert res["unit"] == "tokens/s" and res["higher_is_better"] is True
    assert res["steps"] == 3 and res["warmup"] == 3 and res["value"] > 0
    w = W.WORKLOADS["tiny"]
    want = bench.workload_config(w, W.unique_bytes(w, W.generate(w).ids), args)
    assert {k: v for k, v in res["config"].items() if k != "parallelism"} == want
    assert res["e2e"] == {"value": res["value"], "unit": "tokens/s",
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = res["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == res["value"] and cb["cores"] >= 1
    assert "tokens" in cb["sample"]
