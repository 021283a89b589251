"""The multi-rank path of bench.py on the CPU (gloo, world size 2).

Requests are independent (no term of the rule couples two requests), so
ranks shard the work by requests with no collective on the data path: each
rank verifies its own batch, and the only cross-rank steps are the barrier
around the timed region and the maximum of the ranks' times.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
import oracle  # noqa: E402
from speculative_decoding_verify_sample_gb300 import synth  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        bench.barrier(torch, world)
        # each rank times its own batch; the job's time is the slowest rank's
        slowest = bench.max_over_ranks(torch, world, 10.0 + 5.0 * rank, cpu)
        bench.barrier(torch, world)
        # each rank's batch, verified on its own (no cross-rank data)
        inp = synth.make_inputs("tiny", bench.rank_seed(synth.DEFAULT_SEED["tiny"], rank))
        acc, out, _ = oracle.verify_sample(inp)
        queue.put((rank, slowest, inp["uniforms"][0, 0].item(), acc.tolist(), out.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_only_the_slowest_time():
    ctx = torch.multiprocessing.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(2):
            rank, slowest, u0, acc, out = queue.get(timeout=180)
            results[rank] = (slowest, u0, acc, out)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert results[0][0] == results[1][0] == 15.0          # max over ranks
    assert results[0][1] != results[1][1]                   # different requests per rank
    # each rank's outputs equal the oracle run on that rank's batch alone
    for rank in (0, 1):
        inp = synth.make_inputs("tiny", bench.rank_seed(synth.DEFAULT_SEED["tiny"], rank))
        acc, out, _ = oracle.verify_sample(inp)
        assert results[rank][2] == acc.tolist() and results[rank][3] == out.tolist()


def test_sharding_by_requests_needs_no_exchange():
    # the rule has no cross-request term: verifying two ranks' batches as one
    # batch gives each rank's results unchanged
    a = synth.make_inputs("tiny", bench.rank_seed(synth.DEFAULT_SEED["tiny"], 0))
    b = synth.make_inputs("tiny", bench.rank_seed(synth.DEFAULT_SEED["tiny"], 1))
    both = dict(a)
    both["B"] = a["B"] + b["B"]
    for k in ("target", "draft", "draft_tokens", "draft_len", "temperature", "uniforms",
              "uniforms_resample"):
        if a.get(k) is not None:
            both[k] = np.concatenate([np.asarray(a[k]), np.asarray(b[k])])
    acc_a, out_a, _ = oracle.verify_sample(a)
    acc_b, out_b, _ = oracle.verify_sample(b)
    acc, out, _ = oracle.verify_sample(both)
    assert np.array_equal(acc, np.concatenate([acc_a, acc_b]))
    assert np.array_equal(out, np.concatenate([out_a, out_b]))


def test_job_rate_counts_every_rank():
    # 2 ranks x 20 steps x 160 rows in 0.5 s (the slowest rank) = 12800 rows/s
    assert bench.job_rate(160, 20, 2, 0.5) == 12800.0
    assert bench.job_rate(160, 20, 1, 0.5) == 6400.0


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        impl, workload, seed, steps, warmup = "reference", "tiny", None, 1, 3
    assert bench.run_reference(Args, 2, 1) is None


def test_reference_arm_json_line_keys():
    # the reference arm's line carries the contract's keys (tiny workload, CPU)
    class Args:
        impl, workload, seed, steps, warmup = "reference", "tiny", None, 1, 3
    line = bench.run_reference(Args, 1, 0)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert "workload" in line["config"]


def test_cpu_baseline_helpers():
    inp = synth.make_inputs("tiny")
    rate, cores, sample = bench.cpu_oracle_rate(inp, budget_s=0.2)
    assert rate > 0 and cores >= 1 and "requests" in sample
    assert bench.cpu_oracle_single_thread_rate(inp, budget_s=0.05) > 0
    model = bench.cpu_model()
    assert isinstance(model, str) and model
