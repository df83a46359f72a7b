"""The bench's multi-rank host logic on CPU, with two gloo ranks: every rank
runs its own independently seeded batch (no data-path collective), the time
reported is the slowest rank's, and the throughput counts every rank's work.
The reference arm runs on rank 0 only."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
from exact_attention_91_gb300 import inputs as fin  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank
        out[rank] = bench.max_over_ranks(ms, world, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_over_gloo():
    world = 2
    ctx = torch.multiprocessing.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_ranks_get_independent_batches_of_one_shape():
    w = fin.custom(1, 2, 64, 64, False, seed=9)
    w0, w1 = bench.rank_workload(w, 0, 2), bench.rank_workload(w, 1, 2)
    assert (w0.B, w0.H, w0.N, w0.d) == (w1.B, w1.H, w1.N, w1.d)
    assert w0.seed != w1.seed
    assert bench.rank_workload(w, 0, 1) is w
    x0, x1 = fin.make_inputs(w0), fin.make_inputs(w1)
    assert not (x0.q == x1.q).all()


def test_throughput_counts_every_rank():
    assert bench.job_throughput(1, 10, 1e12, 1000.0) == pytest.approx(10.0)
    assert bench.job_throughput(4, 10, 1e12, 1000.0) == pytest.approx(40.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 1, 0
    assert bench.run_reference(Args(), fin.WORKLOADS["tiny"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line of the bench contract:
    the oracle's throughput on the same workload, its cores and sample, and an
    e2e object with no host-device copies."""
    import json
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 1.5)

    class Args:
        steps, warmup = 2, 1
    assert bench.run_reference(Args(), fin.WORKLOADS["tiny"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == "tiny" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_is_reported_only_for_the_captured_kernel(monkeypatch, tmp_path):
    """roofline.traffic comes from the committed ncu capture only while the
    kernel sources still hash to the captured build; otherwise it is null."""
    import json
    t = tmp_path / "traffic.json"
    t.write_text(json.dumps({"llm_prefill": {"bytes_per_launch": 123, "kernel_sha": bench.kernel_sha()},
                             "long_sequence": {"bytes_per_launch": 456, "kernel_sha": "0" * 16}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(t))
    assert bench.load_traffic("llm_prefill") == 123
    assert bench.load_traffic("long_sequence") is None      # captured on other kernel sources
    assert bench.load_traffic("max_shift") is None          # never captured
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.load_traffic("llm_prefill") is None


def test_strong_scaling_ranks_share_one_problem_by_heads():
    """--scaling strong: the ranks' head ranges cover the one workload's
    heads once, their inputs are those heads' slices of its inputs, and the
    job counts the workload's flops once per step (weak: once per rank)."""
    w = fin.custom(2, 3, 64, 64, True, seed=11)
    x = fin.make_inputs(w)
    BH = w.B * w.H
    got = []
    for rank in range(4):
        _, (q, k, v), B, H, job = bench.local_problem(w, rank, 4, "strong")
        assert B == 1 and q.shape == (1, H, w.N, w.d) and job == w.flops
        got.append(q[0])
    assert np.array_equal(np.concatenate(got), x.q.reshape(BH, w.N, w.d))
    _, (q, _, _), B, H, job = bench.local_problem(w, 1, 4, "weak")
    assert (B, H) == (w.B, w.H) and job == 4 * w.flops and not np.array_equal(q, x.q)
    assert bench.workload_config(w, 4, "strong")["parallelism"].startswith("one problem")
