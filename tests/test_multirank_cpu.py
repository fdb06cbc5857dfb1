"""The bench's multi-rank path on CPU: two gloo ranks, one process each.

The path has no exchange step (replicas only); what crosses ranks is the
timing: the job time is the slowest rank's, and the whole-job throughput
counts every rank's batch.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r + 1) ms for the device loop and (10 - r) ms end to end
    got = bench.max_over_ranks([rank + 1.0, 10.0 - rank])
    results[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        assert dict(results) == {0: [2.0, 10.0], 1: [2.0, 10.0]}


def test_whole_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.aggregate_gbs(1, 1e9, 10, 1000.0)     # 10 GB in 1 s
    assert one == pytest.approx(10.0)
    assert bench.aggregate_gbs(4, 1e9, 10, 1000.0) == pytest.approx(40.0)
    assert bench.max_over_ranks([3.0, 1.0]) == [3.0, 1.0]   # no process group: unchanged


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_gqa_06_gb300 import workloads as W
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 3, 3
    assert bench.run_reference(Args(), W.make_workload("tiny"), 4) is None


def test_reference_arm_line_keeps_the_contract(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_gqa_06_gb300 import workloads as W
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)

    class Args:
        steps, warmup = 2, 1
    line = bench.run_reference(Args(), W.make_workload("tiny"), 4)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("tiny")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_cpu_baseline_reports_all_cores_and_one_thread():
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_gqa_06_gb300 import workloads as W
    cb = bench.cpu_baseline(W.make_workload("tiny"), 4, budget_s=0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0 and cb["cores"] >= 1
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["unit"] == "GB/s"


def test_output_check_of_the_cpu_leg_reports_max_abs_error():
    """check_outputs (run in the CPU-baseline leg) puts each workload's
    max-abs error against the oracle into the line and its per_config entry."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    from paged_kv_gqa_06_gb300 import workloads as W
    wl = W.make_workload("tiny")
    t = wl.layer(0)
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle.paged_kv_append(t["k_new"], t["v_new"], wl.slot_mapping, kc, vc)
    ref = oracle.paged_gqa_decode(t["q"], kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    got = ref.copy()
    got[1, 2, 3] += 1e-3
    line = {"config": {"workload": "tiny: x"}, "max_abs_err": None, "per_config": {"tiny": {"max_abs_err": None}}}
    bench.check_outputs(line, {"tiny": (wl, t, got)})
    assert line["max_abs_err"] == pytest.approx(1e-3, rel=1e-9)
    assert line["per_config"]["tiny"]["max_abs_err"] == line["max_abs_err"]
    got[0, 0, 0] = np.nan
    bench.check_outputs(line, {"tiny": (wl, t, got)})
    assert line["max_abs_err"] == float("inf")


def test_reference_arm_has_the_gpu_arms_config():
    """Both arms state the same config (workload, sizes, launch and L2 handling)."""
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_gqa_06_gb300 import workloads as W
    wl = W.make_workload("qwen3_4b")

    class Args:
        steps, warmup, graphs = 20, 5, True
    cfg = bench._config_dict(wl, Args(), 2)
    assert cfg["l2"].startswith("no flush") and cfg["launch"] == "CUDA graphs of 20 steps replayed"
    assert cfg["bytes_per_step"] == wl.bytes_decode(2) and cfg["layers"] == 1
    small = bench._config_dict(W.make_workload("qwen3_0_6b"), Args(), 2)
    assert "copies of the KV pools rotated" in small["l2"]


def test_profile_traffic_is_read_only_for_matching_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary only when the
    summary names the hash of the sources the bench is running."""
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    prof = tmp_path / "profiles" / "k.md"
    prof.write_text("# k\n\n- source_sha256: `abc123`\n- dram_bytes_per_prefill_call: `1234`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic_from_profile("abc123", "", "k.md", "dram_bytes_per_prefill_call") == 1234
    assert bench._traffic_from_profile("other", "", "k.md", "dram_bytes_per_prefill_call") is None
    assert bench._traffic_from_profile("abc123", "", "k.md", "dram_bytes_per_decode_call") is None
    assert bench._traffic_from_profile("abc123", "", "missing.md") is None
    # each latency-bound workload reads its own key from the shared summary
    monkeypatch.setattr(bench, "_decode_source_hash", lambda: "abc123")
    (tmp_path / "profiles" / bench.LATENCY_PROFILE).write_text(
        "- source_sha256: `abc123`\n- dram_bytes_per_decode_call_qwen3_0_6b: `11`\n"
        "- dram_bytes_per_decode_call_skewed: `22`\n")
    assert bench._decode_traffic("qwen3_0_6b", "online") == 11
    assert bench._decode_traffic("skewed", "online") == 22
    assert bench._decode_traffic("skewed", "two_pass") is None
    assert bench._decode_traffic("cb36", "online") is None
    monkeypatch.undo()
    # the hashes cover the kernel sources and differ between the two paths
    monkeypatch.setattr(bench, "ROOT", ROOT)
    assert bench._decode_source_hash() != bench._prefill_source_hash()
    assert len(bench._decode_source_hash()) == 16
