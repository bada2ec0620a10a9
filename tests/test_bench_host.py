"""Host-side logic of bench.py that needs no GPU: the stored DRAM-traffic figure of the
dominant GEMM is reported only for the kernel, size and sources it was captured on,
and the reference arm does its work on rank 0 alone."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_only_for_the_captured_kernel_and_size():
    assert bench.dominant_traffic("q.fwd", 8192) is None
    assert bench.dominant_traffic("gate_up.fwd", 4096) is None


def test_traffic_follows_the_source_hash(monkeypatch):
    t = dict(bench.GU_FWD_TRAFFIC)
    t["sha256"] = bench.sources_sha256(t["sources"])
    monkeypatch.setattr(bench, "GU_FWD_TRAFFIC", t)
    assert bench.dominant_traffic("gate_up.fwd", 8192) == t["bytes"]
    t["sha256"] = "0" * 64  # any change to the sources drops the figure
    assert bench.dominant_traffic("gate_up.fwd", 8192) is None


def test_traffic_figure_is_plausible():
    # one launch moves the operands once and the output once: Xq 14.2 MB, W 28.3 MB,
    # LoRA operands 1.6 MB, Y 268.4 MB; writes still in L2 at the end are not counted
    algorithmic = 14.2e6 + 28.3e6 + 1.6e6 + 268.4e6
    assert 0.7 * algorithmic < bench.GU_FWD_TRAFFIC["bytes"] < 1.1 * algorithmic


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 3, 2

    def boom(*a, **k):
        raise AssertionError("rank 1 must not run the oracle")

    monkeypatch.setattr(bench.wl, "layer3b", boom)
    assert bench.run_reference(Args()) == 0


def test_both_arms_report_one_configuration():
    # the GPU arm asserts its stack matches this dictionary; it must describe the
    # layer-3b workload the stack is built from
    cfg = bench.step_config(1)
    d = bench.wl.layer3b()
    m = d["x"].shape[0]
    flops = 2.0 * sum(2.0 * m * d[k].W.shape[0] * d[k].W.shape[1] for k in bench.PROJS)
    assert cfg["tokens_per_step"] == m and cfg["gemm_flops_per_step"] == flops
    assert cfg["workload"] == "layer-3b" and bench.step_config(4)["parallelism"] == "replicas x4"
