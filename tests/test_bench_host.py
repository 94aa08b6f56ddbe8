"""Host-side logic of bench.py (CPU only): which kernel sources a workload's
measurement depends on, and when a committed ncu traffic figure applies."""
import os

import bench
import workloads


def test_every_workload_maps_to_existing_kernel_sources():
    for name, w in workloads.WORKLOADS.items():
        units = bench.kernel_units(w)
        for u in units:
            assert os.path.exists(os.path.join(bench.CSRC, u)), (name, u)
        closure = bench._include_closure([os.path.join(bench.CSRC, u) for u in units])
        assert all(os.path.dirname(f) == bench.CSRC for f in closure)
        assert len(bench.source_hash(w)) == 12


def test_source_hash_separates_operations():
    W = workloads.WORKLOADS
    h = {n: bench.source_hash(W[n]) for n in ("fused_add_rmsnorm_bf16_8192x4096",
                                              "layernorm_bf16_8192x4096",
                                              "softmax_sweep_f32_N4096",
                                              "logsumexp_argmax_vocab_bf16_64x152064")}
    assert len(set(h.values())) == len(h)
    # same kernels, same hash: the sweep rows all run the fp32 softmax units
    assert bench.source_hash(W["softmax_sweep_f32_N32"]) == h["softmax_sweep_f32_N4096"]


def test_traffic_applies_only_to_the_same_sources_and_plan(tmp_path, monkeypatch):
    w = workloads.WORKLOADS["softmax_sweep_f32_N4096"]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.md").write_text(
        "| workload | source hash | plan | kernel | traffic | algorithmic |\n|---|---|---|---|---|---|\n"
        f"| {w.name} | {bench.source_hash(w)} | `rows g=256 ept=16 vec` | k | 480,000,000 | 1 |\n"
        f"| {w.name} | 000000000000 | `rows g=128 ept=16 vec` | k | 7 | 1 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic(w, "rows g=256 ept=16 vec") == 480_000_000
    assert bench.profiled_traffic(w, "rows g=128 ept=16 vec") is None   # stale sources
    assert bench.profiled_traffic(w, "rows g=512 ept=16 vec") is None   # other plan


def test_quantiles_and_the_metric_configurations():
    v = [float(i) for i in range(21)]
    assert bench.quantile(v, 0.5) == 10.0
    assert bench.quantile(v, 0.1) == 2.0 and bench.quantile(v, 0.9) == 18.0
    assert bench.quantile([3.0, 1.0], 0.5) == 2.0
    # every configuration of the metric is a workload the suite times
    assert len(bench.BASELINE_CONFIGS) == 10
    for tag, name in bench.BASELINE_CONFIGS:
        assert name in workloads.WORKLOADS, (tag, name)


def test_cpu_baseline_reports_all_cores_and_one(monkeypatch):
    w = workloads.WORKLOADS["rmsnorm_f32_64x3584"]
    cb = bench.cpu_baseline_for(w, budget_s=0.05)
    assert cb["cores"] == (os.cpu_count() or 1) and cb["nproc"] == cb["cores"]
    assert cb["single_thread"]["cores"] == 1 and cb["value"] > 0 and cb["single_thread"]["value"] > 0
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
