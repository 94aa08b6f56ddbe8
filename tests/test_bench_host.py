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
