"""Host logic of the benchmark (no GPU): the flop count of a layer step, the
grouping of a layer's projections, the roofline arithmetic of the dominant
kernel kind, the workload names, and that traffic figures are read only while
the library sources they were taken on are unchanged.

The flop counts are checked against the definitions written out (forward
2MNK + 2Mr(N+K), backward dX 2MNK + 2MKr, V 2MNr, dA 2MKr, dB 2MNr), so that a
dropped term, a transposed shape or a wrong factor in bench.py fails here.
"""
import json
import os

import pytest

import bench
from bit_quantized_lora_double_b300 import synth


def test_step_flops_is_the_sum_of_the_passes():
    wl = synth.WORKLOADS[bench.WORKLOAD]
    M, r = wl["M"], wl["r"]
    want = 0
    for _, n, k in wl["projections"]:
        fwd = 2 * M * n * k + 2 * M * k * r + 2 * M * r * n        # X W'^T, U = X A^T, U B^T
        dx = 2 * M * n * k + 2 * M * n * r + 2 * M * r * k        # dY W', V = dY B, V A
        grads = 2 * M * r * k + 2 * M * n * r                     # dA = V^T X, dB = dY^T U
        want += fwd + dx + grads
    assert bench.step_flops(M, wl["projections"], r) == want


def test_kind_flops_cover_the_step():
    # the GEMM kinds plus the side path (U, V, dA, dB) add up to the step
    wl = synth.WORKLOADS[bench.LAYER8B]
    M, r = wl["M"], wl["r"]
    side = sum(2 * M * k * r + 2 * M * n * r + 2 * M * r * k + 2 * M * n * r for _, n, k in wl["projections"])
    gemm = sum(bench.KIND_FLOPS[kind](M, n, k, r) for kind in ("fwd_gemm", "dx_gemm")
               for _, n, k in wl["projections"])
    assert gemm + side == bench.step_flops(M, wl["projections"], r)


def test_groups_of_the_layer():
    wl = synth.WORKLOADS[bench.WORKLOAD]
    names = [nm for nm, _, _ in wl["projections"]]
    groups = bench.groups_of([{"name": nm} for nm in names])
    assert [[names[i] for i in g] for g in groups] == [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
    assert sorted(i for g in groups for i in g) == list(range(len(names)))


def test_roofline_of_scales_to_the_graph_step():
    wl = synth.WORKLOADS[bench.LAYER8B]
    M, r, P = wl["M"], wl["r"], wl["projections"]
    pk = dict(hbm=6500.0, bf16=1756.5, bf16_sus=1352.2, src="measured")
    kind_ms = {"fwd_gemm": 0.8, "dx_gemm": 0.9, "lora_pre": 0.15, "grads": 0.15}
    kind_n = {"fwd_gemm": 4, "dx_gemm": 4, "lora_pre": 8, "grads": 4}
    rf = bench.roofline_of(kind_ms, kind_n, 1.8, M, P, r, pk, {"reasons": ["sw_power_cap"]})
    assert rf["kernel"] == "dx_gemm"
    assert rf["scale_to_graph_step"] == pytest.approx(1.8 / 2.0)
    fl = sum(2 * M * n * k + 2 * M * k * r for _, n, k in P)
    assert rf["flops_per_step"] == fl
    assert rf["achieved"] == pytest.approx(fl / (0.9 * 0.9e-3) / 1e12)
    assert rf["frac"] == pytest.approx(rf["achieved"] / pk["bf16"])
    assert "sw_power_cap" in rf["peak_note"]


def test_workload_names_are_the_same_for_both_arms():
    wl = synth.WORKLOADS[bench.WORKLOAD]
    name = bench.workload_name(wl)
    assert wl["name"] in name and "r=64" in name


def test_traffic_follows_the_sources(tmp_path, monkeypatch):
    # figures are returned only while the sources hash matches the file's
    d = {"sources_sha256": bench.sources_sha256(), "per_launch_bytes": {"dx_gemm": 123}}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "roofline_traffic.json").write_text(json.dumps(d))
    real = bench.sources_sha256()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "sources_sha256", lambda: real)
    assert bench.measured_traffic("dx_gemm") == 123
    monkeypatch.setattr(bench, "sources_sha256", lambda: "0" * 64)
    assert bench.measured_traffic("dx_gemm") is None


def test_committed_traffic_file():
    # the committed figures name the sources they were taken on and the
    # command that took them; bench.py reports them only while those match
    p = os.path.join(bench.ROOT, "profiles", "roofline_traffic.json")
    d = json.load(open(p))
    assert len(d["sources_sha256"]) == 64 and "ncu" in d["command"]
    assert set(d["per_launch_bytes"]) == {"fwd_gemm", "dx_gemm"}
    assert all(v > 0 for v in d["per_launch_bytes"].values())
