"""Host arithmetic of bench.py: the roofline's algorithmic bytes and GEMM FLOPs of the
headline workload worked out by hand, and the ncu traffic tables (reported only while the
kernel sources match the capture)."""

import pytest

import bench
from tile_level_sync_gb300 import synth


def test_headline_algorithmic_bytes_and_flops():
    # X [256,12288], W1 [12288,6144], H [256,6144] written and read, W2 [6144,12288],
    # Y [256,12288], all bf16
    M, K, N1, N2 = 256, 12288, 6144, 12288
    by_hand = 2 * (M * K + K * N1 + 2 * M * N1 + N1 * N2 + M * N2)
    wl = synth.WORKLOADS["gpt3_mlp_m256"]
    assert bench.algorithmic_bytes(wl) == by_hand == 320_864_256
    assert wl.gemm_flops() == 2 * M * K * N1 + 2 * M * N1 * N2


def test_swiglu_counts_both_producer_weights():
    wl = synth.WORKLOADS["swiglu_m256"]
    d = wl.dims
    by_hand = 2 * (d["M"] * d["K"] + d["K"] * 2 * d["N1"] + 2 * d["M"] * d["N1"] + d["N1"] * d["N2"]
                   + d["M"] * d["N2"])
    assert bench.algorithmic_bytes(wl) == by_hand


def test_traffic_tables_name_real_workloads_and_follow_the_sources(monkeypatch):
    for key in bench.NCU_TRAFFIC:
        assert key[0] in synth.WORKLOADS and key[2] in ("persistent", "pdl")
    for name, (traffic, _) in bench.NCU_ROW_TRAFFIC.items():
        assert name in synth.WORKLOADS and traffic > 0
    key = ("gpt3_mlp_m256", "ROW", "persistent", 256, 2)
    traffic, src = bench.NCU_TRAFFIC[key]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: src)
    assert bench.measured_traffic(*key) == traffic
    # once the kernels change, the recorded counters no longer describe them
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.measured_traffic(*key) is None
    assert bench.measured_traffic("gpt3_mlp_m256", "TILE", "pdl", 256, 2) is None


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_every_workload_has_positive_work(name):
    wl = synth.WORKLOADS[name]
    assert wl.gemm_flops() > 0 and bench.algorithmic_bytes(wl) > 0
