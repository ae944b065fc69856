"""Host-side arithmetic of bench.py (CPU only): the algorithmic bytes and
flops the roofline divides by, the choice of bound and kernel, and the
lookup of committed ncu traffic by kernel-source hash."""

import json

import pytest

import bench
from weight_quantized_moe_gb300 import synth

W = synth.WORKLOADS


def test_algorithmic_bytes_mixtral_decode_t64():
    """Mixtral-shaped W8A16 at T=64, all 8 experts touched.  Written out by
    hand: w13 is 2·14336·4096 int8 codes plus 2·14336 float32 scales per
    expert; the gate/up launch also reads x (64·4096 bf16) and writes act
    (128 slots · 14336 bf16); the down launch reads w2 (4096·14336 codes,
    4096 scales), act, and writes 128 · 4096 float32 partial sums."""
    w = bench.algorithmic_work(W["mixtral_decode"], 64, touched=list(range(8)))
    w13 = 2 * 14336 * 4096 + 4 * 2 * 14336
    w2 = 4096 * 14336 + 4 * 4096
    assert w["gemm1"]["bytes"] == 8 * w13 + 64 * 4096 * 2 + 128 * 14336 * 2 == 944_635_904
    assert w["gemm2"]["bytes"] == 8 * w2 + 128 * 14336 * 2 + 128 * 4096 * 4
    assert w["gemm1"]["flops"] == 4 * 128 * 14336 * 4096
    assert w["gemm2"]["flops"] == 2 * 128 * 14336 * 4096
    assert w["layer"]["bytes"] == w["gemm1"]["bytes"] + w["gemm2"]["bytes"]


def test_algorithmic_bytes_w4a16_counts_packed_codes_scales_and_zeros():
    wl = W["w4a16"]  # E=64, k=6, H=2048, I=1408, gs=128, zero points
    w = bench.algorithmic_work(wl, 1, touched=[3, 9, 17, 20, 41, 60])
    G13, G2 = 2048 // 128, 1408 // 128
    w13 = 1408 * 2048 + 2 * 2 * 1408 * G13 + 1408 * G13   # uint4 codes, f16 scales, packed zeros
    w2 = 2048 * 1408 // 2 + 2 * 2048 * G2 + 1024 * G2
    assert w["gemm1"]["bytes"] == 6 * w13 + 2048 * 2 + 6 * 1408 * 2
    assert w["gemm2"]["bytes"] == 6 * w2 + 6 * 1408 * 2 + 6 * 2048 * 4


PEAKS = {"hbm_gbs": 6697.5, "bf16_tflops": 1873.2, "bf16_tflops_sustained": 1700.0,
         "source": "measured"}


def test_roofline_decode_is_hbm_bound_on_the_slowest_gemm():
    wl = W["mixtral_decode"]
    prof = {"gemm1": (1.52, 10), "gemm2": (0.82, 10), "align": (0.1, 10)}  # ms total, launches
    r = bench.roofline_of(wl, 64, prof, list(range(8)), PEAKS, long_run=False)
    assert r["kernel"] == "gemm1" and r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["ms_per_launch"] == pytest.approx(0.152)
    assert r["achieved"] == pytest.approx(944_635_904 / 0.152e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6697.5)
    assert r["traffic"] is None  # no workload key given


def test_roofline_prefill_is_tensor_bound_burst_or_sustained():
    wl = W["mixtral_prefill"]
    prof = {"gemm1": (15.5, 10), "gemm2": (8.6, 10)}
    flops = 4 * 4096 * 2 * 14336 * 4096
    for long_run, peak in ((False, 1873.2), (True, 1700.0)):
        r = bench.roofline_of(wl, 4096, prof, list(range(8)), PEAKS, long_run=long_run)
        assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
        assert r["achieved"] == pytest.approx(flops / 1.55e-3 / 1e12)
        assert r["peak"] == peak and r["frac"] == pytest.approx(r["achieved"] / peak)


def test_roofline_picks_the_one_launch_layer_when_it_ran():
    wl = W["fine"]
    prof = {"layer": (0.92, 10), "combine": (0.11, 10)}
    r = bench.roofline_of(wl, 512, prof, list(range(33)), PEAKS, long_run=False)
    assert r["kernel"] == "layer"
    work = bench.algorithmic_work(wl, 512, list(range(33)))["layer"]
    assert r["algorithmic_bytes_per_launch"] == work["bytes"]


def test_ncu_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    sha = bench.kernel_source_sha()
    table = {"gemm1@mixtral_decode_T64": {"dram_bytes_per_launch": 945_200_000, "source_sha": sha},
             "gemm2@mixtral_decode_T64": {"dram_bytes_per_launch": 480_000_000,
                                          "source_sha": "0" * 16}}
    (tmp_path / "traffic.json").write_text(json.dumps(table))
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.ncu_traffic("gemm1", "mixtral_decode_T64") == 945_200_000
    assert bench.ncu_traffic("gemm2", "mixtral_decode_T64") is None   # other sources
    assert bench.ncu_traffic("layer", "mixtral_decode_T64") is None   # not captured
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path / "absent"))
    assert bench.ncu_traffic("gemm1", "mixtral_decode_T64") is None


def test_measured_peaks_fall_back_when_the_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.measured_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["bf16_tflops"] == 1900.0
