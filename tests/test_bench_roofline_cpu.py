"""The benchmark's roofline block is self-consistent (CPU, synthetic timings):
every fraction it prints is a quotient of its own kernel times, the step's
8 N V D flops and the measured peaks, so a reader can recompute `frac` from the
line's `kernels` block and MEASURED_PEAKS.json. The DRAM-traffic record is found
only for the kernel sources and plan it was captured with."""
import json
import os

import pytest

import bench


def _synthetic(steps=3):
    # one LSE GEMM, 8 chunks of (gradient, dH + dW), merge, reduce, rounding per step
    per_launch = {"lse_gemm": 4.9, "lse_merge": 0.02, "loss_reduce": 0.015, "grad_gemm": 0.63,
                  "dwdh_gemm": 1.28, "dh_round": 0.031}
    launches = {"lse_gemm": 1, "lse_merge": 1, "loss_reduce": 1, "grad_gemm": 8, "dwdh_gemm": 8,
                "dh_round": 1}
    n_kind = {k: launches[k] * steps for k in launches}
    per_kind = {k: per_launch[k] * n_kind[k] for k in launches}
    kernel_ms = {k: per_kind[k] / steps for k in launches}
    return kernel_ms, n_kind, per_kind, steps


def test_fractions_are_quotients_of_the_block_and_the_peaks():
    N, V, D = 8192, 128256, 4096
    peaks = bench.load_peaks()
    kernel_ms, n_kind, per_kind, steps = _synthetic()
    r = bench.make_roofline(N, V, D, kernel_ms, n_kind, per_kind, steps, peaks, 1.0e9)
    k = r["kernels"]
    assert r["peak"] == peaks["bf16_tflops"]
    # the dominant kernel: two 2 N V D products over its time per step
    want = 2 * (2.0 * N * V * D) / (k["dwdh_gemm"]["ms_per_step"] / 1e3) / 1e12
    assert r["achieved"] == pytest.approx(want, rel=1e-12)
    assert r["achieved"] == pytest.approx(k["dwdh_gemm"]["tflops"], rel=1e-12)
    assert r["frac"] == pytest.approx(r["achieved"] / peaks["bf16_tflops"], rel=1e-12)
    assert r["frac_of_sustained"] == pytest.approx(
        r["achieved"] / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), rel=1e-12)
    for name, kern in (("lse", "lse_gemm"), ("gradient", "grad_gemm"), ("dW + dH", "dwdh_gemm")):
        p = r["products"][name]
        assert p["tflops"] == pytest.approx(k[kern]["tflops"], rel=1e-12)
        assert p["frac"] == pytest.approx(k[kern]["tflops"] / r["peak"], rel=1e-12)
    assert sum(v["share"] for v in k.values()) == pytest.approx(1.0, rel=1e-12)
    assert r["launches_per_step"] == 8
    assert r["ms_per_launch_avg"] == pytest.approx(1.28, rel=1e-12)
    assert r["flops_per_launch_avg"] == pytest.approx(2 * 2.0 * N * V * D / 8, rel=1e-12)
    assert r["traffic"] == 1.0e9


def test_traffic_record_matches_only_its_kernel_sources_and_plan():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.json")
    with open(path) as f:
        records = json.load(f)["records"]
    sha = bench.kernel_source_sha()
    current = [r for r in records if r["kernel_sha"] == sha]
    for r in current:
        assert bench.measured_traffic(r["kernel"], r["workload"], r["v_chunk"]) == r["bytes_per_launch"]
        assert bench.measured_traffic(r["kernel"], r["workload"], r["v_chunk"] + 256) is None
    assert bench.measured_traffic("flce_gemm_kernel<EPI_F32>", "no_such_workload", 16128) is None


def test_hbm_passes_report_algorithmic_bandwidth():
    """The passes around the GEMMs carry their algorithmic bytes (one read of what
    each reads, one write of what each writes) and GB/s = bytes / time, as a
    fraction of the measured copy bandwidth; the dH rounding only when there are
    several chunks."""
    N, V, D = 8192, 128256, 4096
    peaks = bench.load_peaks()
    kernel_ms, n_kind, per_kind, steps = _synthetic()
    plan = {"v_splits": 101, "n_chunks": 8, "n_block": N}
    nbytes = bench.small_pass_bytes(N, D, plan)
    assert nbytes["dh_round"] == 6 * N * D                      # fp32 read + bf16 write
    assert nbytes["loss_reduce"] == 8 * N                       # NLL + labels
    assert nbytes["lse_merge"] == 8 * 101 * N + 32 * N          # partials + zt, labels + 3 outputs
    r = bench.make_roofline(N, V, D, kernel_ms, n_kind, per_kind, steps, peaks, None,
                            hbm_bytes_per_step=nbytes)
    for k in ("lse_merge", "loss_reduce", "dh_round"):
        kk = r["kernels"][k]
        assert kk["bound"] == "hbm"
        assert kk["gbs"] == pytest.approx(nbytes[k] / (kernel_ms[k] / 1e3) / 1e9, rel=1e-12)
        assert kk["frac_of_hbm"] == pytest.approx(kk["gbs"] / peaks["hbm_gbs"], rel=1e-12)
    assert "gbs" not in r["kernels"]["lse_gemm"]
    assert "dh_round" not in bench.small_pass_bytes(N, D, dict(plan, n_chunks=1))
