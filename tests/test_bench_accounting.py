"""CPU checks of the bench's roofline accounting: the algorithmic bytes and FLOPs of the
expert GEMMs, the kernel it names for each workload, the peak it divides by, and the
committed DRAM-traffic figure's source-hash guard."""

import numpy as np

import bench
import workloads


def _counts(cfg, active):
    c = np.zeros(cfg.E, dtype=np.int64)
    c[:active] = 1
    return c


def test_gate_up_bytes_at_v3_from_tensor_sizes():
    cfg, T = workloads.V3, workloads.V3.T
    active = 153                                          # + the shared expert = 154
    rows = T * cfg.K + T                                  # 36,864 expert rows
    weights = 154 * (4096 * 7168 + 32 * 56 * 4)           # E4M3 W1|W3 and their 128x128 scales
    rows_in = rows * 7168 + rows * 56 * 4                 # gathered E4M3 rows and 1x128 scales
    h_out = rows * 2048 + rows * 16 * 4                   # E4M3 h and its scales
    assert bench.gate_up_bytes(cfg, _counts(cfg, active), T) == weights + rows_in + h_out
    assert bench.gate_up_flops(cfg, T) == 2 * rows * 4096 * 7168


def test_down_bytes_at_v3_from_tensor_sizes():
    cfg, T = workloads.V3, workloads.V3.T
    rows = T * cfg.K + T
    weights = 154 * (7168 * 2048 + 56 * 16 * 4)
    h_in = rows * 2048 + rows * 16 * 4
    y_out = rows * 7168 * 2                               # BF16 expert outputs
    assert bench.down_bytes(cfg, _counts(cfg, 153), T) == weights + h_in + y_out


def test_gate_up_kernel_follows_the_library_rule():
    # segments averaging at most 16 rows (rows <= 16 * (E + 1)) run on the swapped-operand
    # kernel in either recipe; anything larger on the recipe's grouped GEMM
    assert "swap" in bench.gate_up_kernel_name(workloads.DECODE, 128, False, "auto")
    assert "swap" in bench.gate_up_kernel_name(workloads.DECODE, 128, True, "auto")
    assert bench.gate_up_kernel_name(workloads.V3, 4096, False, "auto").startswith(
        "fp8_gemm_kernel<SwiGLU>")
    assert bench.gate_up_kernel_name(workloads.V3, 4096, True, "auto").startswith(
        "fp8_mx_gemm_kernel<SwiGLU>")
    assert "swap" in bench.gate_up_kernel_name(workloads.V3, 4096, False, "swap")
    # the boundary itself: 16 rows per segment on average
    cfg = workloads.DECODE
    T_edge = 16 * (cfg.E + 1) // (cfg.K + 1)
    assert "swap" in bench.gate_up_kernel_name(cfg, T_edge, False, "auto")
    assert "swap" not in bench.gate_up_kernel_name(cfg, T_edge + 1, False, "auto")


def test_fp8_peak_takes_the_sustained_figure_only_under_the_power_cap_or_low_clocks():
    pk = {"hbm_gbs": 6494.3, "bf16_tflops": 1747.0, "bf16_tflops_sustained": 1379.0}
    burst, _ = bench.fp8_peak_for(pk, {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []})
    capped, _ = bench.fp8_peak_for(pk, {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0,
                                        "reasons": ["sw_power_cap"]})
    slow, _ = bench.fp8_peak_for(pk, {"sm_mhz": 1700.0, "sm_max_mhz": 2032.0, "reasons": []})
    assert burst == 2 * 1747.0
    assert capped == slow == 2 * 1379.0


def test_kernel_roofline_takes_the_longer_bound():
    pk = {"hbm_gbs": 6494.3}
    # 4.87 GB and 2.16 TFLOP in 1.56 ms against a 3,494 TF peak: HBM-bound (0.75 vs 0.62 ms)
    r = bench.kernel_roofline("k", 4_872_919_040, 2_164_663_517_184, 1.56, pk, 3494.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 4_872_919_040 / 1.56e-3 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6494.3) < 1e-4
    # the same work against a tenth of the tensor peak: tensor-bound
    r = bench.kernel_roofline("k", 4_872_919_040, 2_164_663_517_184, 1.56, pk, 349.4)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"


def test_committed_traffic_is_dropped_when_the_kernel_source_changes(monkeypatch):
    # the committed summary carries the hash of the kernel source it was measured on
    assert bench.committed_traffic() is not None
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    assert bench.committed_traffic() is None
