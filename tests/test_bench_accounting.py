"""The benchmark's work accounting on the CPU: algorithmic bytes follow the
method's data sizes (one read of each input, int4 codes at half a byte, int8
codes at one byte, the scales), the maximum pre-passes and the layout pass
are credited with nothing, and a GEMM's roof is max(ops / tensor peak,
bytes / HBM peak)."""
import importlib.util
import os

import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_acct",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
         "source": "test"}


def test_hq_rows_bytes_on_vitb_qkv():
    b = _bench()
    wl = workloads.WORKLOADS[1]        # T 12608, Cout 2304, bf16, per-token
    kind, nbytes = b.algorithmic("hq_rows_quant", wl)
    # g_y read (bf16) + packed int4 codes + one fp32 scale per token
    assert kind == "hbm"
    assert nbytes == 12608 * 2304 * 2 + 12608 * 2304 // 2 + 4 * 12608 == 72_672_512


def test_prepasses_and_layout_pass_are_not_credited():
    b = _bench()
    wl = workloads.WORKLOADS[2]
    for k in ("hq_rows_amax", "hq_cols_amax", "hla_gy_amax", "hla_x_amax", "widen_xbar"):
        assert b.algorithmic(k, wl)[1] == 0, k
    T, Cin, Cout, Tp = wl.T, wl.Cin, wl.Cout, wl.Tp
    assert b.algorithmic("hla_gy_quant", wl)[1] == T * Cout * 2 + Cout * Tp + 4
    assert b.algorithmic("hla_x_quant", wl)[1] == T * Cin * 2 + Cin * Tp + 4
    assert b.algorithmic("hla_x_quant", wl, xbar_bits=4)[1] == T * Cin * 2 + Cin * Tp // 2 + 4
    assert b.algorithmic("hq_cols_quant", wl)[1] == Cout * Cin * 2 + Cin * Cout // 2 + 4


def test_kernel_table_fraction_reproduces_by_hand():
    b = _bench()
    wl = workloads.WORKLOADS[1]
    launches = [("hq_rows_quant", 0.060), ("hq_rows_quant", 0.066),
                ("gemm_gx_tc", 0.025), ("hla_gy_amax", 0.02)]
    kernels, rows = b.kernel_table(launches, wl, PEAKS)
    k = kernels["hq_rows_quant"]
    assert k["avg_us"] == pytest.approx(63.0)
    assert k["frac"] == pytest.approx(72_672_512 / 63e-6 / 1e9 / 6800.0)
    assert kernels["hla_gy_amax"]["frac"] == 0.0
    # ViT-B qkv g_x: 44.6 G ops over 3.8 POPS exceeds 46 MB over 6.8 TB/s
    g = kernels["gemm_gx_tc"]
    assert g["bound"] == "tensor" and g["peak"] == pytest.approx(3800.0)
    assert g["frac"] == pytest.approx(2 * 12608 * 768 * 2304 / 25e-6 / 1e12 / 3800.0)
    assert set(rows) == {"a2", "a4", "a5"}
    assert rows["a2"]["us"] == pytest.approx(63.0)


def test_gemm_output_bound_for_resnet_gx():
    b = _bench()
    wl = workloads.WORKLOADS[4]        # T 50176, Cin 2304, Cout 256: fp32 g_x dominates
    work = b.algorithmic("gemm_gx_tc", wl)
    ops, nbytes = work[1], work[2]
    assert nbytes == 50176 * 256 // 2 + 2304 * 256 // 2 + 50176 * 2304 * 4
    r = b.roofline_of("gemm_gx_tc", work, 100e-6, PEAKS)
    assert ops / 3800e12 < nbytes / 6800e9
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(nbytes / 100e-6 / 6800e9)


def test_default_workload_is_the_largest_layer():
    b = _bench()
    big = max(workloads.WORKLOADS, key=lambda w: w.T * w.Cin * w.Cout)
    assert b.DEFAULT_WORKLOAD is big and b.parse_args([]).workload == big.name


def test_fused_reader_credited_once_with_both_codes():
    """The fused reader of g_y (per-tensor g_y scale) reads g_y once for both
    quantizers: its codes pass carries one read plus the int4 HQ codes and the
    int8 HLA codes, its maxima pass nothing; its row combines a2 and a5."""
    b = _bench()
    wl = workloads.WORKLOADS[4]        # ResNet-50 im2col, per-tensor g_y
    T, Cout, Tp = wl.T, wl.Cout, wl.Tp
    assert b.algorithmic("gy_fused_amax", wl)[1] == 0
    assert b.algorithmic("gy_fused_quant", wl)[1] == T * Cout * 2 + T * Cout // 2 + 4 + Cout * Tp + 4
    kernels, rows = b.kernel_table([("gy_fused_amax", 0.02), ("gy_fused_quant", 0.04)], wl, PEAKS)
    assert rows["a2+a5"]["kernels"] == ["gy_fused_amax", "gy_fused_quant"]
    assert "a2" not in rows and "a5" not in rows
