"""Parity at the full workload sizes, through the same entry points and
launch configuration the benchmark times.

The oracle recomputes every code and scale (bit-exact) where per-tensor
scales need the whole tensor, and the integer GEMM rows of a seeded sample
of tokens / output channels; the tensor-core GEMMs are also compared in
full with the CUDA-core reference GEMM (integer sums, bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import assert_equal, assert_rel, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()
    oracle.build()


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_sampled(idx):
    wl = workloads.WORKLOADS[idx]
    inp = workloads.make_inputs(wl)
    x, gy, w = (to_dev(inp, n, wl.dtype) for n in ("x", "g_y", "w"))
    rng = np.random.default_rng(1000 + idx)
    n_rows = 32 if wl.Cin * wl.Cout > 20_000_000 else 96

    # ---- g_x path --------------------------------------------------------
    r = hlq.hlq_debug_gx_parts(gy, w, gran_gy=wl.gran_gy, rnd=hlq.SR,
                               seed=wl.seed)
    gx_pub = hlq.hlq_linear_backward_gx(gy, w, gran_gy=wl.gran_gy,
                                        rnd=hlq.SR, seed=wl.seed)
    assert torch.equal(gx_pub, r["g_x"])
    Wt = oracle.hq_transform(inp["w"], 1)
    qWt, s_w = oracle.hq_quantize(Wt, oracle.PER_TENSOR, oracle.SR, wl.seed,
                                  oracle.STREAM_W)
    qW = np.ascontiguousarray(qWt.T)
    assert_equal(host(r["sw"]), s_w, "s_w")
    assert_equal(host(r["qw"]), qW, "qW")
    rows = np.sort(rng.choice(wl.T, n_rows, replace=False))
    if wl.gran_gy == workloads.PER_TOKEN:
        Yr = oracle.hq_transform(inp["g_y"][rows], 0)
        qYr, s_r = oracle.hq_quantize_rows(Yr, rows, oracle.PER_TOKEN,
                                           oracle.SR, wl.seed, oracle.STREAM_GY)
        assert_equal(host(r["sgy"])[rows], s_r, "s_gy rows")
    else:
        Y = oracle.hq_transform(inp["g_y"], 0)
        qYr, s_r = oracle.hq_quantize_rows(Y[rows], rows, oracle.PER_TENSOR,
                                           oracle.SR, wl.seed, oracle.STREAM_GY,
                                           tensor_amax=oracle.amax(Y))
        assert_equal(host(r["sgy"]), s_r, "s_gy")
        del Y
    assert_equal(host(r["qgy"])[rows], qYr, "qY rows")
    acc_rows = oracle.gemm_i64(qYr, qW)
    assert_equal(host(r["acc"])[rows].astype(np.int64), acc_rows, "acc_gx rows")
    s_sel = s_r if wl.gran_gy == workloads.PER_TOKEN else s_r
    assert_rel(host(r["g_x"])[rows],
               oracle.dequant_gx(acc_rows, s_sel, wl.gran_gy, s_w[0]), 1e-5,
               "g_x rows")
    # whole GEMM against the CUDA-core reference (integer sums)
    ref_acc = hlq.hlq_debug_reference_gemm(r["qgy"], r["qw"])
    assert torch.equal(ref_acc, r["acc"])
    del r, gx_pub, ref_acc
    torch.cuda.empty_cache()

    # ---- ACBP + g_w path -------------------------------------------------
    xbar, sx = hlq.hlq_compress_activation(x, rank=wl.rank)
    qX, s_x = oracle.compress_activation(inp["x"], wl.rank)
    assert_equal(host(sx)[0], s_x, "s_x")
    assert_equal(host(xbar), qX, "xbar")
    g = hlq.hlq_debug_gw_parts(gy, xbar, sx, rank=wl.rank)
    gw_pub = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=wl.rank)
    assert torch.equal(gw_pub, g["g_w"])
    Gb = oracle.hla_transform(inp["g_y"], wl.rank)
    qG, s_g = oracle.int8_quantize(Gb)
    del Gb
    assert_equal(host(g["sg"])[0], s_g, "s_g")
    assert_equal(host(g["qg"]), qG, "qG")
    orows = np.sort(rng.choice(wl.Cout, min(n_rows, wl.Cout), replace=False))
    acc_o = oracle.gemm_i64(qG[orows], qX)
    assert_equal(host(g["acc"])[orows].astype(np.int64), acc_o, "acc_gw rows")
    assert_rel(host(g["g_w"])[orows], oracle.dequant_gw(acc_o, s_g, s_x), 1e-5,
               "g_w rows")
    ref_acc = hlq.hlq_debug_reference_gemm(g["qg"], xbar)
    assert torch.equal(ref_acc, g["acc"])
    assert hlq.hlq_read_device_status(clear=True) == 0
