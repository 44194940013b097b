"""Parity at the full workload sizes, through the same entry points and
launch configuration the benchmark times.

The oracle recomputes every code and scale (bit-exact): whole tensors where
per-tensor scales need them, every row of the per-token HQ of g_y; and the
integer GEMM rows of at least 1024 tokens / output channels (or all of
them), chosen across every 128-row tile edge, the ragged tail and at
random; the tensor-core GEMMs are also compared in full with the CUDA-core
reference GEMM (integer sums, bit-exact).
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


def _row_blocks(n, parts=16):
    step = -(-n // parts)
    return [np.arange(a, min(n, a + step)) for a in range(0, n, step)]


def _pmap(fn, items):
    """The oracle's own routines on disjoint row blocks in parallel threads
    (ctypes releases the interpreter lock); the result is the same as one
    call over all rows."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=16) as ex:
        return list(ex.map(fn, items))


def _gemm_rows(A_rows, B):
    parts = _pmap(lambda ix: oracle.gemm_i64(A_rows[ix], B), _row_blocks(len(A_rows)))
    return np.concatenate(parts, axis=0)


def _sample_rows(n, k, rng, tile=128):
    """Rows across the GEMM's row tiles: the first and last row of every
    128-row tile (and of the 256-row tiles of CTA pairs), the ragged tail,
    and random rows, at least min(k, n) of them."""
    edges = {0, n - 1, max(0, n - 2)}
    for t in range(0, n, tile):
        edges.update((t, min(n - 1, t + tile - 1)))
    rows = np.array(sorted(edges), dtype=np.int64)
    if len(rows) < min(k, n):
        rest = np.setdiff1d(np.arange(n), rows)
        extra = rng.choice(rest, min(k, n) - len(rows), replace=False)
        rows = np.sort(np.r_[rows, extra])
    return rows


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_sampled(idx):
    wl = workloads.WORKLOADS[idx]
    inp = workloads.make_inputs(wl)
    x, gy, w = (to_dev(inp, n, wl.dtype) for n in ("x", "g_y", "w"))
    rng = np.random.default_rng(1000 + idx)

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
    assert_equal(host(r["qw_packed"]), oracle.pack_int4(qW), "qW packed int4")
    rows = _sample_rows(wl.T, 1024, rng)
    if wl.gran_gy == workloads.PER_TOKEN:
        # every row's codes and scale (rows are independent under per-token
        # scales: each block of rows quantized alone keeps its Philox words)
        def quant_block(ix):
            Yb = oracle.hq_transform(inp["g_y"][ix], 0)
            return oracle.hq_quantize_rows(Yb, ix, oracle.PER_TOKEN, oracle.SR, wl.seed,
                                           oracle.STREAM_GY)
        parts = _pmap(quant_block, _row_blocks(wl.T, 64))
        qY_all = np.concatenate([p[0] for p in parts], axis=0)
        s_all = np.concatenate([p[1] for p in parts])
        assert_equal(host(r["sgy"]), s_all, "s_gy (every row)")
        assert_equal(host(r["qgy"]), qY_all, "qY (every row)")
        assert_equal(host(r["qgy_packed"]), oracle.pack_int4(qY_all),
                     "qY packed int4 (every row)")
        qYr, s_r = qY_all[rows], s_all[rows]
        del qY_all, parts
    else:
        Y = oracle.hq_transform(inp["g_y"], 0)
        qYr, s_r = oracle.hq_quantize_rows(Y[rows], rows, oracle.PER_TENSOR,
                                           oracle.SR, wl.seed, oracle.STREAM_GY,
                                           tensor_amax=oracle.amax(Y))
        assert_equal(host(r["sgy"]), s_r, "s_gy")
        del Y
    assert_equal(host(r["qgy"])[rows], qYr, "qY rows")
    acc_rows = _gemm_rows(qYr, qW)
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
    orows = _sample_rows(wl.Cout, 1024, rng)
    acc_o = _gemm_rows(qG[orows], qX)
    assert_equal(host(g["acc"])[orows].astype(np.int64), acc_o, "acc_gw rows")
    assert_rel(host(g["g_w"])[orows], oracle.dequant_gw(acc_o, s_g, s_x), 1e-5,
               "g_w rows")
    ref_acc = hlq.hlq_debug_reference_gemm(g["qg"], xbar)
    assert torch.equal(ref_acc, g["acc"])
    assert hlq.hlq_read_device_status(clear=True) == 0
