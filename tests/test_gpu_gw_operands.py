"""The g_w GEMM's operand layouts (hlq_set_gw_operands): x-bar widened to
fp16 by its own kernel, x-bar read as int8 by the GEMM and widened in shared
memory, and both operands (the HLA codes of g_y too) kept int8 in HBM.  Each
mode is compared with the oracle (codes, scales and integer accumulators
bit-exact, g_w within 1e-5 of its fp64 dequantization), and the modes with
each other bit for bit, through every entry point that runs a g_w GEMM.  The
HLQ page's TL;DR fixes int8 on the g_w path; the layouts only move where the
codes are widened for the fp16 tensor cores."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import assert_equal, assert_rel, host, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-5
MODES = (hlq.GW_WIDEN, hlq.GW_INT8_X, hlq.GW_INT8_BOTH)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()
    oracle.build()


@pytest.fixture(autouse=True)
def _restore_mode():
    yield
    hlq.hlq_set_gw_operands(hlq.GW_AUTO)


def _inputs(wl_idx, T, Cin, Cout):
    wl = dataclasses.replace(workloads.WORKLOADS[wl_idx], Cin=Cin, Cout=Cout)
    return wl, workloads.make_inputs(wl, T=T)


def _gw_parts(mode, gy, xbar, sx, **kw):
    hlq.hlq_set_gw_operands(mode)
    assert hlq.hlq_get_gw_operands() == mode
    return hlq.hlq_debug_gw_parts(gy, xbar, sx, **kw)


# T' = T / 16 * rank: multiples of 16 (the in-GEMM widening) and ragged ones
# (T' = 264, 132: those calls widen x-bar with the kernel in every mode);
# several ranks, fp32 and bf16, a ragged channel tail, per-channel x-bar
# scales, and int4 x-bar (widened by the kernel in every mode)
@pytest.mark.parametrize("wl_idx,T,Cin,Cout,dtype,rank,bits,per_ch", [
    (1, 512, 768, 256, "bf16", 8, 8, False),
    (1, 528, 768, 256, "bf16", 8, 8, False),
    (3, 1024, 400, 272, "bf16", 4, 8, False),
    (3, 528, 272, 400, "f32", 4, 8, False),
    (3, 2048, 1040, 512, "bf16", 16, 8, True),
    (2, 768, 528, 768, "bf16", 8, 8, False),
    (1, 512, 256, 256, "bf16", 8, 4, False),
    (0, 256, 64, 128, "f32", 8, 8, False),
])
def test_gw_operand_modes_match_oracle(wl_idx, T, Cin, Cout, dtype, rank, bits, per_ch):
    wl, inp = _inputs(wl_idx, T, Cin, Cout)
    x, gy = to_dev(inp, "x", dtype), to_dev(inp, "g_y", dtype)
    xbar, sx = hlq.hlq_compress_activation(x, rank=rank, xbar_bits=bits,
                                           xbar_per_channel=per_ch)
    q_ref, s_ref = oracle.compress_activation(inp["x"], rank, bits=bits, per_channel=per_ch)
    ref = oracle.gw_path(inp["g_y"], q_ref, s_ref, rank)
    first = None
    for mode in MODES:
        r = _gw_parts(mode, gy, xbar, sx, rank=rank, xbar_bits=bits, xbar_per_channel=per_ch)
        what = f"mode {mode}"
        assert_equal(host(r["sg"])[0], ref["s_g"], f"s_g, {what}")
        assert_equal(host(r["qg"]), ref["qG"], f"qG, {what}")
        assert_equal(host(r["acc"]).astype(np.int64), ref["acc"], f"acc_gw, {what}")
        assert_rel(host(r["g_w"]), ref["g_w"], TOL, f"g_w, {what}")
        gw = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=rank, xbar_bits=bits,
                                        xbar_per_channel=per_ch)
        assert torch.equal(gw, r["g_w"]), what
        if first is None:
            first = r
        else:
            assert torch.equal(r["g_w"], first["g_w"]), what
            assert torch.equal(r["acc"], first["acc"]), what
    assert hlq.hlq_read_device_status(clear=True) == 0


@pytest.mark.parametrize("idx", [1, 3])
def test_gw_operand_modes_agree_at_full_size(idx):
    """The workload shapes in full (ViT-B qkv: one wave of 128-wide tiles;
    Llama down_proj: CTA pairs of 256-wide tiles over 128 k-blocks): the
    three layouts give the same integer accumulators and g_w, bit for bit;
    the accumulator rows are also checked against the oracle's int64 GEMM."""
    wl = workloads.WORKLOADS[idx]
    inp = workloads.make_inputs(wl)
    x, gy = to_dev(inp, "x", wl.dtype), to_dev(inp, "g_y", wl.dtype)
    xbar, sx = hlq.hlq_compress_activation(x, rank=wl.rank)
    del x
    outs = []
    for mode in MODES:
        r = _gw_parts(mode, gy, xbar, sx, rank=wl.rank)
        outs.append((r["g_w"].clone(), r["acc"].clone(), r["qg"].clone()))
        del r
    for g, a, q in outs[1:]:
        assert torch.equal(g, outs[0][0]) and torch.equal(a, outs[0][1])
        assert torch.equal(q, outs[0][2])
    rng = np.random.default_rng(77 + idx)
    rows = np.sort(rng.choice(wl.Cout, 24, replace=False))
    rows = np.unique(np.r_[rows, 0, 127, 128, 255, 256, wl.Cout - 1])
    want = oracle.gemm_i64(host(outs[0][2])[rows], host(xbar))
    assert_equal(host(outs[0][1])[rows].astype(np.int64), want, "acc rows")
    assert hlq.hlq_read_device_status(clear=True) == 0


@pytest.mark.parametrize("idx,T,Cin,Cout", [(1, 1024, 768, 768), (3, 2048, 1024, 512),
                                            (2, 528, 768, 256)])
def test_gw_operand_modes_every_entry_point(idx, T, Cin, Cout):
    """hlq_linear_backward (separate and fused g_y reader), hlq_layer_step
    and hlq_layer_step_host give the same g_x and g_w in every mode."""
    wl, inp = _inputs(idx, T, Cin, Cout)
    dt = wl.dtype
    x, gy, w = (to_dev(inp, n, dt) for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x, rank=wl.rank)
    gran = wl.gran_gy
    results = {}
    for mode in MODES:
        hlq.hlq_set_gw_operands(mode)
        res = []
        res += hlq.hlq_linear_backward(gy, w, xbar, sx, rank=wl.rank, gran_gy=gran,
                                       seed=wl.seed)
        res += hlq.hlq_linear_backward(gy, w, xbar, sx, rank=wl.rank, gran_gy=gran,
                                       seed=wl.seed, fused_gy=True)
        st = hlq.hlq_layer_step(x, gy, w, rank=wl.rank, gran_gy=gran, seed=wl.seed)
        res += st[:2]
        xh, gyh, wh = (t.cpu().pin_memory() for t in (x, gy, w))
        xb2 = torch.empty_like(xbar)
        sx2 = torch.empty_like(sx)
        gx_h, gw_h = hlq.hlq_layer_step_host(xh, gyh, wh, xb2, sx2, rank=wl.rank,
                                             gran_gy=gran, seed=wl.seed, chunk_tokens=256)
        torch.cuda.synchronize()
        res += [gx_h.cuda(), gw_h.cuda()]
        results[mode] = res
    base = results[hlq.GW_WIDEN]
    for mode in MODES[1:]:
        for i, (a, b) in enumerate(zip(base, results[mode])):
            assert torch.equal(a, b), (mode, i)
    # the g_w of every entry point equals the separate call's
    for i in (3, 5, 7):
        assert torch.equal(base[i], base[1]), i
    assert hlq.hlq_read_device_status(clear=True) == 0
