"""Per-channel scales of the stored activation: one scale per input channel
of the compressed x (the per-layer granularity choice of HOT, Approach,
carried to the ACBP buffer, whose token dim is the g_w contraction dim), and
the g_w GEMM dequantizing with s_x[i] per column.  Codes and scales bit-exact
against the oracle, integer accumulators exact, g_w within 1e-5 of the
oracle's fp64 dequant; the combined, host-buffer and per-tensor special-case
entry points agree bit for bit."""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()
    oracle.build()


def _inputs(wl_idx, T, Cin, Cout):
    """Workload inputs at reduced sizes (same distributions: for the Llama
    shapes, 1 % of the channels x50)."""
    wl = dataclasses.replace(workloads.WORKLOADS[wl_idx], Cin=Cin, Cout=Cout)
    return wl, workloads.make_inputs(wl, T=T)


# Llama-like inputs (1 % of the channels x50) at small T and Cin; fp32 and
# bf16; int8 and int4 codes; several ranks and a ragged channel tail
@pytest.mark.parametrize("wl_idx,T,Cin,dtype,rank,bits", [
    (3, 256, 1040, "bf16", 8, 8), (3, 272, 528, "bf16", 4, 4), (3, 256, 272, "f32", 8, 8),
    (3, 512, 400, "bf16", 1, 8), (3, 256, 400, "bf16", 16, 4), (1, 528, 768, "bf16", 2, 8)])
def test_per_channel_acbp_parity(wl_idx, T, Cin, dtype, rank, bits):
    wl, inp = _inputs(wl_idx, T, Cin, 256)
    x, gy = to_dev(inp, "x", dtype), to_dev(inp, "g_y", dtype)
    xbar, sx = hlq.hlq_compress_activation(x, rank=rank, xbar_bits=bits,
                                           xbar_per_channel=True)
    assert tuple(sx.shape) == (Cin,)
    q_ref, s_ref = oracle.compress_activation(inp["x"], rank, bits=bits, per_channel=True)
    assert_equal(host(sx), s_ref, "s_x per channel")
    assert_equal(host(xbar), oracle.pack_int4(q_ref) if bits == 4 else q_ref, "xbar")
    r = hlq.hlq_debug_gw_parts(gy, xbar, sx, rank=rank, xbar_bits=bits,
                               xbar_per_channel=True)
    ref = oracle.gw_path(inp["g_y"], q_ref, s_ref, rank)
    assert_equal(host(r["sg"])[0], ref["s_g"], "s_g")
    assert_equal(host(r["qg"]), ref["qG"], "qG")
    assert_equal(host(r["acc"]).astype(np.int64), ref["acc"], "acc_gw")
    assert_rel(host(r["g_w"]), ref["g_w"], TOL, "g_w")
    gw = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=rank, xbar_bits=bits,
                                    xbar_per_channel=True)
    assert_equal(host(gw), host(r["g_w"]), "g_w public vs parts")


def test_per_channel_with_equal_maxima_is_per_tensor():
    """Every channel's largest coefficient the same number: per-channel
    scales, codes and g_w equal the per-tensor ones bit for bit (the
    per-column dequant multiplies in the same order as the tensor one)."""
    rng = np.random.default_rng(31)
    T, Cin, Cout = 256, 96, 128
    x = rng.standard_normal((T, Cin)).astype(np.float32)
    x[:16, :] = 40.0
    gy = rng.standard_normal((T, Cout)).astype(np.float32)
    xd, gyd = torch.from_numpy(x).cuda(), torch.from_numpy(gy).cuda()
    xc, sc = hlq.hlq_compress_activation(xd, xbar_per_channel=True)
    xt, st = hlq.hlq_compress_activation(xd)
    torch.cuda.synchronize()
    assert torch.equal(xc, xt) and bool(torch.all(sc == st))
    gc = hlq.hlq_linear_backward_gw(gyd, xc, sc, xbar_per_channel=True)
    gt = hlq.hlq_linear_backward_gw(gyd, xt, st)
    torch.cuda.synchronize()
    assert torch.equal(gc, gt)


def test_per_channel_combined_and_host_step():
    wl, inp = _inputs(3, 512, 528, 512)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x, rank=8, xbar_per_channel=True)
    gx1 = hlq.hlq_linear_backward_gx(gy, w, seed=3)
    gw1 = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=8, xbar_per_channel=True)
    gx2, gw2 = hlq.hlq_linear_backward(gy, w, xbar, sx, rank=8, seed=3,
                                       xbar_per_channel=True)
    torch.cuda.synchronize()
    assert torch.equal(gx1, gx2) and torch.equal(gw1, gw2)
    hx, hgy, hw = (t.cpu().pin_memory() for t in (x, gy, w))
    xb3 = torch.empty_like(xbar)
    sx3 = torch.empty_like(sx)
    h_gx, h_gw = hlq.hlq_layer_step_host(hx, hgy, hw, xb3, sx3, rank=8, seed=3,
                                         chunk_tokens=256, xbar_per_channel=True)
    torch.cuda.synchronize()
    assert torch.equal(xb3, xbar) and torch.equal(sx3, sx)
    assert torch.equal(h_gx, gx1.cpu()) and torch.equal(h_gw, gw1.cpu())


def test_per_channel_lowers_error_on_outlier_channels():
    """On Llama-like inputs the per-channel scales give a g_w closer to the
    unquantized fp64 product of the same low-rank operands than one tensor
    scale does (the small channels keep their resolution)."""
    wl, inp = _inputs(3, 512, 1040, 256)
    x, gy = to_dev(inp, "x", "bf16"), to_dev(inp, "g_y", "bf16")
    want = (oracle.hla_transform(inp["g_y"], 8).astype(np.float64)
            @ oracle.hla_transform(inp["x"], 8).astype(np.float64).T) / 16.0
    errs = []
    for pc in (False, True):
        xb, s = hlq.hlq_compress_activation(x, xbar_per_channel=pc)
        g = host(hlq.hlq_linear_backward_gw(gy, xb, s, xbar_per_channel=pc))
        errs.append(np.linalg.norm(g - want) / np.linalg.norm(want))
    assert errs[1] < errs[0]
