"""int4 storage of the stored activation (HLQ TL;DR: int4 activation
compression, ACBP): the compressed x as two's-complement int4
codes packed two per byte, then the g_w path reading it.  Codes (as packed
bytes), scales and integer accumulators bit-exact against the oracle, g_w
within 1e-5 of the oracle's fp64 dequant; the combined and host-buffer
entry points give the same bits as the separate calls."""
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


@pytest.mark.parametrize("wl_idx,T,dtype,rank", [(0, 256, "f32", 8), (1, 528, "bf16", 8),
                                                 (1, 528, "bf16", 2), (2, 256, "bf16", 16),
                                                 (3, 272, "bf16", 4)])
def test_int4_acbp_parity(wl_idx, T, dtype, rank):
    wl = workloads.WORKLOADS[wl_idx]
    inp = workloads.make_inputs(wl, T=T)
    x, gy = to_dev(inp, "x", dtype), to_dev(inp, "g_y", dtype)
    xbar, sx = hlq.hlq_compress_activation(x, rank=rank, xbar_bits=4)
    assert tuple(xbar.shape) == (wl.Cin, T // 16 * rank // 2)
    q_ref, s_ref = oracle.compress_activation(inp["x"], rank, bits=4)
    assert np.all(np.abs(q_ref) <= 7)
    assert_equal(host(sx)[0], s_ref, "s_x")
    assert_equal(host(xbar), oracle.pack_int4(q_ref), "packed xbar")
    r = hlq.hlq_debug_gw_parts(gy, xbar, sx, rank=rank, xbar_bits=4)
    # the oracle's GEMM on sampled output channels for the large shape
    rows = (np.random.default_rng(5).choice(wl.Cout, 64, replace=False)
            if wl.Cout * wl.Cin > 4_000_000 else None)
    ref = oracle.gw_path(inp["g_y"], q_ref, s_ref, rank, rows=rows)
    sel = ref["rows"]
    assert_equal(host(r["sg"])[0], ref["s_g"], "s_g")
    assert_equal(host(r["qg"]), ref["qG"], "qG")
    assert_equal(host(r["acc"])[sel].astype(np.int64), ref["acc"], "acc_gw")
    assert_rel(host(r["g_w"])[sel], ref["g_w"], TOL, "g_w")
    gw = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=rank, xbar_bits=4)
    assert_equal(host(gw), host(r["g_w"]), "g_w public vs parts")


def test_int4_acbp_combined_and_host_step():
    wl = workloads.WORKLOADS[1]
    inp = workloads.make_inputs(wl, T=1024)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x, rank=8, xbar_bits=4)
    gx1 = hlq.hlq_linear_backward_gx(gy, w, seed=3)
    gw1 = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=8, xbar_bits=4)
    gx2, gw2 = hlq.hlq_linear_backward(gy, w, xbar, sx, rank=8, seed=3, xbar_bits=4)
    torch.cuda.synchronize()
    assert torch.equal(gx1, gx2) and torch.equal(gw1, gw2)
    hx, hgy, hw = (t.cpu().pin_memory() for t in (x, gy, w))
    xb3 = torch.empty_like(xbar)
    sx3 = torch.empty_like(sx)
    h_gx, h_gw = hlq.hlq_layer_step_host(hx, hgy, hw, xb3, sx3, rank=8, seed=3,
                                         chunk_tokens=256, xbar_bits=4)
    torch.cuda.synchronize()
    assert torch.equal(xb3, xbar) and torch.equal(sx3, sx)
    assert torch.equal(h_gx, gx1.cpu()) and torch.equal(h_gw, gw1.cpu())


def test_int4_acbp_saves_memory():
    """Stored bytes per token and channel: bf16 x 2, int8 codes 0.5 (rank 8,
    T' = T/2), int4 codes 0.25, i.e. 75 % and 87.5 % saved."""
    T, Cin = 12608, 768
    b16 = T * Cin * 2
    b8 = int(np.prod(hlq.xbar_shape(T, Cin, 8, 8)))
    b4 = int(np.prod(hlq.xbar_shape(T, Cin, 8, 4)))
    assert 1 - b8 / b16 == 0.75 and 1 - b4 / b16 == 0.875
    x = torch.randn(T, Cin, device="cuda").to(torch.bfloat16)
    xb8, _ = hlq.hlq_compress_activation(x, xbar_bits=8)
    xb4, _ = hlq.hlq_compress_activation(x, xbar_bits=4)
    assert xb8.numel() * xb8.element_size() == b8
    assert xb4.numel() * xb4.element_size() == b4
