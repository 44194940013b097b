"""One layer step from device buffers (hlq_layer_step): the ACBP compression
of x on the g_w branch, beside the g_x branch, and both gradients.  Every
output bit (g_x, g_w, the stored codes and scales) equals
hlq_compress_activation followed by hlq_linear_backward, which the other
parity tests pin to the oracle; also inside a captured CUDA graph."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()


def _inputs(wl_idx, T, Cin=None, Cout=None):
    wl = workloads.WORKLOADS[wl_idx]
    if Cin or Cout:
        wl = dataclasses.replace(wl, Cin=Cin or wl.Cin, Cout=Cout or wl.Cout)
    inp = workloads.make_inputs(wl, T=T)
    return wl, inp


def _separate(x, gy, w, **kw):
    bits = kw.get("xbar_bits", 8)
    pc = kw.get("xbar_per_channel", False)
    rank = kw.get("rank", 8)
    xbar, sx = hlq.hlq_compress_activation(x, rank=rank, xbar_bits=bits, xbar_per_channel=pc)
    gx, gw = hlq.hlq_linear_backward(gy, w, xbar, sx, **kw)
    return gx, gw, xbar, sx


@pytest.mark.parametrize("wl_idx,T,Cin,Cout,dtype,kw", [
    (1, 512, None, None, "bf16", dict(seed=3)),
    (0, 256, None, None, "f32", dict(rank=4, gran_gy=hlq.PER_TENSOR)),
    (3, 256, 528, 400, "bf16", dict(xbar_per_channel=True, rank=2)),
    (2, 272, None, None, "bf16", dict(xbar_bits=4, rnd=hlq.RNE)),
    (1, 256, 64, 400, "bf16", dict(rank=1)),
    (1, None, None, None, "bf16", dict(seed=9))])
def test_layer_step_equals_separate_calls(wl_idx, T, Cin, Cout, dtype, kw):
    wl, inp = _inputs(wl_idx, T, Cin, Cout)
    x, gy, w = (to_dev(inp, n, dtype) for n in ("x", "g_y", "w"))
    ref = _separate(x, gy, w, **kw)
    got = hlq.hlq_layer_step(x, gy, w, **kw)
    torch.cuda.synchronize()
    assert hlq.hlq_read_device_status(clear=True) == 0
    for name, a, b in zip(("g_x", "g_w", "xbar", "xbar_scale"), ref, got):
        assert torch.equal(a, b), name


def test_layer_step_in_a_graph():
    wl, inp = _inputs(1, 1024)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    ref = _separate(x, gy, w, seed=4)
    T, Cin, Cout = 1024, wl.Cin, wl.Cout
    outs = (torch.empty((T, Cin), dtype=torch.float32, device="cuda"),
            torch.empty((Cout, Cin), dtype=torch.float32, device="cuda"),
            torch.empty(hlq.xbar_shape(T, Cin), dtype=torch.int8, device="cuda"),
            torch.empty(1, dtype=torch.float32, device="cuda"))
    ws = hlq.workspace(hlq.OP_LAYER_STEP, T, Cin, Cout, 16, 8, x.device)

    def step():
        hlq.hlq_layer_step(x, gy, w, seed=4, out_gx=outs[0], out_gw=outs[1], xbar=outs[2],
                           xbar_scale=outs[3], ws=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("fused_gy", [False, True])
def test_serialized_branches_give_the_same_bits(fused_gy):
    """hlq_debug_serialize_branches runs the same kernels on one stream (the
    bench's per-kernel trace): every output equals the forked run's."""
    wl, inp = _inputs(3, 512, 528, 400)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    ref_step = hlq.hlq_layer_step(x, gy, w, seed=5)
    ref_bwd = hlq.hlq_linear_backward(gy, w, ref_step[2], ref_step[3], seed=5,
                                      fused_gy=fused_gy)
    hlq.hlq_debug_serialize_branches(True)
    try:
        got_step = hlq.hlq_layer_step(x, gy, w, seed=5)
        got_bwd = hlq.hlq_linear_backward(gy, w, ref_step[2], ref_step[3], seed=5,
                                          fused_gy=fused_gy)
    finally:
        hlq.hlq_debug_serialize_branches(False)
    torch.cuda.synchronize()
    for a, b in zip(ref_step + ref_bwd, got_step + got_bwd):
        assert torch.equal(a, b)
    assert hlq.hlq_read_device_status(clear=True) == 0
