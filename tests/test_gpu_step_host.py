"""The host-buffer layer step (hlq_layer_step_host): copies pipelined with
the computation in chunks of tokens, results bit-identical to the device
entry points on the same inputs, for one and several chunks, a ragged last
chunk, per-token and per-tensor g_y scales, bf16 and fp32."""
import numpy as np
import pytest
import torch

import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()


def _host(inp, name, dtype):
    if dtype == "bf16":
        bits = np.ascontiguousarray(inp[name + "_bits"])
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(np.ascontiguousarray(inp[name], np.float32)).pin_memory()


# (0, 5120, 128): 40 chunks, more than the event set of the first version
# held; (0, 8960, 128): 70 requested, widened to 35 chunks of 256 tokens
@pytest.mark.parametrize("wl_idx,T,chunk", [(1, 1024, 256), (1, 1024, 0), (2, 528, 128),
                                            (0, 256, 128), (0, 5120, 128), (0, 8960, 128)])
def test_step_host_matches_device_path(wl_idx, T, chunk):
    wl = workloads.WORKLOADS[wl_idx]
    inp = workloads.make_inputs(wl, T=T)
    x, gy, w = (_host(inp, n, wl.dtype) for n in ("x", "g_y", "w"))
    Tp = T // 16 * wl.rank
    xbar = torch.empty((wl.Cin, Tp), dtype=torch.int8, device="cuda")
    sx = torch.empty(1, dtype=torch.float32, device="cuda")
    hlq.hlq_read_device_status(clear=True)
    h_gx, h_gw = hlq.hlq_layer_step_host(x, gy, w, xbar, sx, rank=wl.rank, gran_gy=wl.gran_gy,
                                         gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed,
                                         chunk_tokens=chunk)
    torch.cuda.synchronize()
    # the device path on the same inputs
    dx, dgy, dw = x.cuda(), gy.cuda(), w.cuda()
    xbar_ref, sx_ref = hlq.hlq_compress_activation(dx, rank=wl.rank)
    gx_ref = hlq.hlq_linear_backward_gx(dgy, dw, gran_gy=wl.gran_gy, gran_w=wl.gran_w,
                                        rnd=hlq.SR, seed=wl.seed)
    gw_ref = hlq.hlq_linear_backward_gw(dgy, xbar_ref, sx_ref, rank=wl.rank)
    torch.cuda.synchronize()
    assert hlq.hlq_read_device_status() == 0
    assert torch.equal(xbar.cpu(), xbar_ref.cpu())
    assert torch.equal(sx.cpu(), sx_ref.cpu())
    assert torch.equal(h_gx, gx_ref.cpu())
    assert torch.equal(h_gw, gw_ref.cpu())


def test_step_host_empty_tokens():
    wl = workloads.WORKLOADS[1]
    x = torch.empty((0, wl.Cin), dtype=torch.bfloat16).pin_memory()
    gy = torch.empty((0, wl.Cout), dtype=torch.bfloat16).pin_memory()
    w = torch.randn(wl.Cout, wl.Cin).to(torch.bfloat16).pin_memory()
    xbar = torch.empty((wl.Cin, 0), dtype=torch.int8, device="cuda")
    sx = torch.full((1,), 7.0, device="cuda")
    h_gx, h_gw = hlq.hlq_layer_step_host(x, gy, w, xbar, sx, rank=wl.rank)
    torch.cuda.synchronize()
    assert h_gx.shape == (0, wl.Cin)
    assert torch.count_nonzero(h_gw) == 0 and float(sx.cpu()) == 0.0
