"""Fused reader of g_y (hlq_linear_backward_fused): the HQ of g_y and the HLA
of g_y taken from the same TMA-staged 16-token x 256-column tiles, in two
passes (maxima, then codes) instead of three reads.  Every output bit equals
the separate path's (hlq_linear_backward), which the other parity tests pin
to the oracle; one case is also compared with the oracle directly.  Shapes
cover ragged column tiles (Cout not a multiple of 256 or of 32), both g_y
granularities, fp32 and bf16, every rank, int4 and per-channel stored
activations, RNE and SR."""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()
    oracle.build()


def _inputs(wl_idx, T, Cin=None, Cout=None):
    wl = workloads.WORKLOADS[wl_idx]
    if Cin or Cout:
        wl = dataclasses.replace(wl, Cin=Cin or wl.Cin, Cout=Cout or wl.Cout)
    return wl, workloads.make_inputs(wl, T=T)


def _both(gy, w, xbar, sx, **kw):
    a = hlq.hlq_linear_backward(gy, w, xbar, sx, **kw)
    b = hlq.hlq_linear_backward(gy, w, xbar, sx, fused_gy=True, **kw)
    torch.cuda.synchronize()
    assert hlq.hlq_read_device_status(clear=True) == 0
    return a, b


@pytest.mark.parametrize("wl_idx,T,Cin,Cout,dtype,rank,gran", [
    (1, 512, None, None, "bf16", 8, 1), (1, 528, None, None, "bf16", 8, 0),
    (0, 256, None, None, "f32", 8, 1), (0, 256, None, None, "f32", 4, 0),
    (2, 272, None, None, "bf16", 16, 1), (4, 400, None, None, "bf16", 2, 0),
    (1, 256, 64, 400, "bf16", 1, 1), (1, 256, 96, 272, "bf16", 8, 1),
    (3, 256, 528, 208, "bf16", 4, 1), (1, 2048, None, None, "bf16", 8, 1)])
@pytest.mark.parametrize("rnd", [hlq.SR, hlq.RNE])
def test_fused_gy_equals_separate(wl_idx, T, Cin, Cout, dtype, rank, gran, rnd):
    wl, inp = _inputs(wl_idx, T, Cin, Cout)
    x, gy, w = (to_dev(inp, n, dtype) for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x, rank=rank)
    (gx1, gw1), (gx2, gw2) = _both(gy, w, xbar, sx, rank=rank, gran_gy=gran, rnd=rnd, seed=11)
    assert torch.equal(gx1, gx2), "g_x"
    assert torch.equal(gw1, gw2), "g_w"


@pytest.mark.parametrize("bits,per_channel", [(4, False), (8, True), (4, True)])
def test_fused_gy_with_stored_activation_formats(bits, per_channel):
    wl, inp = _inputs(3, 256, 528, 400)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x, xbar_bits=bits, xbar_per_channel=per_channel)
    kw = dict(xbar_bits=bits, xbar_per_channel=per_channel, seed=5)
    (gx1, gw1), (gx2, gw2) = _both(gy, w, xbar, sx, **kw)
    assert torch.equal(gx1, gx2) and torch.equal(gw1, gw2)


def test_fused_gy_against_oracle():
    wl, inp = _inputs(1, 528)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x)
    gx, gw = hlq.hlq_linear_backward(gy, w, xbar, sx, seed=3, fused_gy=True)
    rows = np.random.default_rng(4).choice(528, 64, replace=False)
    ref_x = oracle.gx_path(inp["g_y"], inp["w"], seed=3, rows=rows)
    assert_rel(host(gx)[ref_x["rows"]], ref_x["g_x"], 1e-5, "g_x")
    q_ref, s_ref = oracle.compress_activation(inp["x"], 8)
    ocs = np.random.default_rng(5).choice(wl.Cout, 64, replace=False)
    ref_w = oracle.gw_path(inp["g_y"], q_ref, s_ref, 8, rows=ocs)
    assert_rel(host(gw)[ref_w["rows"]], ref_w["g_w"], 1e-5, "g_w")


def test_fused_gy_full_size_equals_separate():
    """ViT-B qkv at full size (T = 12608), the bench's workload."""
    wl, inp = _inputs(1, None)
    x, gy, w = (to_dev(inp, n, "bf16") for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x)
    (gx1, gw1), (gx2, gw2) = _both(gy, w, xbar, sx, seed=wl.seed)
    assert torch.equal(gx1, gx2) and torch.equal(gw1, gw2)
