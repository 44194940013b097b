"""Launch tracing (hlq_trace_*): per-kernel device times of the library's
launches, recorded from eager calls and from replays of a captured graph,
without disturbing the launches themselves (outputs equal untraced ones)."""
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


def _inputs():
    wl = workloads.WORKLOADS[1]          # ViT-B qkv shapes, 512 tokens
    inp = workloads.make_inputs(wl, T=512)
    return wl, to_dev(inp, "g_y", "bf16"), to_dev(inp, "w", "bf16")


def test_trace_eager_calls():
    wl, gy, w = _inputs()
    ref = hlq.hlq_linear_backward_gx(gy, w, seed=3)
    hlq.hlq_trace_begin(64)
    got = hlq.hlq_linear_backward_gx(gy, w, seed=3)
    torch.cuda.synchronize()
    rec = hlq.hlq_trace_end()
    names = [n for n, _ in rec]
    assert "hq_rows_quant" in names and "gemm_gx_tc" in names
    assert all(ms > 0 for _, ms in rec)
    assert torch.equal(ref, got)


def test_trace_graph_replays():
    wl, gy, w = _inputs()
    out = torch.empty((gy.shape[0], w.shape[1]), dtype=torch.float32, device="cuda")
    ws = hlq.workspace(hlq.OP_BACKWARD_GX, gy.shape[0], w.shape[1], w.shape[0], 16, 8,
                       gy.device)
    ref = hlq.hlq_linear_backward_gx(gy, w, seed=5)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        hlq.hlq_linear_backward_gx(gy, w, seed=5, out=out, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    hlq.hlq_trace_begin(64)
    with torch.cuda.graph(g):
        hlq.hlq_linear_backward_gx(gy, w, seed=5, out=out, ws=ws)
    n = hlq.hlq_trace_end(keep=True)
    assert n >= 3
    try:
        for _ in range(2):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            rec = hlq.hlq_trace_read()
            assert len(rec) == n and all(ms > 0 for _, ms in rec)
            assert torch.equal(ref, out)
    finally:
        hlq.hlq_trace_free()
