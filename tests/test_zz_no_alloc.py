"""hlq_linear_backward_gx_noalloc, the g_x entry point for callers that
cannot allocate device memory (plugins of a runtime that owns all device
memory, loops that forbid cudaMalloc once running): called through the C ABI
twice in a row, it must give bit for bit what the workspace entry point
gives (both run the same kernels), and match the oracle: integer codes
dequantized within 1e-5 relative of the oracle's fp64 g_x.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process (the
first call on the device does the one-time set-up of the scratch array)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import assert_rel, host, to_dev

pytestmark = pytest.mark.gpu


def call_noalloc(L, gy, w, dt, gran, seed, out):
    T, Cout = gy.shape
    Cin = w.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.hlq_linear_backward_gx_noalloc(
        ctypes.c_void_p(gy.data_ptr()), ctypes.c_void_p(w.data_ptr()), dt, T, Cin,
        Cout, 16, gran, hlq.PER_TENSOR, hlq.SR, seed,
        ctypes.c_void_p(out.data_ptr()), stream)


def test_noalloc_gx_matches_workspace_entry_point_on_two_calls():
    hbuild.build()
    L = hlq.lib()
    assert L.hlq_noalloc_scratch_bytes() == 40 << 20
    cases = []
    # call 1: ViT-B qkv shapes (T shortened), bf16, per-tensor g_y scale;
    # oracle rows across GEMM tiles and the last ones
    wl = workloads.WORKLOADS[1]
    inp = workloads.make_inputs(wl, T=4096)
    rows = np.unique(np.r_[np.arange(0, 4096, 37), 127, 128, 255, 256, 4094, 4095])
    cases.append((inp, to_dev(inp, "g_y", "bf16"), to_dev(inp, "w", "bf16"), hlq.BF16,
                  hlq.PER_TENSOR, 7, rows))
    # call 2: the fp32 single-linear workload, per-token g_y scales, every row
    wl0 = workloads.WORKLOADS[0]
    inp0 = workloads.make_inputs(wl0)
    cases.append((inp0, to_dev(inp0, "g_y", "f32"), to_dev(inp0, "w", "f32"), hlq.F32,
                  hlq.PER_TOKEN, 0, None))
    for inp_c, gy, w, dt, gran, seed, sel in cases:
        out = torch.full((gy.shape[0], w.shape[1]), float("nan"), device="cuda")
        rc = call_noalloc(L, gy, w, dt, gran, seed, out)
        assert rc == 0, hlq.status_string(rc)
        want = hlq.hlq_linear_backward_gx(gy, w, gran_gy=gran, rnd=hlq.SR, seed=seed)
        torch.cuda.synchronize()
        assert torch.equal(out, want), "noalloc g_x differs from the workspace entry"
        ref = oracle.gx_path(inp_c["g_y"], inp_c["w"], gran_gy=gran, rnd=oracle.SR,
                             seed=seed, rows=sel)
        got = host(out) if sel is None else host(out)[sel]
        assert_rel(got, ref["g_x"], 1e-5, "noalloc g_x vs oracle")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    hbuild.build()
    L = hlq.lib()
    gy = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((16, 16), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # claims T = 16384, Cout = 4096 (64 MiB of codes): refused before any launch
    rc = L.hlq_linear_backward_gx_noalloc(
        ctypes.c_void_p(gy.data_ptr()), ctypes.c_void_p(w.data_ptr()), hlq.BF16,
        16384, 16, 4096, 16, hlq.PER_TOKEN, hlq.PER_TENSOR, hlq.SR, 0,
        ctypes.c_void_p(out.data_ptr()), stream)
    assert rc == 5 and hlq.status_string(rc) == "HLQ_ERR_WORKSPACE"
