"""Ablation of the activation-gradient path (hlq_ablation_gx_hla): HLA along
Cout of g_y (its rows) and of w (its first dim), per-tensor RNE int8 codes
and an exact integer GEMM over Cout*rank/16 on the bf16 tensor cores.  The
accumulator is bit-exact against the oracle (so every code matched), g_x
within 1e-5 of the oracle's fp64 dequant, for fp32 and bf16 inputs, every
rank and ragged tiles."""
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


@pytest.mark.parametrize("wl_idx,T,dtype,rank", [
    (0, 256, "f32", 8), (1, 528, "bf16", 8), (1, 272, "bf16", 1), (2, 400, "bf16", 2),
    (4, 512, "bf16", 4), (1, 256, "bf16", 16), (0, 128, "f32", 16)])
def test_gx_hla_ablation_parity(wl_idx, T, dtype, rank):
    wl = workloads.WORKLOADS[wl_idx]
    inp = workloads.make_inputs(wl, T=T)
    gy, w = to_dev(inp, "g_y", dtype), to_dev(inp, "w", dtype)
    gx, acc = hlq.hlq_ablation_gx_hla(gy, w, rank=rank, with_acc=True)
    rows = (np.random.default_rng(9).choice(T, 96, replace=False)
            if T * wl.Cin * wl.Cout > 400_000_000 else None)
    ref = oracle.gx_hla_path(inp["g_y"], inp["w"], rank, rows=rows)
    sel = ref["rows"]
    assert_equal(host(acc)[sel].astype(np.int64), ref["acc"], "acc")
    assert_rel(host(gx)[sel], ref["g_x"], 1e-5, "g_x")
    assert hlq.hlq_read_device_status(clear=True) == 0
    gx2 = hlq.hlq_ablation_gx_hla(gy, w, rank=rank)
    torch.cuda.synchronize()
    assert torch.equal(gx, gx2)


def test_gx_hla_ablation_error_grows_as_rank_drops():
    """The low-rank product loses more of g_y . w as fewer Walsh rows are
    kept (numerical-error study the ablation exists for), and rank 16 is
    close to the exact product up to the int8 rounding."""
    wl = workloads.WORKLOADS[1]
    inp = workloads.make_inputs(wl, T=512)
    gy, w = to_dev(inp, "g_y", "bf16"), to_dev(inp, "w", "bf16")
    want = inp["g_y"].astype(np.float64) @ inp["w"].astype(np.float64)
    err = {}
    for r in (1, 2, 4, 8, 16):
        g = host(hlq.hlq_ablation_gx_hla(gy, w, rank=r)).astype(np.float64)
        err[r] = np.linalg.norm(g - want) / np.linalg.norm(want)
    assert err[1] > err[2] > err[4] > err[8] > err[16]
    assert err[16] < 0.05
