"""Ablation of the weight-gradient path (hlq_ablation_gw_hq): HQ of g_y and
x along tokens with int4 codes and an exact integer GEMM over T.  The
accumulator is bit-exact against the oracle (so every code matched), g_w
within 1e-5 of the oracle's fp64 dequant, for fp32 and bf16 inputs, ragged
tiles, RNE and SR."""
import numpy as np
import pytest

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


@pytest.mark.parametrize("wl_idx,T,dtype", [(0, 256, "f32"), (1, 528, "bf16"),
                                            (2, 272, "bf16"), (4, 512, "bf16")])
@pytest.mark.parametrize("rnd", [0, 1])
def test_gw_hq_ablation_parity(wl_idx, T, dtype, rnd):
    wl = workloads.WORKLOADS[wl_idx]
    inp = workloads.make_inputs(wl, T=T)
    gy, x = to_dev(inp, "g_y", dtype), to_dev(inp, "x", dtype)
    gw, acc = hlq.hlq_ablation_gw_hq(gy, x, rnd=rnd, seed=7, with_acc=True)
    ref = oracle.gw_hq_path(inp["g_y"], inp["x"], rnd=rnd, seed=7)
    assert_equal(host(acc).astype(np.int64), ref["acc"], "acc")
    assert_rel(host(gw), ref["g_w"], 1e-5, "g_w")
    assert hlq.hlq_read_device_status(clear=True) == 0
