"""The per-tensor amax passes of the HLA must see the exactly rounded
coefficients.  Here the column holding the true maximum coefficient has a
plain fp32 butterfly value below another column's exact value (2^24 plus
ones rounds away in fp32), so an amax taken from inexact sums would pick the
wrong maximum: scales and codes must match the oracle bit for bit, for every
rank and both input types."""
import numpy as np
import pytest
import torch

import oracle
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import assert_equal, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()
    oracle.build()


def _tricky(T=64, C=96, seed=0):
    rng = np.random.default_rng(seed)
    x = np.round(rng.standard_normal((T, C)) * 64.0).astype(np.float32)  # bf16-exact
    x[16:32, 5] = 1.0
    x[16, 5] = 2.0 ** 24                      # exact sum 2^24 + 15 -> RN 2^24 + 16
    x[16:32, 40] = 0.0
    x[16, 40] = 2.0 ** 24
    x[17, 40], x[18, 40], x[19, 40] = 8.0, 4.0, 2.0   # exact 2^24 + 14
    return x


@pytest.mark.parametrize("rank", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_amax_sees_the_exact_maximum(rank, dtype):
    x = _tricky(seed=rank)
    xd = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xd = xd.to(torch.bfloat16)
        assert torch.equal(xd.float().cpu(), torch.from_numpy(x))   # inputs exact
    xbar, s = hlq.hlq_compress_activation(xd, rank=rank)
    q_ref, s_ref = oracle.compress_activation(x, rank)
    assert_equal(host(s)[0], s_ref, "scale")
    assert_equal(host(xbar), q_ref, "codes")
    # the g_y side of the g_w path uses the same amax pass
    gy = xd
    r = hlq.hlq_debug_gw_parts(gy, xbar, s, rank=rank)
    ref = oracle.gw_path(x, q_ref, s_ref, rank)
    assert_equal(host(r["sg"])[0], ref["s_g"], "s_g")
    assert_equal(host(r["qg"]), ref["qG"], "qG")
