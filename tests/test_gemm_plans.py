"""The GEMM plans the layer entries choose (host logic, no GPU): tile widths
and K splits of the two GEMMs on a 152-SM GB300, and when the g_w GEMM is
ordered after the g_x GEMM.  The expected plans are the ones measured
fastest on GB300 for these shapes (tile-plan sweep: g_x 256-wide 26.6 us vs
128-wide 32.3; g_w unsplit 128-wide 38.9 us vs 256-wide x 2 splits 48.3;
Llama down_proj 2219 us per step with the GEMMs in sequence vs 2497 side by
side)."""
import pytest

import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()


# CTA pairs only where they were measured faster: long contractions over
# several waves of tiles (Llama down_proj); not for the short-K g_x GEMMs of
# fc2 and ResNet-50, nor for the single-wave g_w GEMMs of ViT-B.
@pytest.mark.parametrize("T,Cin,Cout,gx,gw,seq,gx_pair,gw_pair", [
    (12608, 768, 2304, (256, 1), (128, 1), False, False, False),   # ViT-B qkv
    (12608, 3072, 768, (256, 1), (128, 1), False, False, False),   # ViT-B fc2
    (16384, 14336, 4096, (256, 1), (256, 1), True, True, True),    # Llama down_proj
    (50176, 2304, 256, (256, 1), (128, 4), False, False, False),   # ResNet-50 im2col
])
def test_layer_plans_on_gb300(T, Cin, Cout, gx, gw, seq, gx_pair, gw_pair):
    p = hlq.hlq_debug_gemm_plan(T, Cin, Cout, rank=8, sms=152)
    assert p["gx"] == gx and p["gw"] == gw and p["in_sequence"] == seq
    assert p["gx_pair"] is gx_pair and p["gw_pair"] is gw_pair


def test_pairs_need_more_than_one_row_tile():
    # a g_x GEMM over 128 tokens, a g_w GEMM over 128 output channels
    p = hlq.hlq_debug_gemm_plan(128, 768, 128, rank=8, sms=152)
    assert p["gx_pair"] is False and p["gw_pair"] is False


def test_plan_rules():
    # a 96-wide tile only where it needs fewer waves than a 128-wide one
    p = hlq.hlq_debug_gemm_plan(12608, 768, 2304, rank=8, sms=152)
    assert p["gw"][0] != 96
    # few tiles and a long contraction: K splits (at most 16, each at least
    # two 1024-code chunks long) with 128-wide tiles; a short one stays unsplit
    p = hlq.hlq_debug_gemm_plan(65536, 256, 128, rank=8, sms=152)
    assert p["gw"] == (128, 16)
    assert hlq.hlq_debug_gemm_plan(4096, 256, 128, rank=8, sms=152)["gw"][1] == 1
    # the E4M3 GEMM never splits
    for T in (256, 4096, 65536):
        assert hlq.hlq_debug_gemm_plan(T, 64, 128, rank=8, sms=152)["gx"][1] == 1
    # more SMs than units on either side: side by side
    assert not hlq.hlq_debug_gemm_plan(16384, 14336, 4096, rank=8, sms=100000)["in_sequence"]


def test_plan_argument_validation():
    with pytest.raises(RuntimeError):
        hlq.hlq_debug_gemm_plan(256, 64, 128, rank=3)
    with pytest.raises(RuntimeError):
        hlq.hlq_debug_gemm_plan(256, 64, 128, sms=0)
