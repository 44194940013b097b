"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Codes, scales and integer accumulators must match bit for bit; fp32 g_x and
g_w must be within 1e-5 relative of the oracle's fp64 dequant of the same
integers (exactly zero where the accumulator is zero).
"""
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


def _ref_gx(inp, gran, rnd, seed):
    return oracle.gx_path(inp["g_y"], inp["w"], gran_gy=gran, rnd=rnd, seed=seed)


def check_gx(inp, dtype, gran, rnd, seed):
    gy, w = to_dev(inp, "g_y", dtype), to_dev(inp, "w", dtype)
    r = hlq.hlq_debug_gx_parts(gy, w, gran_gy=gran, rnd=rnd, seed=seed)
    ref = _ref_gx(inp, gran, rnd, seed)
    assert_equal(host(r["sgy"]), ref["s_gy"], "s_gy")
    assert_equal(host(r["sw"]), ref["s_w"], "s_w")
    assert_equal(host(r["qgy"]), ref["qY"], "qY")
    assert_equal(host(r["qw"]), ref["qW"], "qW")
    # the same codes in the method's packed int4 layout
    assert_equal(host(r["qgy_packed"]), oracle.pack_int4(ref["qY"]), "qY packed int4")
    assert_equal(host(r["qw_packed"]), oracle.pack_int4(ref["qW"]), "qW packed int4")
    assert_equal(host(r["acc"]).astype(np.int64), ref["acc"], "acc_gx")
    assert_rel(host(r["g_x"]), ref["g_x"], TOL, "g_x")
    # the public entry point runs the same kernels
    gx = hlq.hlq_linear_backward_gx(gy, w, gran_gy=gran, rnd=rnd, seed=seed)
    assert_equal(host(gx), host(r["g_x"]), "g_x public vs parts")
    return r, ref


def check_gw(inp, dtype, rank):
    x, gy = to_dev(inp, "x", dtype), to_dev(inp, "g_y", dtype)
    xbar, sx = hlq.hlq_compress_activation(x, rank=rank)
    qx_ref, sx_ref = oracle.compress_activation(inp["x"], rank)
    assert_equal(host(sx)[0], sx_ref, "s_x")
    assert_equal(host(xbar), qx_ref, "xbar")
    r = hlq.hlq_debug_gw_parts(gy, xbar, sx, rank=rank)
    ref = oracle.gw_path(inp["g_y"], qx_ref, sx_ref, rank)
    assert_equal(host(r["sg"])[0], ref["s_g"], "s_g")
    assert_equal(host(r["qg"]), ref["qG"], "qG")
    assert_equal(host(r["acc"]).astype(np.int64), ref["acc"], "acc_gw")
    assert_rel(host(r["g_w"]), ref["g_w"], TOL, "g_w")
    gw = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=rank)
    assert_equal(host(gw), host(r["g_w"]), "g_w public vs parts")


# ------------------------------------------------------------- transforms

def _adversarial(shape, rng, dtype):
    a = rng.standard_normal(shape)
    # scatter tiny and huge values so some 16-blocks span many binades
    m = rng.random(shape)
    a[m < 0.05] *= 2.0 ** -20
    a[(m >= 0.05) & (m < 0.08)] *= 2.0 ** -70
    a[(m >= 0.08) & (m < 0.10)] *= 2.0 ** 40
    a[(m >= 0.10) & (m < 0.11)] = 0.0
    a[(m >= 0.11) & (m < 0.115)] *= 2.0 ** -130     # subnormal range
    a32 = a.astype(np.float32)
    if dtype == "bf16":
        bits = workloads.f32_to_bf16_bits(a32)
        return workloads.bf16_bits_to_f32(bits), bits
    return a32, None


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_hq_transform_bit_exact(dtype):
    rng = np.random.default_rng(100)
    for rows, cols in [(48, 64), (16, 2304), (96, 128)]:
        v, bits = _adversarial((rows, cols), rng, dtype)
        inp = {"s": v, "s_bits": bits}
        d = to_dev(inp, "s", dtype)
        for axis in (0, 1):
            got = host(hlq.hlq_debug_hq_transform(d, axis))
            want = oracle.hq_transform(v, axis)
            assert_equal(got, want, f"HQ transform axis {axis} {rows}x{cols}")
    assert hlq.hlq_read_device_status(clear=True) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rank", [1, 2, 4, 8, 16])
def test_hla_transform_bit_exact(dtype, rank):
    rng = np.random.default_rng(200 + rank)
    v, bits = _adversarial((80, 48), rng, dtype)
    d = to_dev({"s": v, "s_bits": bits}, "s", dtype)
    got = host(hlq.hlq_debug_hla_transform(d, rank))
    assert_equal(got, oracle.hla_transform(v, rank), f"HLA transform r={rank}")


# ------------------------------------------------------- the two paths

@pytest.mark.parametrize("gran", [workloads.PER_TOKEN, workloads.PER_TENSOR])
@pytest.mark.parametrize("rnd", [oracle.SR, oracle.RNE])
def test_gx_single_linear(gran, rnd):
    wl = workloads.WORKLOADS[0]
    check_gx(workloads.make_inputs(wl), wl.dtype, gran, rnd, seed=0)


def test_gw_single_linear():
    wl = workloads.WORKLOADS[0]
    check_gw(workloads.make_inputs(wl), wl.dtype, wl.rank)


@pytest.mark.parametrize("T,Cin,Cout,dtype", [
    (16, 16, 16, "bf16"),          # one block everywhere
    (48, 80, 144, "bf16"),         # odd block counts
    (272, 96, 2304, "bf16"),       # ragged HLA tile tail (17 token blocks)
    (4112, 176, 48, "bf16"),       # many tiles + ragged tail in T
    (64, 48, 32, "f32"),
    (528, 1040, 64, "f32"),        # Cin not a multiple of 64
])
def test_paths_ragged_shapes(T, Cin, Cout, dtype):
    inp = workloads.make_custom(T, Cin, Cout, dtype, data_seed=T + Cin,
                                gy_scale=1e-3, w_scale=0.02)
    for gran in (workloads.PER_TOKEN, workloads.PER_TENSOR):
        check_gx(inp, dtype, gran, oracle.SR, seed=T * 7 + 1)
    for rank in (1, 2, 4, 8, 16):
        check_gw(inp, dtype, rank)


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_paths_workload_shapes_short(idx):
    """Each workload's Cin/Cout, value distribution and quantizer choice, at
    T = 528 tokens (33 HLA blocks: several tiles and a ragged tail)."""
    wl = workloads.WORKLOADS[idx]
    inp = workloads.make_inputs(wl, T=528)
    check_gx(inp, wl.dtype, wl.gran_gy, oracle.SR, wl.seed)
    check_gw(inp, wl.dtype, wl.rank)


def test_zero_inputs_give_zero_scales_and_outputs():
    T, Cin, Cout = 64, 32, 48
    z = torch.zeros((T, Cout), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((Cout, Cin), dtype=torch.bfloat16, device="cuda")
    r = hlq.hlq_debug_gx_parts(z, w)
    assert torch.all(r["qgy"] == 0) and torch.all(r["sgy"] == 0)
    assert torch.all(r["g_x"] == 0) and torch.all(r["acc"] == 0)
    x = torch.zeros((T, Cin), dtype=torch.bfloat16, device="cuda")
    xb, sx = hlq.hlq_compress_activation(x)
    assert torch.all(xb == 0) and float(sx) == 0.0
    gw = hlq.hlq_linear_backward_gw(z, xb, sx)
    assert torch.all(gw == 0)


def test_empty_token_dim():
    Cin, Cout = 32, 48
    gy = torch.zeros((0, Cout), dtype=torch.bfloat16, device="cuda")
    w = torch.randn((Cout, Cin), device="cuda").to(torch.bfloat16)
    gx = hlq.hlq_linear_backward_gx(gy, w)
    assert gx.shape == (0, Cin)
    x = torch.zeros((0, Cin), dtype=torch.bfloat16, device="cuda")
    xb, sx = hlq.hlq_compress_activation(x)
    assert xb.shape == (Cin, 0)
    gw = hlq.hlq_linear_backward_gw(gy, xb, sx)
    torch.cuda.synchronize()
    assert torch.all(gw == 0)


def test_extreme_magnitudes_clamp_and_scale():
    """Values near the admitted maximum and a single dominant value."""
    T, Cin, Cout = 32, 16, 32
    rng = np.random.default_rng(5)
    gy = rng.standard_normal((T, Cout)).astype(np.float32)
    gy[3, 5] = 1e37
    gy[7] = 0.0
    w = (rng.standard_normal((Cout, Cin)) * 1e-30).astype(np.float32)
    inp = {"g_y": gy, "w": w, "x": rng.standard_normal((T, Cin)).astype(np.float32)}
    for gran in (workloads.PER_TOKEN, workloads.PER_TENSOR):
        check_gx(inp, "f32", gran, oracle.SR, seed=11)
    check_gw(inp, "f32", 8)


def test_nonfinite_input_sets_status_flag():
    hlq.hlq_read_device_status(clear=True)
    gy = torch.randn((32, 32), device="cuda").to(torch.bfloat16)
    gy[4, 9] = float("nan")
    w = torch.randn((32, 16), device="cuda").to(torch.bfloat16)
    hlq.hlq_linear_backward_gx(gy, w)
    assert hlq.hlq_read_device_status(clear=True) & hlq.DEV_NONFINITE
    assert hlq.hlq_read_device_status() == 0


def test_seed_changes_codes_deterministically():
    wl = workloads.WORKLOADS[0]
    inp = workloads.make_inputs(wl)
    gy, w = to_dev(inp, "g_y", "f32"), to_dev(inp, "w", "f32")
    a = hlq.hlq_debug_gx_parts(gy, w, seed=1)["qgy"]
    b = hlq.hlq_debug_gx_parts(gy, w, seed=1)["qgy"]
    c = hlq.hlq_debug_gx_parts(gy, w, seed=(1 << 40) + 1)["qgy"]
    assert torch.equal(a, b) and not torch.equal(a, c)


# ------------------------------------------- accumulator exactness at the limits

def _lossless_rows(signs, scale, H):
    """Rows whose 16-blocks transform (by H16) to exactly 7*scale*signs."""
    T, n = signs.shape
    out = np.zeros((T, n), np.float64)
    for b in range(n // 16):
        out[:, 16 * b:16 * b + 16] = (7.0 * scale * signs[:, 16 * b:16 * b + 16]) @ H / 16.0
    return out.astype(np.float32)


def test_gx_accumulator_exact_at_max_magnitude():
    """All int4 codes +-7 with rows of qY equal to rows of qW: |acc| reaches
    49 * Cout, the largest the g_x GEMM admits a chunk to hold."""
    H = oracle.hadamard16().astype(np.float64)
    rng = np.random.default_rng(31)
    T, Cin, Cout = 256, 64, 4096
    sw = rng.choice([-1.0, 1.0], size=(Cin, Cout))
    sy = rng.choice([-1.0, 1.0], size=(T, Cout))
    sy[:Cin] = sw                      # acc[t, t] = 49 * Cout for t < Cin
    sy[Cin:2 * Cin] = -sw
    gy = _lossless_rows(sy, 2.0 ** -8, H)
    wT = _lossless_rows(sw, 2.0 ** -4, H)          # [Cin, Cout]
    inp = {"g_y": gy, "w": np.ascontiguousarray(wT.T),
           "x": np.zeros((T, Cin), np.float32)}
    r, ref = check_gx(inp, "f32", workloads.PER_TENSOR, oracle.RNE, 0)
    acc = host(r["acc"])
    assert acc[0, 0] == 49 * Cout and acc[Cin, 0] == -49 * Cout


def _hla_lossless(signs, scale, rank=8):
    """Tokens whose HLA coefficients (rank lowest-sequency rows per 16-token
    block) are exactly 127*scale*signs; signs [T', C]."""
    H = oracle.hadamard16().astype(np.float64)
    sigma = oracle.sequency_order()
    Tp, C = signs.shape
    T = Tp // rank * 16
    x = np.zeros((T, C), np.float64)
    for b in range(T // 16):
        c = 127.0 * scale * signs[rank * b:rank * b + rank]        # [rank, C]
        x[16 * b:16 * b + 16] = (H[sigma[:rank]].T @ c) / 16.0
    return x.astype(np.float32)


def test_gw_accumulator_exact_beyond_2_24():
    """All int8 codes +-127 with matching signs: acc = 127^2 * T' = 66e6,
    beyond the 2^24 an fp32 accumulator holds exactly; the chunked drain and
    any K split must still give the exact integer."""
    rng = np.random.default_rng(32)
    T, Cin, Cout, rank = 8192, 32, 48, 8
    Tp = T // 16 * rank
    sx = rng.choice([-1.0, 1.0], size=(Tp, Cin))
    sg = rng.choice([-1.0, 1.0], size=(Tp, Cout))
    sg[:, :Cin] = sx                     # acc[o, o] = 127^2 * T' for o < Cin
    x = _hla_lossless(sx, 2.0 ** -3, rank)
    gy = _hla_lossless(sg, 2.0 ** -9, rank)
    inp = {"x": x, "g_y": gy, "w": np.zeros((Cout, Cin), np.float32)}
    check_gw(inp, "f32", rank)
    xbar, s = hlq.hlq_compress_activation(to_dev(inp, "x", "f32"), rank=rank)
    r = hlq.hlq_debug_gw_parts(to_dev(inp, "g_y", "f32"), xbar, s, rank=rank)
    acc = host(r["acc"])
    assert acc[0, 0] == 127 * 127 * Tp and acc[5, 5] == 127 * 127 * Tp


@pytest.mark.parametrize("idx", [0, 1, 4])
def test_combined_backward_matches_separate_calls(idx):
    """hlq_linear_backward (g_w branch forked onto a second stream) gives
    bit-identical g_x and g_w to the two separate entry points, and its
    output is ordered before later work on the caller's stream."""
    wl = workloads.WORKLOADS[idx]
    inp = workloads.make_inputs(wl, T=min(wl.T, 1024))
    x, gy, w = (to_dev(inp, n, wl.dtype) for n in ("x", "g_y", "w"))
    xbar, sx = hlq.hlq_compress_activation(x, rank=wl.rank)
    gx1 = hlq.hlq_linear_backward_gx(gy, w, gran_gy=wl.gran_gy, seed=3)
    gw1 = hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=wl.rank)
    for _ in range(2):
        gx2, gw2 = hlq.hlq_linear_backward(gy, w, xbar, sx, rank=wl.rank,
                                           gran_gy=wl.gran_gy, seed=3)
        total = gw2.sum() + gx2.sum()   # consumes the outputs on the same stream
        assert torch.equal(gx1, gx2) and torch.equal(gw1, gw2)
        assert torch.isfinite(total)
