"""CPU oracle of the HLQ/HOT linear-layer backward pass (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product library never imports, links or runs
it, and it shares no code with the CUDA sources.  ``hlq_oracle.c`` holds the
arithmetic (explicit Hadamard matrix, exact transform sums, scalar
quantizers, Philox4x32-10, int64 GEMM, fp64 dequant); this module is ctypes
marshalling plus the composition of those steps into the two gradient paths
of "HLQ: Fast and Efficient Backpropagation via Hadamard Low-rank
Quantization" (TL;DR formulas) and "HOT: Hadamard-based Optimized Training"
(Approach).

Parity status: every function below is pinned by the CPU tests
(closed forms, brute force on tiny shapes, quantizer error bounds; the
Philox4x32-10 words against cuRAND's host-side Philox4x32-10 generator).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hlq_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libhlq_oracle.so")
_lock = threading.Lock()
_lib = None

PER_TENSOR, PER_TOKEN = 0, 1
RNE, SR = 0, 1
STREAM_GY, STREAM_W = 0, 1
STREAM_GY_T, STREAM_X_T = 2, 3        # the along-tokens HQ of the g_w ablation


def build(force: bool = False) -> str:
    """Compile the oracle with plain gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and \
            os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-fno-fast-math", "-ffp-contract=off", "-Wall",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, u32, u64 = (ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_uint32, ctypes.c_uint64)
            sig = {
                "orc_hadamard16": (i32, [P]),
                "orc_sequency_order": (i32, [P]),
                "orc_exact_sum_f32": (ctypes.c_float, [P, P, i32]),
                "orc_hq_transform": (i32, [P, i64, i64, i32, P]),
                "orc_hla_transform": (i32, [P, i64, i64, i32, P]),
                "orc_hq_transform_f64": (i32, [P, i64, i64, i32, P]),
                "orc_hla_transform_f64": (i32, [P, i64, i64, i32, P]),
                "orc_philox4x32_10": (None, [P, P, P]),
                "orc_philox_word": (u32, [u64, u32, u64]),
                "orc_hq_quantize": (i32, [P, i64, i64, i32, i32, u64, u32, P, P]),
                "orc_hq_quantize_rows": (i32, [P, i64, i64, P, i32,
                                               ctypes.c_float, i32, u64, u32,
                                               P, P]),
                "orc_amax": (ctypes.c_float, [P, i64]),
                "orc_int8_quantize": (i32, [P, i64, P, P]),
                "orc_rne_quantize": (i32, [P, i64, i32, P, P]),
                "orc_pack_int4": (i32, [P, i64, P]),
                "orc_gemm_i64": (None, [P, P, i64, i64, i64, P]),
                "orc_dequant_gx": (None, [P, P, i32, ctypes.c_float, i64, i64, P]),
                "orc_dequant_gw": (None, [P, ctypes.c_float, ctypes.c_float,
                                          i64, i64, P]),
                "orc_dequant_gw_cols": (None, [P, ctypes.c_float, P, i64, i64, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# --------------------------------------------------------------------------
# building blocks
# --------------------------------------------------------------------------

def hadamard16() -> np.ndarray:
    H = np.zeros((16, 16), dtype=np.int32)
    _load().orc_hadamard16(_p(H))
    return H


def sequency_order() -> np.ndarray:
    s = np.zeros(16, dtype=np.int32)
    _check(_load().orc_sequency_order(_p(s)), "sequency_order")
    return s


def exact_sum_f32(h, v) -> np.float32:
    h = np.ascontiguousarray(h, dtype=np.int32)
    v = _f32(v)
    assert h.shape == v.shape and h.ndim == 1
    return np.float32(_load().orc_exact_sum_f32(_p(h), _p(v), len(v)))


def hq_transform(src, axis: int) -> np.ndarray:
    """axis 0: blocks of 16 along columns (g_y [T,Cout]); axis 1: along rows
    (w [Cout,Cin]).  Output has the input's layout, fp32 (exact sum, one RN)."""
    src = _f32(src)
    Y = np.empty_like(src)
    _check(_load().orc_hq_transform(_p(src), src.shape[0], src.shape[1], axis,
                                    _p(Y)), "hq_transform")
    return Y


def hla_transform(src, rank: int) -> np.ndarray:
    """src [T, C] -> [C, T*rank/16] (lowest-sequency rows per 16 tokens)."""
    src = _f32(src)
    T, C = src.shape
    out = np.empty((C, T // 16 * rank), dtype=np.float32)
    _check(_load().orc_hla_transform(_p(src), T, C, rank, _p(out)),
           "hla_transform")
    return out


def hq_transform_f64(src, axis: int) -> np.ndarray:
    src = np.ascontiguousarray(src, dtype=np.float64)
    Y = np.empty_like(src)
    _check(_load().orc_hq_transform_f64(_p(src), src.shape[0], src.shape[1],
                                        axis, _p(Y)), "hq_transform_f64")
    return Y


def hla_transform_f64(src, rank: int) -> np.ndarray:
    src = np.ascontiguousarray(src, dtype=np.float64)
    T, C = src.shape
    out = np.empty((C, T // 16 * rank), dtype=np.float64)
    _check(_load().orc_hla_transform_f64(_p(src), T, C, rank, _p(out)),
           "hla_transform_f64")
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def philox_word(seed: int, stream: int, e: int) -> int:
    return int(_load().orc_philox_word(seed, stream, e))


def hq_quantize(Y, gran: int, rnd: int, seed: int, stream: int):
    """int4 codes [rows, cols] (int8 in [-7,7]) and fp32 scales."""
    Y = _f32(Y)
    rows, cols = Y.shape
    codes = np.empty((rows, cols), dtype=np.int8)
    scales = np.empty(rows if gran == PER_TOKEN else 1, dtype=np.float32)
    _check(_load().orc_hq_quantize(_p(Y), rows, cols, gran, rnd, seed, stream,
                                   _p(codes), _p(scales)), "hq_quantize")
    return codes, scales


def hq_quantize_rows(Yrows, row_ids, gran: int, rnd: int, seed: int,
                     stream: int, tensor_amax=0.0):
    """Quantize some rows of a larger transformed tensor (row numbers
    ``row_ids`` in the full tensor; ``tensor_amax`` = its max |Y| for the
    per-tensor scale)."""
    Yrows = _f32(Yrows)
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    n, cols = Yrows.shape
    assert ids.shape == (n,)
    codes = np.empty((n, cols), dtype=np.int8)
    scales = np.empty(n if gran == PER_TOKEN else 1, dtype=np.float32)
    _check(_load().orc_hq_quantize_rows(_p(Yrows), n, cols, _p(ids), gran,
                                        float(tensor_amax), rnd, seed, stream,
                                        _p(codes), _p(scales)),
           "hq_quantize_rows")
    return codes, scales


def amax(v) -> np.float32:
    v = _f32(v)
    return np.float32(_load().orc_amax(_p(v), v.size))


def int8_quantize(v):
    v = _f32(v)
    codes = np.empty(v.shape, dtype=np.int8)
    s = np.zeros(1, dtype=np.float32)
    _check(_load().orc_int8_quantize(_p(v), v.size, _p(codes), _p(s)),
           "int8_quantize")
    return codes, np.float32(s[0])


def rne_quantize(v, qmax: int):
    """Per-tensor RNE quantizer with qmax 127 (int8) or 7 (int4)."""
    v = _f32(v)
    codes = np.empty(v.shape, dtype=np.int8)
    s = np.zeros(1, dtype=np.float32)
    _check(_load().orc_rne_quantize(_p(v), v.size, int(qmax), _p(codes), _p(s)),
           "rne_quantize")
    return codes, np.float32(s[0])


def pack_int4(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.int8)
    packed = np.empty(c.shape[:-1] + (c.shape[-1] // 2,), dtype=np.uint8)
    _check(_load().orc_pack_int4(_p(c), c.size, _p(packed)), "pack_int4")
    return packed


def gemm_i64(A, B) -> np.ndarray:
    """C = A . B^T with A [M,K], B [N,K] int8, int64 sums."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    C = np.empty((M, N), dtype=np.int64)
    _load().orc_gemm_i64(_p(A), _p(B), M, N, K, _p(C))
    return C


def dequant_gx(acc, s_gy, gran_gy: int, s_w) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    s_gy = _f32(s_gy)
    T, Cin = acc.shape
    out = np.empty((T, Cin), dtype=np.float64)
    _load().orc_dequant_gx(_p(acc), _p(s_gy), gran_gy, float(s_w), T, Cin,
                           _p(out))
    return out


def dequant_gw(acc, s_g, s_x) -> np.ndarray:
    """g_w = acc * s_g * s_x / 16; s_x a scalar (per tensor) or one scale per
    input channel (column of g_w)."""
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    Cout, Cin = acc.shape
    out = np.empty((Cout, Cin), dtype=np.float64)
    if np.size(s_x) == 1 and Cin != 1:
        sx0 = float(np.asarray(s_x, dtype=np.float32).reshape(-1)[0])
        _load().orc_dequant_gw(_p(acc), float(s_g), sx0, Cout, Cin, _p(out))
    else:
        sx = _f32(s_x).reshape(-1)
        assert sx.size == Cin
        _load().orc_dequant_gw_cols(_p(acc), float(s_g), _p(sx), Cout, Cin, _p(out))
    return out


# --------------------------------------------------------------------------
# the three steps of the backward pass, composed
# --------------------------------------------------------------------------

def gx_path(g_y, w, gran_gy=PER_TOKEN, rnd=SR, seed=0, rows=None):
    """Activation-gradient path g_x = g_y . w with int4 HQ.

    g_y [T, Cout], w [Cout, Cin] (fp32 values).  Returns a dict:
    qY [T, Cout] int8 codes, s_gy, qW [Cin, Cout] int8 codes (transposed,
    contraction dim contiguous), s_w, acc [T, Cin] int64, g_x [T, Cin] fp64.
    ``rows`` (optional index array) restricts acc/g_x to those tokens; the
    codes and scales are always computed for the whole tensors.
    """
    Y = hq_transform(g_y, axis=0)
    qY, s_gy = hq_quantize(Y, gran_gy, rnd, seed, STREAM_GY)
    Wt = hq_transform(w, axis=1)                      # [Cout, Cin]
    qWt, s_w = hq_quantize(Wt, PER_TENSOR, rnd, seed, STREAM_W)
    qW = np.ascontiguousarray(qWt.T)                  # [Cin, Cout]
    sel = np.arange(qY.shape[0]) if rows is None else np.asarray(rows)
    acc = gemm_i64(qY[sel], qW)
    s_sel = s_gy[sel] if gran_gy == PER_TOKEN else s_gy
    g_x = dequant_gx(acc, s_sel, gran_gy, s_w[0])
    return dict(Y=Y, qY=qY, s_gy=s_gy, Wt=Wt, qW=qW, s_w=s_w, acc=acc,
                g_x=g_x, rows=sel)


def hq_mse(Y, gran: int) -> float:
    """Mean squared error of the int4 HQ quantizer with round-to-nearest-even
    on transformed values Y [T, Cout] at granularity `gran`: mean over all
    elements of (q * s - Y)^2, each term exact in fp64 before squaring."""
    q, s = hq_quantize(Y, gran, RNE, 0, STREAM_GY)
    sc = (np.asarray(s, np.float64)[:, None] if gran == PER_TOKEN
          else np.float64(s[0]))
    err = q.astype(np.float64) * sc - np.asarray(Y, np.float64)
    return float(np.mean(err * err))


def lqs_select(g_y, threshold: float = 1.5):
    """Layer-wise quantizer selection for the HQ of g_y (HOT summary page,
    Approach: per-token or per-tensor quantizer chosen per layer; Limitations:
    the choice comes from calibration data, switching where the two
    quantizers' errors differ by half): per-token iff the
    per-tensor MSE exceeds the per-token MSE by more than 50 %.  Returns
    (choice, mse_per_tensor, mse_per_token)."""
    Y = hq_transform(g_y, axis=0)
    m_tensor = hq_mse(Y, PER_TENSOR)
    m_token = hq_mse(Y, PER_TOKEN)
    choice = PER_TOKEN if m_tensor > threshold * m_token else PER_TENSOR
    return choice, m_tensor, m_token


def gw_hq_path(g_y, x, rnd=SR, seed=0, rows=None):
    """Ablation of the weight-gradient path (HOT summary page, ablation
    table: Hadamard-transformed 4-bit quantization on a gradient path, the
    table's path labels read as swapped since as printed they contradict the
    method's assignment of HQ to g_x and HLA to g_w; here on the
    weight-gradient path in place of HLA + int8): g_y and x are both
    transformed along tokens in blocks of 16 (the g_w contraction dim),
    quantized to int4 per tensor (SR on Philox streams 2 and 3, element
    index t*C + c of the transformed [T, C] tensor), and
    g_w = (1/16) acc * s_g * s_x with acc = qGᵀ qX exact over T.
    Returns qG [Cout, T], s_g, qX [Cin, T], s_x, acc, g_w (``rows``: output
    channels to compute)."""
    Yg = hq_transform(g_y, axis=1)                   # along tokens
    qg, s_g = hq_quantize(Yg, PER_TENSOR, rnd, seed, STREAM_GY_T)
    Yx = hq_transform(x, axis=1)
    qx, s_x = hq_quantize(Yx, PER_TENSOR, rnd, seed, STREAM_X_T)
    qG = np.ascontiguousarray(qg.T)                  # [Cout, T]
    qX = np.ascontiguousarray(qx.T)                  # [Cin, T]
    sel = np.arange(qG.shape[0]) if rows is None else np.asarray(rows)
    acc = gemm_i64(qG[sel], qX)
    g_w = dequant_gw(acc, s_g[0], s_x[0])
    return dict(qG=qG, s_g=s_g, qX=qX, s_x=s_x, acc=acc, g_w=g_w, rows=sel)


def gx_hla_path(g_y, w, rank=8, rows=None):
    """Ablation of the activation-gradient path (HOT summary page, ablation
    table: internal HLA on a gradient path, the table's path labels read as
    swapped as for gw_hq_path; here on the activation-gradient path, with
    the int8 quantizer HLA is paired with on the g_w path): the
    contraction dim of g_x = g_y . w is Cout, so g_y (along its rows) and w
    (along its first dim) both keep the `rank` lowest-sequency Walsh rows of
    each 16-block of Cout,
      Gb[t, r*b + k] = RN_f32(sum_j H16[sigma(k)][j] g_y[t, 16b + j]),
      Wb[i, r*b + k] = RN_f32(sum_j H16[sigma(k)][j] w[16b + j, i]),
    per-tensor RNE int8 codes, acc = qG . qW^T exact over Cout*rank/16, and
    g_x = acc * s_g * s_w / 16.  Returns Gb, qG [T, Cout'], s_g, Wb, qW
    [Cin, Cout'], s_w, acc [T, Cin], g_x (``rows``: tokens to compute)."""
    Gb = hla_transform(np.ascontiguousarray(_f32(g_y).T), rank)   # [T, Cout']
    Wb = hla_transform(w, rank)                                    # [Cin, Cout']
    qG, s_g = int8_quantize(Gb)
    qW, s_w = int8_quantize(Wb)
    sel = np.arange(qG.shape[0]) if rows is None else np.asarray(rows)
    acc = gemm_i64(qG[sel], qW)
    g_x = dequant_gx(acc, np.array([s_g], np.float32), PER_TENSOR, s_w)
    return dict(Gb=Gb, qG=qG, s_g=s_g, Wb=Wb, qW=qW, s_w=s_w, acc=acc, g_x=g_x,
                rows=sel)


def compress_activation(x, rank=8, bits=8, per_channel=False):
    """ACBP at forward time: x [T, Cin] -> codes [Cin, T*rank/16] (int8
    values: [-127, 127] for bits=8, [-7, 7] for bits=4; pack_int4 gives the
    stored nibbles of the latter) and the per-tensor scale.

    per_channel: one scale per input channel instead (a row of the code
    matrix; the reading of "per-token vs per-tensor" granularity carried to
    the stored activation, whose token dim is the g_w contraction dim, so
    only a per-channel scale factors out of the integer GEMM).  Each row is
    quantized on its own with the same RNE rule; returns an fp32 array
    [Cin] of scales."""
    Xb = hla_transform(x, rank)
    qmax = 127 if bits == 8 else 7
    if not per_channel:
        return rne_quantize(Xb, qmax)
    q = np.empty(Xb.shape, dtype=np.int8)
    s = np.empty(Xb.shape[0], dtype=np.float32)
    for c in range(Xb.shape[0]):
        q[c], s[c] = rne_quantize(Xb[c], qmax)
    return q, s


def gw_path(g_y, xbar_codes, s_x, rank=8, rows=None):
    """Weight-gradient path g_w = (1/16) gbar_y^T xbar with HLA + int8.

    g_y [T, Cout]; xbar_codes [Cin, T'] int8; s_x fp32 (a scalar, or one
    scale per input channel from compress_activation(per_channel=True)).
    Returns qG
    [Cout, T'] int8, s_g, acc [Cout, Cin] int64 and g_w [Cout, Cin] fp64
    (``rows`` restricts acc/g_w to those output channels)."""
    Gb = hla_transform(g_y, rank)
    qG, s_g = int8_quantize(Gb)
    sel = np.arange(qG.shape[0]) if rows is None else np.asarray(rows)
    acc = gemm_i64(qG[sel], xbar_codes)
    g_w = dequant_gw(acc, s_g, s_x)
    return dict(Gb=Gb, qG=qG, s_g=s_g, acc=acc, g_w=g_w, rows=sel)
