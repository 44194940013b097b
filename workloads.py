"""Seeded synthetic inputs for the HLQ linear-backward workloads.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the method's arithmetic (no transform, no quantizer, no GEMM),
so it can feed both the CPU oracle and the CUDA path.

The five workloads are shape/distribution stand-ins for the layers the HOT
paper times and trains (ViT-B qkv and fc2 on ImageNet, a Llama-3-8B MLP, a
ResNet-50 3x3 conv as an im2col GEMM); no dataset or trained weight is used.

Recipe: values are drawn in fp64 with numpy's PCG64 generator seeded by the
workload's ``data_seed``, rounded to fp32 (round-to-nearest-even) and, for bf16
workloads, from fp32 to bf16 (round-to-nearest-even on the bit pattern).
Draw order is fixed: w, then x, then g_y, then any auxiliary draw (outlier
channel choice).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PER_TENSOR = 0
PER_TOKEN = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    Cin: int
    Cout: int
    dtype: str            # "f32" or "bf16": storage dtype of x, g_y, w
    x_dist: str
    gy_dist: str
    w_std: float
    gran_gy: int          # quantizer granularity of g_y on the g_x path
    gran_w: int = PER_TENSOR
    block: int = 16
    rank: int = 8
    seed: int = 0         # quantization (Philox) seed
    data_seed: int = 0    # numpy seed of the synthetic data

    @property
    def Tp(self) -> int:
        return self.T * self.rank // self.block


WORKLOADS = [
    Workload("single-linear-T256-Cin64-Cout128", 256, 64, 128, "f32",
             "normal1", "normal1", 1.0 / 8.0, PER_TOKEN, data_seed=1),
    Workload("vitb-qkv-T12608-Cin768-Cout2304", 12608, 768, 2304, "bf16",
             "normal1", "normal1e-3", 0.02, PER_TOKEN, data_seed=2),
    Workload("vitb-fc2-T12608-Cin3072-Cout768", 12608, 3072, 768, "bf16",
             "gelu_normal1", "normal1e-3", 0.02, PER_TENSOR, data_seed=3),
    Workload("llama3-8b-down_proj-T16384-Cin14336-Cout4096", 16384, 14336,
             4096, "bf16", "normal1_outlier1pct_x50", "student_t3_1e-3",
             0.02, PER_TOKEN, data_seed=4),
    Workload("resnet50-conv3x3-im2col-T50176-Cin2304-Cout256", 50176, 2304,
             256, "bf16", "relu_normal1", "normal1e-4",
             math.sqrt(2.0 / 2304.0), PER_TENSOR, data_seed=5),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + np.uint32(0x7FFF) + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _gelu_erf(z: np.ndarray) -> np.ndarray:
    from scipy.special import erf
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def _draw_x(rng, dist, T, Cin):
    z = rng.standard_normal((T, Cin))
    if dist == "normal1":
        return z
    if dist == "gelu_normal1":
        return _gelu_erf(z)
    if dist == "relu_normal1":
        return np.maximum(z, 0.0)
    if dist == "normal1_outlier1pct_x50":
        n_out = int(round(0.01 * Cin))
        cols = rng.choice(Cin, size=n_out, replace=False)
        z[:, cols] *= 50.0
        return z
    raise ValueError(dist)


def _draw_gy(rng, dist, T, Cout):
    if dist == "normal1":
        return rng.standard_normal((T, Cout))
    if dist == "normal1e-3":
        return rng.standard_normal((T, Cout)) * 1e-3
    if dist == "normal1e-4":
        return rng.standard_normal((T, Cout)) * 1e-4
    if dist == "student_t3_1e-3":
        return rng.standard_t(3, size=(T, Cout)) * 1e-3
    raise ValueError(dist)


def _store(a64: np.ndarray, dtype: str):
    a32 = a64.astype(np.float32)
    if dtype == "f32":
        return a32, None
    bits = f32_to_bf16_bits(a32)
    return bf16_bits_to_f32(bits), bits


def make_inputs(wl: Workload, T: int | None = None):
    """Draw (x, g_y, w) for a workload.

    Returns a dict with float32 arrays ``x [T,Cin]``, ``g_y [T,Cout]``,
    ``w [Cout,Cin]`` holding exactly the stored values, and for bf16 workloads
    the raw bf16 bit patterns ``x_bits``, ``g_y_bits``, ``w_bits`` (uint16).
    ``T`` may shrink the token count (a multiple of 16) for quick cases; the
    first rows then follow the same distribution but not the same values.
    """
    T = wl.T if T is None else T
    rng = np.random.Generator(np.random.PCG64(wl.data_seed))
    w = rng.standard_normal((wl.Cout, wl.Cin)) * wl.w_std
    x = _draw_x(rng, wl.x_dist, T, wl.Cin)
    gy = _draw_gy(rng, wl.gy_dist, T, wl.Cout)
    out = {}
    for name, a in (("x", x), ("g_y", gy), ("w", w)):
        v, bits = _store(a, wl.dtype)
        out[name] = v
        if bits is not None:
            out[name + "_bits"] = bits
    return out


def make_custom(T: int, Cin: int, Cout: int, dtype: str = "bf16",
                data_seed: int = 0, x_scale: float = 1.0,
                gy_scale: float = 1.0, w_scale: float = 0.05):
    """Plain normal inputs of arbitrary (ragged) shape for parity sweeps."""
    rng = np.random.Generator(np.random.PCG64(data_seed))
    w = rng.standard_normal((Cout, Cin)) * w_scale
    x = rng.standard_normal((T, Cin)) * x_scale
    gy = rng.standard_normal((T, Cout)) * gy_scale
    out = {}
    for name, a in (("x", x), ("g_y", gy), ("w", w)):
        v, bits = _store(a, dtype)
        out[name] = v
        if bits is not None:
            out[name + "_bits"] = bits
    return out
