"""Helpers shared by the GPU parity tests (marshalling and comparisons)."""
import numpy as np
import torch


def to_dev(inp, name, dtype):
    """Upload a workload tensor with its stored dtype (bf16 bits or fp32)."""
    if dtype == "bf16":
        bits = np.ascontiguousarray(inp[name + "_bits"])
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(inp[name], np.float32)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_rel(gpu, ref, tol=1e-5, what=""):
    """|gpu - ref| <= tol * |ref| element by element; exact where ref == 0."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bad = err > tol * np.abs(ref)
    if np.any(bad):
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements off; e.g. idx {i} gpu "
            f"{gpu.ravel()[i]} ref {ref.ravel()[i]}")


def assert_equal(gpu, ref, what=""):
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if not np.array_equal(gpu, ref):
        bad = np.flatnonzero(gpu.ravel() != ref.ravel())
        raise AssertionError(
            f"{what}: {bad.size} of {gpu.size} differ; first at {bad[:5]}: "
            f"gpu {gpu.ravel()[bad[:5]]} ref {ref.ravel()[bad[:5]]}")
