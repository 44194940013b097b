"""hadamard_precision_backprop_gb300: GB300 kernels of the HLQ/HOT backward pass.

The compute lives in ``libhlq.so`` (hand-written sm_103a CUDA behind the C
ABI of ``include/hlq.h``); this module is the thin Python binding: it
marshals torch tensors to pointers, allocates outputs and workspaces with
torch, and passes torch's current CUDA stream.  Every step of the path runs
in libhlq's kernels; there is no CPU or PyTorch fallback, and loading fails
loudly when the library has not been built.

Entry points (same names as the C ABI):
  hlq_compress_activation(x, rank)            -> (xbar int8 [Cin, T'], s_x)
  hlq_linear_backward_gx(g_y, w, ...)         -> g_x fp32 [T, Cin]
  hlq_linear_backward_gw(g_y, xbar, s_x, ...) -> g_w fp32 [Cout, Cin]
  hlq_debug_gx_parts / hlq_debug_gw_parts     -> intermediates for checks
  hlq_workspace_bytes, hlq_read_device_status, hlq_status_string
"""
from __future__ import annotations

import ctypes
import os
import threading

PER_TENSOR, PER_TOKEN = 0, 1
RNE, SR = 0, 1
F32, BF16 = 0, 1
OP_COMPRESS_ACTIVATION, OP_BACKWARD_GX, OP_BACKWARD_GW, OP_BACKWARD = 0, 1, 2, 3
OP_SELECT_GRANULARITY, OP_ABLATION_GW_HQ, OP_ABLATION_GX_HLA = 4, 5, 6
OP_BACKWARD_FUSED, OP_LAYER_STEP = 7, 8
XBAR_INT8, XBAR_INT4, XBAR_PER_CHANNEL = 8, 4, 0x100   # format word of the stored activation
DEV_NONFINITE, DEV_TIMEOUT, DEV_BADCODE = 0x1, 0x2, 0x4

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libhlq.so")

EXPORTS = [
    "hlq_workspace_bytes", "hlq_compress_activation", "hlq_linear_backward_gx",
    "hlq_linear_backward_gw", "hlq_debug_gx_parts", "hlq_debug_gw_parts",
    "hlq_read_device_status", "hlq_status_string", "hlq_version",
    "hlq_debug_hq_transform", "hlq_debug_hla_transform",
    "hlq_trace_begin", "hlq_trace_end", "hlq_trace_get", "hlq_trace_free",
    "hlq_debug_reference_gemm", "hlq_debug_tc_gemm", "hlq_debug_tc_gemm_ws_bytes",
    "hlq_linear_backward_gx_noalloc", "hlq_noalloc_scratch_bytes",
    "hlq_linear_backward",
    "hlq_layer_step_host",
    "hlq_layer_step_host_workspace_bytes",
    "hlq_select_gy_granularity",
    "hlq_ablation_gw_hq",
    "hlq_ablation_gx_hla",
    "hlq_linear_backward_fused",
    "hlq_layer_step",
    "hlq_debug_gemm_plan",
    "hlq_debug_wait_timeout",
    "hlq_set_gw_operands", "hlq_get_gw_operands", "hlq_debug_serialize_branches",
]

_lock = threading.Lock()
_lib = None


class HLQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def build_library(force: bool = False) -> str:
    """Compile libhlq.so in-tree (nvcc, sm_103a)."""
    from .build import build as _build
    return _build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded libhlq (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libhlq is not built ({LIB_PATH} missing); run "
                "`python -m hadamard_precision_backprop_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, u64, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_uint64, ctypes.c_size_t)
        sig = {
            "hlq_workspace_bytes": (sz, [i32, i64, i64, i64, i32, i32]),
            "hlq_compress_activation": (i32, [P, i32, i64, i64, i32, i32, i32, P,
                                              P, P, sz, P]),
            "hlq_linear_backward_gx": (i32, [P, P, i32, i64, i64, i64, i32, i32,
                                             i32, i32, u64, P, P, sz, P]),
            "hlq_linear_backward_gw": (i32, [P, i32, P, P, i64, i64, i64, i32,
                                             i32, i32, P, P, sz, P]),
            "hlq_debug_gx_parts": (i32, [P, P, i32, i64, i64, i64, i32, i32,
                                         i32, i32, u64, P, P, sz, P, P, P, P,
                                         P, P, P, P]),
            "hlq_debug_gw_parts": (i32, [P, i32, P, P, i64, i64, i64, i32, i32,
                                         i32, P, P, sz, P, P, P, P]),
            "hlq_read_device_status": (i32, [P, i32, P]),
            "hlq_debug_hq_transform": (i32, [P, i32, i64, i64, i32, P, P]),
            "hlq_debug_hla_transform": (i32, [P, i32, i64, i64, i32, P, P]),
            "hlq_trace_begin": (i32, [i32]),
            "hlq_debug_reference_gemm": (i32, [i32, P, P, i64, i64, i64, P, P]),
            "hlq_debug_tc_gemm": (i32, [i32, P, i64, P, i64, i64, i64, i64, i32,
                                        i32, i32, P, P, sz, P]),
            "hlq_debug_tc_gemm_ws_bytes": (sz, [i64, i64]),
            "hlq_linear_backward_gx_noalloc": (i32, [P, P, i32, i64, i64, i64, i32,
                                                     i32, i32, i32, u64, P, P]),
            "hlq_noalloc_scratch_bytes": (sz, []),
            "hlq_linear_backward": (i32, [P, P, P, P, i32, i64, i64, i64, i32, i32,
                                          i32, i32, i32, i32, u64, P, P, P, sz, P]),
            "hlq_linear_backward_fused": (i32, [P, P, P, P, i32, i64, i64, i64, i32, i32,
                                          i32, i32, i32, i32, u64, P, P, P, sz, P]),
            "hlq_layer_step_host": (i32, [P, P, P, i32, i64, i64, i64, i32, i32, i32,
                                          i32, i32, i32, u64, P, P, P, P, i64, P, sz, P]),
            "hlq_layer_step_host_workspace_bytes": (sz, [i32, i64, i64, i64, i32, i32]),
            "hlq_select_gy_granularity": (i32, [P, i32, i64, i64, i32, ctypes.c_double,
                                                P, P, P, sz, P]),
            "hlq_ablation_gw_hq": (i32, [P, P, i32, i64, i64, i64, i32, i32, u64, P, P, P,
                                         sz, P]),
            "hlq_debug_gemm_plan": (i32, [i64, i64, i64, i32, i32, P, P, P, P, P, P, P]),
            "hlq_debug_wait_timeout": (i32, [u64, P, P]),
            "hlq_layer_step": (i32, [P, P, P, i32, i64, i64, i64, i32, i32, i32, i32, i32,
                                     i32, u64, P, P, P, P, P, sz, P]),
            "hlq_ablation_gx_hla": (i32, [P, P, i32, i64, i64, i64, i32, i32, P, P, P, sz,
                                          P]),
            "hlq_trace_end": (i32, [P]),
            "hlq_trace_get": (i32, [i32, P, P]),
            "hlq_trace_free": (i32, []),
            "hlq_set_gw_operands": (i32, [i32]),
            "hlq_get_gw_operands": (i32, []),
            "hlq_debug_serialize_branches": (i32, [i32]),
            "hlq_status_string": (ctypes.c_char_p, [i32]),
            "hlq_version": (i32, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().hlq_status_string(int(status)).decode()


hlq_status_string = status_string


def _check(rc: int, what: str):
    if rc != 0:
        raise HLQError(rc, what)


# ----------------------------------------------------------------------------
# torch marshalling
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def _need_cuda_contig(*ts, current_device=None):
    """Contiguous CUDA tensors, all on the current device (the library
    launches on the current device and stream)."""
    index = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
        if index is None:
            index = t.device.index
        elif t.device.index != index:
            raise ValueError(f"tensors must be on one device (cuda:{index} and "
                             f"cuda:{t.device.index})")
    if index is not None:
        cur = _torch().cuda.current_device() if current_device is None else current_device
        if index != cur:
            raise ValueError(f"tensors are on cuda:{index} but cuda:{cur} is current; "
                             "make their device current first")


def _need_buf(t, shape, dtype, index, what):
    """A caller-supplied output or buffer: a contiguous CUDA tensor on device
    `index` (the inputs' device) with exactly `shape` (None: any shape) and
    one of the dtypes `dtype`.  The kernels write through these pointers, so
    a wrong device, size or type is refused here rather than written past."""
    if not getattr(t, "is_cuda", False) or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor")
    if t.device.index != index:
        raise ValueError(f"{what} is on cuda:{t.device.index}, the inputs on cuda:{index}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    dts = dtype if isinstance(dtype, tuple) else (dtype,)
    if t.dtype not in dts:
        raise ValueError(f"{what} must be of dtype {' or '.join(map(str, dts))}, "
                         f"not {t.dtype}")


def _ws_bytes(ws, index):
    """Size in bytes of a caller-supplied workspace (any dtype), after the
    same device and contiguity checks as an output."""
    if not getattr(ws, "is_cuda", False) or not ws.is_contiguous():
        raise ValueError("ws must be a contiguous CUDA tensor")
    if ws.device.index != index:
        raise ValueError(f"ws is on cuda:{ws.device.index}, the inputs on cuda:{index}")
    return int(ws.numel()) * int(ws.element_size())


def hlq_workspace_bytes(op: int, T: int, Cin: int, Cout: int, block: int = 16,
                        rank: int = 8) -> int:
    return int(lib().hlq_workspace_bytes(op, T, Cin, Cout, block, rank))


def workspace(op, T, Cin, Cout, block=16, rank=8, device=None):
    torch = _torch()
    n = hlq_workspace_bytes(op, T, Cin, Cout, block, rank)
    return torch.empty(max(n, 256), dtype=torch.uint8,
                       device=device or torch.cuda.current_device())


def _xbar_fmt(xbar_bits: int, per_channel: bool) -> int:
    """Format word of the stored activation: code bits, plus the per-channel
    flag."""
    return int(xbar_bits) | (XBAR_PER_CHANNEL if per_channel else 0)


def _check_xbar_scale(xbar_scale, Cin: int, per_channel: bool):
    need = Cin if per_channel else 1
    if xbar_scale.dtype != _torch().float32 or xbar_scale.numel() != need:
        raise ValueError(f"xbar_scale must hold {need} fp32 value(s)")


def xbar_shape(T: int, Cin: int, rank: int = 8, xbar_bits: int = 8):
    """Shape of the ACBP buffer: [Cin, T'] int8 codes, or [Cin, T'/2] bytes
    of packed int4 codes."""
    Tp = T // 16 * rank
    return (Cin, Tp if xbar_bits == 8 else Tp // 2)


def _check_xbar(xbar, xbar_scale, T: int, Cin: int, rank: int, xbar_bits: int,
                per_channel: bool, index: int):
    """The ACBP buffer and its scales as the library reads or writes them:
    one-byte codes of exactly xbar_shape(...), fp32 scales [1] or [Cin]."""
    torch = _torch()
    _need_buf(xbar, xbar_shape(T, Cin, rank, xbar_bits), (torch.int8, torch.uint8), index,
              "xbar")
    _need_buf(xbar_scale, None, torch.float32, index, "xbar_scale")
    _check_xbar_scale(xbar_scale, Cin, per_channel)


def hlq_compress_activation(x, rank: int = 8, block: int = 16, out=None,
                            scale=None, ws=None, xbar_bits: int = 8, stream=None,
                            xbar_per_channel: bool = False):
    """ACBP: x [T, Cin] -> (codes, fp32 scale [1], or [Cin] with
    xbar_per_channel); codes are int8 [Cin, T*rank/16] (xbar_bits 8) or uint8
    [Cin, T*rank/32] holding two int4 codes per byte (xbar_bits 4)."""
    torch = _torch()
    _need_cuda_contig(x)
    T, Cin = x.shape
    dev = x.device
    if out is None:
        out = torch.empty(xbar_shape(T, Cin, rank, xbar_bits),
                          dtype=torch.int8 if xbar_bits == 8 else torch.uint8,
                          device=dev)
    if scale is None:
        scale = torch.empty(Cin if xbar_per_channel else 1, dtype=torch.float32,
                            device=dev)
    _check_xbar(out, scale, T, Cin, rank, xbar_bits, xbar_per_channel, dev.index)
    if ws is None:
        ws = workspace(OP_COMPRESS_ACTIVATION, T, Cin, 16, block, rank, dev)
    _check(lib().hlq_compress_activation(
        _ptr(x), _dtype_code(x), T, Cin, block, rank,
        _xbar_fmt(xbar_bits, xbar_per_channel), _ptr(out),
        _ptr(scale), _ptr(ws), _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_compress_activation")
    return out, scale


def hlq_linear_backward_gx(g_y, w, gran_gy: int = PER_TOKEN,
                           gran_w: int = PER_TENSOR, rnd: int = SR,
                           seed: int = 0, block: int = 16, out=None, ws=None,
                           stream=None):
    """g_x [T, Cin] (fp32) of y = x w^T from g_y [T, Cout] and w [Cout, Cin]."""
    torch = _torch()
    _need_cuda_contig(g_y, w)
    T, Cout = g_y.shape
    Cout2, Cin = w.shape
    if Cout2 != Cout or g_y.dtype != w.dtype:
        raise ValueError("shape/dtype mismatch between g_y and w")
    dev = g_y.device
    if out is None:
        out = torch.empty((T, Cin), dtype=torch.float32, device=dev)
    _need_buf(out, (T, Cin), torch.float32, dev.index, "out")
    if ws is None:
        ws = workspace(OP_BACKWARD_GX, T, Cin, Cout, block, 16, dev)
    _check(lib().hlq_linear_backward_gx(
        _ptr(g_y), _ptr(w), _dtype_code(g_y), T, Cin, Cout, block, gran_gy,
        gran_w, rnd, seed, _ptr(out), _ptr(ws), _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_linear_backward_gx")
    return out


def hlq_linear_backward_gw(g_y, xbar, xbar_scale, rank: int = 8,
                           block: int = 16, out=None, ws=None, xbar_bits: int = 8,
                           stream=None, xbar_per_channel: bool = False):
    """g_w [Cout, Cin] (fp32) from g_y [T, Cout] and the ACBP buffer."""
    torch = _torch()
    _need_cuda_contig(g_y, xbar, xbar_scale)
    T, Cout = g_y.shape
    Cin = xbar.shape[0]
    dev = g_y.device
    _check_xbar(xbar, xbar_scale, T, Cin, rank, xbar_bits, xbar_per_channel, dev.index)
    if out is None:
        out = torch.empty((Cout, Cin), dtype=torch.float32, device=dev)
    _need_buf(out, (Cout, Cin), torch.float32, dev.index, "out")
    if ws is None:
        ws = workspace(OP_BACKWARD_GW, T, Cin, Cout, block, rank, dev)
    _check(lib().hlq_linear_backward_gw(
        _ptr(g_y), _dtype_code(g_y), _ptr(xbar), _ptr(xbar_scale), T, Cin,
        Cout, block, rank, _xbar_fmt(xbar_bits, xbar_per_channel), _ptr(out), _ptr(ws),
        _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_linear_backward_gw")
    return out


def hlq_linear_backward_gx_noalloc(g_y, w, gran_gy: int = PER_TOKEN,
                                   gran_w: int = PER_TENSOR, rnd: int = SR,
                                   seed: int = 0, block: int = 16, out=None,
                                   stream=None):
    """hlq_linear_backward_gx without a workspace: for callers that cannot
    allocate device memory, the library uses its own fixed scratch array
    (see include/hlq.h for the size limit and the sharing rules).  `out`
    lets such callers pass a preallocated g_x as well."""
    torch = _torch()
    _need_cuda_contig(g_y, w)
    T, Cout = g_y.shape
    Cout2, Cin = w.shape
    if Cout2 != Cout or g_y.dtype != w.dtype:
        raise ValueError("shape/dtype mismatch between g_y and w")
    if out is None:
        out = torch.empty((T, Cin), dtype=torch.float32, device=g_y.device)
    _need_buf(out, (T, Cin), torch.float32, g_y.device.index, "out")
    _check(lib().hlq_linear_backward_gx_noalloc(
        _ptr(g_y), _ptr(w), _dtype_code(g_y), T, Cin, Cout, block, gran_gy,
        gran_w, rnd, seed, _ptr(out), _stream(stream)),
        "hlq_linear_backward_gx_noalloc")
    return out


def hlq_linear_backward(g_y, w, xbar, xbar_scale, rank: int = 8,
                        gran_gy: int = PER_TOKEN, gran_w: int = PER_TENSOR,
                        rnd: int = SR, seed: int = 0, block: int = 16,
                        out_gx=None, out_gw=None, ws=None, xbar_bits: int = 8,
                        stream=None, xbar_per_channel: bool = False,
                        fused_gy: bool = False):
    """Both gradients of the layer, the g_x and g_w branches overlapped on
    the GPU: returns (g_x [T, Cin], g_w [Cout, Cin]) fp32.  fused_gy: one
    fused reader of g_y for both paths (hlq_linear_backward_fused; same
    bits, workspace of OP_BACKWARD_FUSED)."""
    torch = _torch()
    _need_cuda_contig(g_y, w, xbar, xbar_scale)
    T, Cout = g_y.shape
    Cin = w.shape[1]
    if w.shape[0] != Cout or g_y.dtype != w.dtype or xbar.shape[0] != Cin:
        raise ValueError("shape/dtype mismatch between g_y, w and xbar")
    dev = g_y.device
    _check_xbar(xbar, xbar_scale, T, Cin, rank, xbar_bits, xbar_per_channel, dev.index)
    if out_gx is None:
        out_gx = torch.empty((T, Cin), dtype=torch.float32, device=dev)
    if out_gw is None:
        out_gw = torch.empty((Cout, Cin), dtype=torch.float32, device=dev)
    _need_buf(out_gx, (T, Cin), torch.float32, dev.index, "out_gx")
    _need_buf(out_gw, (Cout, Cin), torch.float32, dev.index, "out_gw")
    if ws is None:
        ws = workspace(OP_BACKWARD_FUSED if fused_gy else OP_BACKWARD, T, Cin, Cout, block,
                       rank, dev)
    fn = lib().hlq_linear_backward_fused if fused_gy else lib().hlq_linear_backward
    _check(fn(
        _ptr(g_y), _ptr(w), _ptr(xbar), _ptr(xbar_scale), _dtype_code(g_y), T,
        Cin, Cout, block, rank, _xbar_fmt(xbar_bits, xbar_per_channel), gran_gy,
        gran_w, rnd, seed, _ptr(out_gx),
        _ptr(out_gw), _ptr(ws), _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_linear_backward_fused" if fused_gy else "hlq_linear_backward")
    return out_gx, out_gw


def hlq_layer_step(x, g_y, w, rank: int = 8, gran_gy: int = PER_TOKEN,
                   gran_w: int = PER_TENSOR, rnd: int = SR, seed: int = 0, block: int = 16,
                   out_gx=None, out_gw=None, xbar=None, xbar_scale=None, ws=None,
                   xbar_bits: int = 8, xbar_per_channel: bool = False, stream=None):
    """The ACBP compression of x and both gradients in one call (the
    compression overlaps the g_x branch): returns (g_x, g_w, xbar,
    xbar_scale)."""
    torch = _torch()
    _need_cuda_contig(x, g_y, w)
    T, Cout = g_y.shape
    Cin = w.shape[1]
    if w.shape[0] != Cout or tuple(x.shape) != (T, Cin) or not (x.dtype == g_y.dtype == w.dtype):
        raise ValueError("shape/dtype mismatch between x, g_y and w")
    dev = g_y.device
    if out_gx is None:
        out_gx = torch.empty((T, Cin), dtype=torch.float32, device=dev)
    if out_gw is None:
        out_gw = torch.empty((Cout, Cin), dtype=torch.float32, device=dev)
    if xbar is None:
        xbar = torch.empty(xbar_shape(T, Cin, rank, xbar_bits),
                           dtype=torch.int8 if xbar_bits == 8 else torch.uint8, device=dev)
    if xbar_scale is None:
        xbar_scale = torch.empty(Cin if xbar_per_channel else 1, dtype=torch.float32,
                                 device=dev)
    _need_buf(out_gx, (T, Cin), torch.float32, dev.index, "out_gx")
    _need_buf(out_gw, (Cout, Cin), torch.float32, dev.index, "out_gw")
    _check_xbar(xbar, xbar_scale, T, Cin, rank, xbar_bits, xbar_per_channel, dev.index)
    if ws is None:
        ws = workspace(OP_LAYER_STEP, T, Cin, Cout, block, rank, dev)
    _check(lib().hlq_layer_step(
        _ptr(x), _ptr(g_y), _ptr(w), _dtype_code(g_y), T, Cin, Cout, block, rank,
        _xbar_fmt(xbar_bits, xbar_per_channel), gran_gy, gran_w, rnd, seed, _ptr(out_gx),
        _ptr(out_gw), _ptr(xbar), _ptr(xbar_scale), _ptr(ws), _ws_bytes(ws, dev.index),
        _stream(stream)),
        "hlq_layer_step")
    return out_gx, out_gw, xbar, xbar_scale


def _need_cpu_contig(*ts):
    for t in ts:
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("host tensors must be contiguous CPU tensors")


def _need_host_out(t, shape, what):
    """A caller-supplied host output: a contiguous fp32 CPU tensor of exactly
    `shape` (the library's copies write its whole extent)."""
    _need_cpu_contig(t)
    if tuple(t.shape) != tuple(shape) or t.dtype != _torch().float32:
        raise ValueError(f"{what} must be a float32 CPU tensor of shape {tuple(shape)}")


def hlq_layer_step_host_workspace_bytes(dtype_code: int, T: int, Cin: int, Cout: int,
                                        block: int = 16, rank: int = 8) -> int:
    return int(lib().hlq_layer_step_host_workspace_bytes(dtype_code, T, Cin, Cout, block,
                                                         rank))


def hlq_layer_step_host(x, g_y, w, xbar, xbar_scale, rank: int = 8,
                        gran_gy: int = PER_TOKEN, gran_w: int = PER_TENSOR,
                        rnd: int = SR, seed: int = 0, block: int = 16,
                        out_gx=None, out_gw=None, ws=None, chunk_tokens: int = 0,
                        xbar_bits: int = 8, stream=None, xbar_per_channel: bool = False):
    """One layer step from host tensors (x, g_y, w on the CPU, pinned for
    speed): compresses x into the device buffers xbar / xbar_scale and
    returns host (g_x, g_w) fp32.  Asynchronous on `stream`: synchronize it
    before reading the results."""
    torch = _torch()
    _need_cpu_contig(x, g_y, w, out_gx, out_gw)
    _need_cuda_contig(xbar, xbar_scale)
    T, Cout = g_y.shape
    Cin = w.shape[1]
    if w.shape[0] != Cout or tuple(x.shape) != (T, Cin) or not (x.dtype == g_y.dtype == w.dtype):
        raise ValueError("shape/dtype mismatch between x, g_y and w")
    index = xbar.device.index
    _check_xbar(xbar, xbar_scale, T, Cin, rank, xbar_bits, xbar_per_channel, index)
    if out_gx is None:
        out_gx = torch.empty((T, Cin), dtype=torch.float32).pin_memory()
    if out_gw is None:
        out_gw = torch.empty((Cout, Cin), dtype=torch.float32).pin_memory()
    _need_host_out(out_gx, (T, Cin), "out_gx")
    _need_host_out(out_gw, (Cout, Cin), "out_gw")
    dt = _dtype_code(g_y)
    if ws is None:
        n = hlq_layer_step_host_workspace_bytes(dt, T, Cin, Cout, block, rank)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=xbar.device)
    _check(lib().hlq_layer_step_host(
        _ptr(x), _ptr(g_y), _ptr(w), dt, T, Cin, Cout, block, rank,
        _xbar_fmt(xbar_bits, xbar_per_channel), gran_gy, gran_w,
        rnd, seed, _ptr(out_gx), _ptr(out_gw), _ptr(xbar), _ptr(xbar_scale),
        chunk_tokens, _ptr(ws), _ws_bytes(ws, index), _stream(stream)),
        "hlq_layer_step_host")
    return out_gx, out_gw


def hlq_select_gy_granularity(g_y, threshold: float = 1.5, block: int = 16,
                              stream=None, mse=None, choice=None, ws=None):
    """Layer-wise quantizer selection on a calibration sample g_y [T, Cout]:
    returns device tensors (mse [2] fp64: per tensor, per token; choice [1]
    int32: PER_TOKEN or PER_TENSOR); mse / choice / ws may be preallocated."""
    torch = _torch()
    _need_cuda_contig(g_y)
    T, Cout = g_y.shape
    dev = g_y.device
    if mse is None:
        mse = torch.empty(2, dtype=torch.float64, device=dev)
    if choice is None:
        choice = torch.empty(1, dtype=torch.int32, device=dev)
    _need_buf(mse, (2,), torch.float64, dev.index, "mse")
    _need_buf(choice, (1,), torch.int32, dev.index, "choice")
    if ws is None:
        ws = workspace(OP_SELECT_GRANULARITY, T, 16, Cout, block, 8, dev)
    _check(lib().hlq_select_gy_granularity(
        _ptr(g_y), _dtype_code(g_y), T, Cout, block, float(threshold), _ptr(mse),
        _ptr(choice), _ptr(ws), _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_select_gy_granularity")
    return mse, choice


def hlq_ablation_gw_hq(g_y, x, rnd: int = SR, seed: int = 0, block: int = 16,
                       with_acc: bool = False, stream=None, out=None, ws=None):
    """g_w [Cout, Cin] through HQ along tokens (the ablation of the g_w path);
    with_acc also returns the int32 accumulator."""
    torch = _torch()
    _need_cuda_contig(g_y, x)
    T, Cout = g_y.shape
    Cin = x.shape[1]
    if x.shape[0] != T or x.dtype != g_y.dtype:
        raise ValueError("shape/dtype mismatch between g_y and x")
    dev = g_y.device
    gw = (torch.empty((Cout, Cin), dtype=torch.float32, device=dev)
          if out is None else out)
    _need_buf(gw, (Cout, Cin), torch.float32, dev.index, "out")
    acc = (torch.empty((Cout, Cin), dtype=torch.int32, device=dev)
           if with_acc else None)
    if ws is None:
        ws = workspace(OP_ABLATION_GW_HQ, T, Cin, Cout, block, 8, dev)
    _check(lib().hlq_ablation_gw_hq(
        _ptr(g_y), _ptr(x), _dtype_code(g_y), T, Cin, Cout, block, rnd, seed, _ptr(gw),
        _ptr(acc), _ptr(ws), _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_ablation_gw_hq")
    return (gw, acc) if with_acc else gw


def hlq_ablation_gx_hla(g_y, w, rank: int = 8, block: int = 16, with_acc: bool = False,
                        stream=None, out=None, ws=None):
    """g_x [T, Cin] through HLA along Cout with int8 codes (the ablation of
    the g_x path); with_acc also returns the int32 accumulator."""
    torch = _torch()
    _need_cuda_contig(g_y, w)
    T, Cout = g_y.shape
    Cin = w.shape[1]
    if w.shape[0] != Cout or w.dtype != g_y.dtype:
        raise ValueError("shape/dtype mismatch between g_y and w")
    dev = g_y.device
    gx = (torch.empty((T, Cin), dtype=torch.float32, device=dev)
          if out is None else out)
    _need_buf(gx, (T, Cin), torch.float32, dev.index, "out")
    acc = (torch.empty((T, Cin), dtype=torch.int32, device=dev)
           if with_acc else None)
    if ws is None:
        ws = workspace(OP_ABLATION_GX_HLA, T, Cin, Cout, block, rank, dev)
    _check(lib().hlq_ablation_gx_hla(
        _ptr(g_y), _ptr(w), _dtype_code(g_y), T, Cin, Cout, block, rank, _ptr(gx),
        _ptr(acc), _ptr(ws), _ws_bytes(ws, dev.index), _stream(stream)),
        "hlq_ablation_gx_hla")
    return (gx, acc) if with_acc else gx


def hlq_debug_gx_parts(g_y, w, gran_gy=PER_TOKEN, gran_w=PER_TENSOR, rnd=SR,
                       seed=0, block=16, stream=None):
    """g_x plus its intermediates: dict(g_x, qgy, sgy, qw, sw, acc, and the
    codes as packed int4 bytes: qgy_packed [T, Cout/2], qw_packed [Cin,
    Cout/2])."""
    torch = _torch()
    _need_cuda_contig(g_y, w)
    T, Cout = g_y.shape
    Cin = w.shape[1]
    dev = g_y.device
    r = dict(
        g_x=torch.empty((T, Cin), dtype=torch.float32, device=dev),
        qgy=torch.empty((T, Cout), dtype=torch.int8, device=dev),
        sgy=torch.empty(T if gran_gy == PER_TOKEN else 1, dtype=torch.float32,
                        device=dev),
        qw=torch.empty((Cin, Cout), dtype=torch.int8, device=dev),
        sw=torch.empty(1, dtype=torch.float32, device=dev),
        acc=torch.empty((T, Cin), dtype=torch.int32, device=dev),
        qgy_packed=torch.empty((T, Cout // 2), dtype=torch.uint8, device=dev),
        qw_packed=torch.empty((Cin, Cout // 2), dtype=torch.uint8, device=dev),
    )
    ws = workspace(OP_BACKWARD_GX, T, Cin, Cout, block, 16, dev)
    _check(lib().hlq_debug_gx_parts(
        _ptr(g_y), _ptr(w), _dtype_code(g_y), T, Cin, Cout, block, gran_gy,
        gran_w, rnd, seed, _ptr(r["g_x"]), _ptr(ws), _ws_bytes(ws, dev.index),
        _ptr(r["qgy"]), _ptr(r["sgy"]), _ptr(r["qw"]), _ptr(r["sw"]),
        _ptr(r["acc"]), _ptr(r["qgy_packed"]), _ptr(r["qw_packed"]), _stream(stream)),
        "hlq_debug_gx_parts")
    return r


def hlq_debug_gw_parts(g_y, xbar, xbar_scale, rank=8, block=16, xbar_bits=8,
                       stream=None, xbar_per_channel=False):
    """g_w plus its intermediates: dict(g_w, qg, sg, acc)."""
    torch = _torch()
    _need_cuda_contig(g_y, xbar, xbar_scale)
    T, Cout = g_y.shape
    Cin = xbar.shape[0]
    _check_xbar_scale(xbar_scale, Cin, xbar_per_channel)
    Tp = T // 16 * rank
    dev = g_y.device
    r = dict(
        g_w=torch.empty((Cout, Cin), dtype=torch.float32, device=dev),
        qg=torch.empty((Cout, Tp), dtype=torch.int8, device=dev),
        sg=torch.empty(1, dtype=torch.float32, device=dev),
        acc=torch.empty((Cout, Cin), dtype=torch.int32, device=dev),
    )
    ws = workspace(OP_BACKWARD_GW, T, Cin, Cout, block, rank, dev)
    _check(lib().hlq_debug_gw_parts(
        _ptr(g_y), _dtype_code(g_y), _ptr(xbar), _ptr(xbar_scale), T, Cin,
        Cout, block, rank, _xbar_fmt(xbar_bits, xbar_per_channel), _ptr(r["g_w"]), _ptr(ws),
        _ws_bytes(ws, dev.index), _ptr(r["qg"]),
        _ptr(r["sg"]), _ptr(r["acc"]), _stream(stream)), "hlq_debug_gw_parts")
    return r


def hlq_debug_hq_transform(src, axis: int, stream=None):
    """fp32 Hadamard coefficients of src [rows, cols] along cols (axis 0) or
    rows (axis 1), each the exact sum rounded once to fp32."""
    torch = _torch()
    _need_cuda_contig(src)
    rows, cols = src.shape
    y = torch.empty((rows, cols), dtype=torch.float32, device=src.device)
    _check(lib().hlq_debug_hq_transform(_ptr(src), _dtype_code(src), rows,
                                        cols, axis, _ptr(y), _stream(stream)),
           "hlq_debug_hq_transform")
    return y


def hlq_debug_hla_transform(src, rank: int = 8, stream=None):
    """fp32 HLA coefficients [C, T*rank/16] of src [T, C]."""
    torch = _torch()
    _need_cuda_contig(src)
    T, C = src.shape
    out = torch.empty((C, T // 16 * rank), dtype=torch.float32,
                      device=src.device)
    _check(lib().hlq_debug_hla_transform(_ptr(src), _dtype_code(src), T, C,
                                         rank, _ptr(out), _stream(stream)),
           "hlq_debug_hla_transform")
    return out


def hlq_debug_reference_gemm(a, b, stream=None):
    """int32 a @ b^T of int8 code matrices a [M, K], b [N, K] on CUDA cores."""
    torch = _torch()
    _need_cuda_contig(a, b)
    M, K = a.shape
    N = b.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device=a.device)
    _check(lib().hlq_debug_reference_gemm(0, _ptr(a), _ptr(b), M, N, K,
                                          _ptr(acc), _stream(stream)),
           "hlq_debug_reference_gemm")
    return acc


def hlq_debug_wait_timeout(limit_ns: int = 1_000_000, stream=None):
    """Run the bounded-wait failure path once (a wait nothing completes,
    given up after limit_ns): returns the device int32 result (0)."""
    torch = _torch()
    out = torch.full((4,), -1, dtype=torch.int32, device=torch.cuda.current_device())
    _check(lib().hlq_debug_wait_timeout(int(limit_ns), _ptr(out), _stream(stream)),
           "hlq_debug_wait_timeout")
    return out[:1]


def hlq_debug_gemm_plan(T: int, Cin: int, Cout: int, rank: int = 8, sms: int = 152):
    """The GEMM plans of a layer on a GPU with `sms` SMs (host only): dict of
    gx (bn, splits), gw (bn, splits) and in_sequence."""
    vals = [ctypes.c_int(0) for _ in range(7)]
    _check(lib().hlq_debug_gemm_plan(T, Cin, Cout, rank, sms,
                                     *[ctypes.byref(v) for v in vals]),
           "hlq_debug_gemm_plan")
    g = [v.value for v in vals]
    return {"gx": (g[0], g[1]), "gw": (g[2], g[3]), "in_sequence": bool(g[4]),
            "gx_pair": bool(g[5]), "gw_pair": bool(g[6])}


def hlq_debug_tc_gemm(kind, a, b, bn=0, splits=0, pair=-1, stream=None):
    """int32 a @ b^T on the tensor cores with an explicit plan.  kind 0: a, b
    are uint8 E4M3 codes [M, K] / [N, K]; kind 1: fp16 codes; kind 2: a fp16,
    b int8 codes (widened in the GEMM); kind 3: a and b int8.  pair: 1 = CTA
    pairs over 256-row tiles, 0 = one CTA per 128-row tile, -1 = the
    library's choice."""
    torch = _torch()
    _need_cuda_contig(a, b)
    M, K = a.shape
    N = b.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device=a.device)
    nws = int(lib().hlq_debug_tc_gemm_ws_bytes(M, N))
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=a.device)
    _check(lib().hlq_debug_tc_gemm(kind, _ptr(a), K, _ptr(b), K, M, N, K, bn,
                                   splits, pair, _ptr(acc), _ptr(ws),
                                   _ws_bytes(ws, a.device.index),
                                   _stream(stream)), "hlq_debug_tc_gemm")
    return acc


GW_AUTO, GW_WIDEN, GW_INT8_X, GW_INT8_BOTH = 0, 1, 2, 3


def hlq_set_gw_operands(mode: int):
    """How the g_w GEMMs take their int8 operands, for the whole process:
    GW_WIDEN (x-bar widened to fp16 by its own kernel), GW_INT8_X (the GEMM
    widens x-bar tiles in shared memory), GW_INT8_BOTH (the HLA codes of g_y
    stay int8 too), GW_AUTO (the library's default).  Results are identical
    in every mode."""
    _check(lib().hlq_set_gw_operands(int(mode)), "hlq_set_gw_operands")


def hlq_get_gw_operands() -> int:
    return int(lib().hlq_get_gw_operands())


def hlq_debug_serialize_branches(on: bool):
    """Run the branches of hlq_linear_backward / hlq_layer_step on the
    caller's stream one after the other (same kernels, for per-kernel
    timing), or forked again (on=False)."""
    _check(lib().hlq_debug_serialize_branches(1 if on else 0),
           "hlq_debug_serialize_branches")


def hlq_trace_begin(capacity: int = 4096):
    """Start recording per-launch device times of libhlq's kernels."""
    _check(lib().hlq_trace_begin(capacity), "hlq_trace_begin")


_trace_n = 0


def hlq_trace_end(keep: bool = False):
    """Stop tracing; return [(kernel name, ms), ...] in launch order.  With
    keep=True return the number of traced launches and keep the events
    alive (for graph replays: hlq_trace_read() after each replay, then
    hlq_trace_free())."""
    global _trace_n
    L = lib()
    n = ctypes.c_int(0)
    _check(L.hlq_trace_end(ctypes.byref(n)), "hlq_trace_end")
    _trace_n = n.value
    if keep:
        return _trace_n
    out = hlq_trace_read()
    L.hlq_trace_free()
    return out


def hlq_trace_read():
    """Per-launch (name, ms) of the last recording of the traced launches."""
    L = lib()
    out = []
    for i in range(_trace_n):
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        _check(L.hlq_trace_get(i, ctypes.byref(name), ctypes.byref(ms)),
               "hlq_trace_get")
        out.append((name.value.decode(), float(ms.value)))
    return out


def hlq_trace_free():
    lib().hlq_trace_free()


def hlq_read_device_status(clear: bool = False, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib().hlq_read_device_status(ctypes.byref(flags), 1 if clear else 0,
                                        _stream(stream)),
           "hlq_read_device_status")
    return int(flags.value)
