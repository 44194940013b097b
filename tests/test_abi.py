"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no device needed)."""
import ctypes
import os
import re

import pytest

import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    hbuild.build()
    return hlq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hlq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hlq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(hlq.EXPORTS)


def test_status_strings_and_version(L):
    assert hlq.status_string(0) == "HLQ_OK"
    assert hlq.status_string(5) == "HLQ_ERR_WORKSPACE"
    assert hlq.status_string(99) == "HLQ_UNKNOWN_STATUS"
    assert L.hlq_version() == 0x000100


def test_workspace_sizes(L):
    for op in (0, 1, 2):
        n = hlq.hlq_workspace_bytes(op, 12608, 768, 2304, 16, 8)
        assert n > 0 and n % 256 == 0
    # g_x workspace holds one byte per int4 code of g_y and of w
    n = hlq.hlq_workspace_bytes(1, 256, 64, 128)
    assert n >= 256 * 128 + 64 * 128
    assert hlq.hlq_workspace_bytes(9, 16, 16, 16) == 0          # unknown op
    assert hlq.hlq_workspace_bytes(1, -16, 16, 16) == 0


# A 16-byte aligned non-null address.  Every call below has one invalid
# argument, so validation rejects it before any CUDA call: nothing is ever
# launched on these fake pointers.
FAKE = 1 << 20
FAKE_WS = 1 << 24


def gx(L, **kw):
    a = dict(gy=FAKE, w=FAKE, dt=1, T=256, Cin=64, Cout=128, block=16,
             gran_gy=1, gran_w=0, rnd=1, seed=0, gx=FAKE, ws=FAKE_WS,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return L.hlq_linear_backward_gx(
        a["gy"], a["w"], a["dt"], a["T"], a["Cin"], a["Cout"], a["block"],
        a["gran_gy"], a["gran_w"], a["rnd"], a["seed"], a["gx"], a["ws"],
        a["ws_bytes"], a["stream"])


def gw(L, **kw):
    a = dict(gy=FAKE, dt=1, xbar=FAKE, xs=FAKE, T=256, Cin=64, Cout=128,
             block=16, rank=8, bits=8, gw=FAKE, ws=FAKE_WS, ws_bytes=1 << 30,
             stream=None)
    a.update(kw)
    return L.hlq_linear_backward_gw(
        a["gy"], a["dt"], a["xbar"], a["xs"], a["T"], a["Cin"], a["Cout"],
        a["block"], a["rank"], a["bits"], a["gw"], a["ws"], a["ws_bytes"], a["stream"])


def test_gx_argument_validation(L):
    assert gx(L, block=8) == 1
    assert gx(L, dt=5) == 1
    assert gx(L, gran_gy=3) == 1
    assert gx(L, rnd=2) == 1
    assert gx(L, T=17) == 2
    assert gx(L, Cin=-16) == 2
    assert gx(L, Cout=100) == 2
    assert gx(L, gy=FAKE + 4) == 3
    assert gx(L, gx=FAKE + 8) == 3
    assert gx(L, ws=FAKE_WS + 16) == 3
    assert gx(L, gran_w=1) == 4
    assert gx(L, ws_bytes=1024) == 5
    assert gx(L, ws=None) == 5
    assert gx(L, gy=None) == 1
    assert gx(L, Cout=342400) == 6            # 49 * Cout >= 2^24


def test_gw_argument_validation(L):
    assert gw(L, rank=3) == 1
    assert gw(L, rank=32) == 1
    assert gw(L, block=32) == 1
    assert gw(L, xs=None) == 1
    assert gw(L, T=8) == 2
    assert gw(L, xbar=FAKE + 1) == 3
    assert gw(L, ws_bytes=0) == 5
    assert gw(L, T=266304) == 6               # T' * 127^2 >= 2^31
    assert gw(L, bits=6) == 1                 # ACBP storage: 8 or 4 bits
    assert gw(L, bits=4, rank=1) == 4         # int4 codes pack two per byte
    assert gw(L, bits=4, T=266304) != 6       # T' * 127 * 7 < 2^31 still
    assert gw(L, bits=8 | 0x200) == 1         # unknown format flag
    assert gw(L, bits=8 | 0x100, ws_bytes=0) == 5   # per-channel scales: valid
    assert gw(L, bits=4 | 0x100, rank=1) == 4


def test_compress_argument_validation(L):
    f = L.hlq_compress_activation
    assert f(FAKE, 1, 256, 64, 15, 8, 8, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 1
    assert f(FAKE, 1, 256, 64, 16, 5, 8, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 1
    assert f(FAKE, 1, 250, 64, 16, 8, 8, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 2
    assert f(FAKE, 1, 256, 64, 16, 8, 8, FAKE, None, FAKE_WS, 1 << 20, None) == 1
    assert f(FAKE + 2, 1, 256, 64, 16, 8, 8, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 3
    assert f(FAKE, 1, 256, 64, 16, 8, 8, FAKE, FAKE, FAKE_WS, 0, None) == 5
    assert f(FAKE, 1, 256, 64, 16, 8, 2, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 1
    assert f(FAKE, 1, 256, 64, 16, 1, 4, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 4
    assert f(FAKE, 1, 256, 64, 16, 8, 8 | 0x200, FAKE, FAKE, FAKE_WS, 1 << 20, None) == 1
    # one amax slot per channel: the workspace grows with Cin
    need = hlq.hlq_workspace_bytes(hlq.OP_COMPRESS_ACTIVATION, 256, 4096, 16)
    assert need >= 256 + 4096 * 4 and need % 256 == 0
    assert f(FAKE, 1, 256, 4096, 16, 8, 8 | 0x100, FAKE, FAKE, FAKE_WS, need - 256,
             None) == 5


def test_tc_gemm_plan_validation(L):
    f = L.hlq_debug_tc_gemm

    def call(bn=128, splits=1, kind=1, M=256, N=256, K=256, pair=-1):
        return f(kind, FAKE, K, FAKE, K, M, N, K, bn, splits, pair, FAKE, FAKE_WS, 1 << 30,
                 None)

    assert call(bn=64) == 1
    assert call(kind=4) == 1
    assert call(kind=-1) == 1
    assert call(splits=65) == 1
    assert call(splits=-2) == 1
    assert call(kind=0, splits=-1) == 1       # stream-K is for the fp16 GEMM
    assert call(splits=-1, pair=1) == 1       # stream-K takes one CTA per tile
    assert call(kind=0, splits=2) == 1        # the E4M3 GEMM runs unsplit
    assert call(bn=192) == 1
    assert call(M=200) == 2
    assert call(pair=2) == 1
    assert call(pair=-2) == 1
    assert call(bn=96, pair=1) == 1           # CTA pairs take 128- and 256-wide tiles


def test_step_host_validation_and_workspace(L):
    f = L.hlq_layer_step_host
    nb = L.hlq_layer_step_host_workspace_bytes
    assert nb(1, 256, 64, 128, 16, 8) > 0 and nb(1, 256, 64, 128, 16, 8) % 256 == 0
    assert nb(0, 256, 64, 128, 16, 8) > nb(1, 256, 64, 128, 16, 8)  # fp32 inputs
    assert nb(7, 256, 64, 128, 16, 8) == 0 and nb(1, -16, 64, 128, 16, 8) == 0

    def call(**kw):
        a = dict(hx=FAKE, hgy=FAKE, hw=FAKE, dt=1, T=256, Cin=64, Cout=128, block=16,
                 rank=8, bits=8, gran_gy=1, gran_w=0, rnd=1, seed=0, hgx=FAKE, hgw=FAKE,
                 xbar=FAKE, xs=FAKE, chunk=0, ws=FAKE_WS, ws_bytes=1 << 30)
        a.update(kw)
        return f(a["hx"], a["hgy"], a["hw"], a["dt"], a["T"], a["Cin"], a["Cout"],
                 a["block"], a["rank"], a["bits"], a["gran_gy"], a["gran_w"], a["rnd"],
                 a["seed"],
                 a["hgx"], a["hgw"], a["xbar"], a["xs"], a["chunk"], a["ws"],
                 a["ws_bytes"], None)

    assert call(hx=None) == 1
    assert call(hgw=None) == 1
    assert call(chunk=-1) == 1
    assert call(rank=3) == 1
    assert call(T=17) == 2
    assert call(ws_bytes=4096) == 5
    assert call(ws=FAKE_WS + 128) == 3
    assert call(xbar=FAKE + 4) == 3
    assert call(xs=None) == 1
    assert call(gran_w=1) == 4
    assert call(bits=5) == 1


def test_select_granularity_validation(L):
    f = L.hlq_select_gy_granularity
    assert L.hlq_workspace_bytes(4, 256, 16, 128, 16, 8) == 256

    def call(gy=FAKE, T=256, Cout=128, block=16, thr=1.5, mse=FAKE, ch=FAKE,
             ws=FAKE_WS, ws_bytes=256):
        return f(gy, 1, T, Cout, block, thr, mse, ch, ws, ws_bytes, None)

    assert call(mse=None) == 1
    assert call(ch=None) == 1
    assert call(thr=-1.0) == 1
    assert call(thr=float("nan")) == 1
    assert call(T=20) == 2
    assert call(mse=FAKE + 4) == 3
    assert call(gy=FAKE + 2) == 3
    assert call(ws_bytes=128) == 5
    assert call(block=8) == 1


def test_ablation_gw_hq_validation(L):
    f = L.hlq_ablation_gw_hq

    def call(gy=FAKE, x=FAKE, T=256, rnd=1, gw=FAKE, ws=FAKE_WS, ws_bytes=1 << 30):
        return f(gy, x, 1, T, 64, 128, 16, rnd, 0, gw, None, ws, ws_bytes, None)

    need = L.hlq_workspace_bytes(5, 256, 64, 128, 16, 8)
    assert need == 512 + 128 * 256 + 64 * 256
    assert call(x=None) == 1
    assert call(rnd=3) == 1
    assert call(T=40) == 2
    assert call(gw=FAKE + 8) == 3
    assert call(T=342400) == 6                 # 49 * T >= 2^24
    assert call(ws_bytes=need - 256) == 5


def test_ablation_gx_hla_validation(L):
    f = L.hlq_ablation_gx_hla

    def call(gy=FAKE, w=FAKE, T=256, Cout=128, rank=8, gx=FAKE, acc=None, ws=FAKE_WS,
             ws_bytes=1 << 30):
        return f(gy, w, 1, T, 64, Cout, 16, rank, gx, acc, ws, ws_bytes, None)

    need = L.hlq_workspace_bytes(6, 256, 64, 128, 16, 8)
    ld = 128 // 16 * 8                         # Cout' = 64 codes, 16-byte rows
    assert need == 512 + 256 * ld * 2 + 64 * ld * 2
    assert L.hlq_workspace_bytes(6, 256, 64, 128, 16, 1) == 512 + 256 * 16 + 64 * 16
    assert call(w=None) == 1
    assert call(rank=3) == 1
    assert call(T=40) == 2
    assert call(acc=FAKE + 4) == 3
    assert call(Cout=1048576, rank=16) != 6    # Cout' * 127^2 < 2^31 still
    assert call(Cout=16 * 65535 + 16) == 4     # over the transform grid limit
    assert call(ws_bytes=need - 256) == 5


def test_fused_backward_workspace_and_validation(L):
    f = L.hlq_linear_backward_fused
    T, Cin, Cout = 256, 64, 128
    need = L.hlq_workspace_bytes(7, T, Cin, Cout, 16, 8)
    assert need == L.hlq_workspace_bytes(3, T, Cin, Cout, 16, 8) + T * 4
    args = [FAKE, FAKE, FAKE, FAKE, 1, T, Cin, Cout, 16, 8, 8, 1, 0, 1, 0, FAKE, FAKE,
            FAKE_WS]
    assert f(*args, need - 256, None) == 5
    bad = list(args)
    bad[8] = 8                                # block
    assert f(*bad, need, None) == 1
    bad = list(args)
    bad[12] = 1                               # per-token w
    assert f(*bad, need, None) == 4


def test_layer_step_workspace_and_validation(L):
    f = L.hlq_layer_step
    T, Cin, Cout = 256, 64, 128
    need = L.hlq_workspace_bytes(8, T, Cin, Cout, 16, 8)
    assert need == (L.hlq_workspace_bytes(0, T, Cin, Cout, 16, 8) +
                    L.hlq_workspace_bytes(3, T, Cin, Cout, 16, 8))

    def call(**kw):
        a = dict(x=FAKE, gy=FAKE, w=FAKE, dt=1, T=T, Cin=Cin, Cout=Cout, block=16, rank=8,
                 fmt=8, gran_gy=1, gran_w=0, rnd=1, seed=0, gx=FAKE, gw=FAKE, xbar=FAKE,
                 xs=FAKE, ws=FAKE_WS, ws_bytes=need)
        a.update(kw)
        return f(*a.values(), None)

    assert call(ws_bytes=need - 256) == 5
    assert call(x=None) == 1
    assert call(xs=None) == 1
    assert call(fmt=6) == 1
    assert call(x=FAKE + 4) == 3
    assert call(T=40) == 2
    assert call(gran_w=1) == 4


def test_wait_timeout_probe_validation(L):
    f = L.hlq_debug_wait_timeout
    assert f(0, FAKE, None) == 1                  # no limit
    assert f(2_000_000_000, FAKE, None) == 1      # over one second
    assert f(1000, None, None) == 1
    assert f(1000, FAKE + 4, None) == 3


def test_read_status_rejects_null(L):
    assert L.hlq_read_device_status(None, 0, None) == 1


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(hlq, "_lib", None)
    monkeypatch.setattr(hlq, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        hlq.lib()


class _FakeTensor:
    """Stands in for a CUDA tensor: only what the binding's checks read."""

    def __init__(self, index, cuda=True, contiguous=True, shape=(4, 4), dtype=None,
                 itemsize=4):
        import torch
        self.is_cuda = cuda
        self._contiguous = contiguous
        self.device = type("Dev", (), {"index": index})()
        self.shape = shape
        self.dtype = torch.float32 if dtype is None else dtype
        self._itemsize = itemsize

    def is_contiguous(self):
        return self._contiguous

    def numel(self):
        n = 1
        for d in self.shape:
            n *= d
        return n

    def element_size(self):
        return self._itemsize


def test_binding_checks_tensors_and_their_device():
    check = hlq._need_cuda_contig
    check(_FakeTensor(0), None, _FakeTensor(0), current_device=0)
    check(_FakeTensor(1), _FakeTensor(1), current_device=1)
    check(None, current_device=0)                       # nothing to check
    with pytest.raises(ValueError, match="contiguous CUDA"):
        check(_FakeTensor(0, cuda=False), current_device=0)
    with pytest.raises(ValueError, match="contiguous CUDA"):
        check(_FakeTensor(0, contiguous=False), current_device=0)
    with pytest.raises(ValueError, match="one device"):
        check(_FakeTensor(0), _FakeTensor(1), current_device=0)
    with pytest.raises(ValueError, match="is current"):
        check(_FakeTensor(1), _FakeTensor(1), current_device=0)


def test_binding_checks_outputs_and_workspaces():
    """Caller-supplied outputs and workspaces get the inputs' device and
    contiguity checks, an exact shape and dtype, and a byte count that does
    not depend on the workspace's dtype (refused before any launch)."""
    import torch
    buf = hlq._need_buf
    buf(_FakeTensor(0, shape=(8, 4)), (8, 4), torch.float32, 0, "out")
    with pytest.raises(ValueError, match="contiguous CUDA"):
        buf(_FakeTensor(0, cuda=False, shape=(8, 4)), (8, 4), torch.float32, 0, "out")
    with pytest.raises(ValueError, match="contiguous CUDA"):
        buf(_FakeTensor(0, contiguous=False, shape=(8, 4)), (8, 4), torch.float32, 0, "out")
    with pytest.raises(ValueError, match="cuda:1, the inputs on cuda:0"):
        buf(_FakeTensor(1, shape=(8, 4)), (8, 4), torch.float32, 0, "out")
    with pytest.raises(ValueError, match="shape"):     # too small: would be written past
        buf(_FakeTensor(0, shape=(4, 4)), (8, 4), torch.float32, 0, "out")
    with pytest.raises(ValueError, match="dtype"):
        buf(_FakeTensor(0, shape=(8, 4), dtype=torch.float16), (8, 4), torch.float32, 0,
            "out")
    buf(_FakeTensor(0, shape=(3, 2), dtype=torch.uint8), (3, 2), (torch.int8, torch.uint8),
        0, "xbar")
    # workspace bytes = numel x element size, whatever its dtype
    assert hlq._ws_bytes(_FakeTensor(0, shape=(1000,), dtype=torch.uint8, itemsize=1), 0) == 1000
    assert hlq._ws_bytes(_FakeTensor(0, shape=(1000,), itemsize=4), 0) == 4000
    with pytest.raises(ValueError, match="contiguous CUDA"):
        hlq._ws_bytes(_FakeTensor(0, cuda=False, shape=(16,)), 0)
    with pytest.raises(ValueError, match="cuda:2"):
        hlq._ws_bytes(_FakeTensor(2, shape=(16,)), 0)


def test_entry_points_refuse_a_wrong_output_before_calling_the_library(monkeypatch):
    """The entry points check `out` before they reach the library: a stub
    library that fails the test if called proves nothing was launched."""
    import torch

    class _NoCall:
        def __getattr__(self, name):
            raise AssertionError(f"library called: {name}")

    monkeypatch.setattr(hlq, "lib", lambda: _NoCall())
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    gy = _FakeTensor(0, shape=(32, 16), dtype=torch.bfloat16)
    w = _FakeTensor(0, shape=(16, 48), dtype=torch.bfloat16)
    small = _FakeTensor(0, shape=(16, 48))
    ws = _FakeTensor(0, shape=(1 << 20,), dtype=torch.uint8, itemsize=1)
    with pytest.raises(ValueError, match="shape"):
        hlq.hlq_linear_backward_gx(gy, w, out=small, ws=ws)
    with pytest.raises(ValueError, match="shape"):
        hlq.hlq_linear_backward_gx_noalloc(gy, w, out=small)
    wrong_dev = _FakeTensor(1, shape=(32, 48))
    with pytest.raises(ValueError, match="cuda:1"):
        hlq.hlq_linear_backward_gx(gy, w, out=wrong_dev, ws=ws)
    xbar = _FakeTensor(0, shape=(48, 16), dtype=torch.int8, itemsize=1)
    sx = _FakeTensor(0, shape=(1,))
    with pytest.raises(ValueError, match="shape"):       # g_w is [Cout, Cin] = [16, 48]
        hlq.hlq_linear_backward_gw(gy, xbar, sx, out=_FakeTensor(0, shape=(48, 16)), ws=ws)
    with pytest.raises(ValueError, match="xbar must have shape"):
        hlq.hlq_linear_backward_gw(gy, _FakeTensor(0, shape=(48, 8), dtype=torch.int8,
                                                    itemsize=1), sx, ws=ws,
                                   out=_FakeTensor(0, shape=(16, 48)))


def test_gw_operand_mode_is_validated(L):
    """The g_w operand layout switch: known modes round-trip, others are
    refused and leave the setting alone (no GPU needed)."""
    for mode in (hlq.GW_WIDEN, hlq.GW_INT8_X, hlq.GW_INT8_BOTH, hlq.GW_AUTO):
        hlq.hlq_set_gw_operands(mode)
        assert hlq.hlq_get_gw_operands() == mode
    for bad in (4, 7, -1):
        with pytest.raises(hlq.HLQError):
            hlq.hlq_set_gw_operands(bad)
        assert hlq.hlq_get_gw_operands() == hlq.GW_AUTO


def test_serialize_branches_switch_is_validated(L):
    assert L.hlq_debug_serialize_branches(1) == 0
    assert L.hlq_debug_serialize_branches(0) == 0
    assert L.hlq_debug_serialize_branches(2) == 1
    assert L.hlq_debug_serialize_branches(-1) == 1
