"""The tensor-core GEMMs alone: exact int32 sums for every tile width and
K split, ragged M/N/K, every operand kind (E4M3 int4 codes; fp16 int8 codes;
int8 codes widened to fp16 in shared memory, for B alone or both operands),
against numpy int64 sums and the CUDA-core reference GEMM."""
import numpy as np
import pytest
import torch

import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild

pytestmark = pytest.mark.gpu

# E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits) bytes of the
# integers 0..7, written out from the format's definition.
E4M3_OF = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, 5: 0x4A, 6: 0x4C, 7: 0x4E}


_E4M3_LUT = np.array([E4M3_OF[abs(v)] | (0x80 if v < 0 else 0) for v in range(-7, 8)],
                     np.uint8)


def e4m3_bytes(codes):
    return _E4M3_LUT[np.asarray(codes) + 7]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()


def _operand(kind, X, which):
    if kind == 0:
        return torch.from_numpy(e4m3_bytes(X)).cuda()
    if kind == 1 or (kind == 2 and which == "a"):
        return torch.from_numpy(X.astype(np.float16)).cuda()
    return torch.from_numpy(X.astype(np.int8)).cuda()


def run(kind, A, B, bn, splits, pair=-1):
    a, b = _operand(kind, A, "a"), _operand(kind, B, "b")
    return hlq.hlq_debug_tc_gemm(kind, a, b, bn=bn, splits=splits, pair=pair)


def test_tc_gemm_pair_one_tile():
    """The smallest CTA-pair GEMM: one 256 x 256 tile (one pair), one and
    several k-blocks, every operand kind; the first GPU check of the pair
    path, kept apart so that it runs before the larger cases."""
    for kind, qmax in ((0, 7), (1, 127), (2, 127), (3, 127)):
        for K in (128, 256, 1024):
            rng = np.random.default_rng(K + kind)
            A = rng.integers(-qmax, qmax + 1, (256, K))
            B = rng.integers(-qmax, qmax + 1, (256, K))
            got = run(kind, A, B, 256, 1, pair=1).cpu().numpy()
            np.testing.assert_array_equal(got.astype(np.int64),
                                          A.astype(np.int64) @ B.astype(np.int64).T)
    assert hlq.hlq_read_device_status() == 0


# Every tile width, unsplit, for every kind, on one CTA per tile and on CTA
# pairs (128- and 256-wide); K splits for the fp16 GEMMs only (the E4M3 GEMM
# runs unsplit: the ABI refuses a split plan for it, which the CPU
# plan-validation test checks).
_KINDS = ((0, 7), (1, 127), (2, 127), (3, 127))
PLANS = ([(kind, qmax, bn, 1, 0) for kind, qmax in _KINDS for bn in (128, 256, 96)]
         + [(kind, qmax, bn, 1, 1) for kind, qmax in _KINDS for bn in (128, 256)]
         + [(kind, 127, bn, splits, 0) for kind in (1, 2, 3)
            for bn, splits in ((128, 3), (256, 2), (96, 2))]
         + [(kind, 127, bn, splits, 1) for kind in (1, 2, 3)
            for bn, splits in ((128, 3), (256, 2))]
         # stream-K: equal k-block runs per SM, partial tiles summed exactly
         + [(kind, 127, bn, -1, 0) for kind in (1, 2, 3) for bn in (128, 256, 96)])


@pytest.mark.parametrize("kind,qmax,bn,splits,pair", PLANS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (16, 32, 16), (272, 400, 208),
                                   (384, 512, 2048), (1040, 144, 4112)])
def test_tc_gemm_exact(kind, qmax, M, N, K, bn, splits, pair):
    rng = np.random.default_rng(M * 7 + N * 3 + K + bn + splits)
    A = rng.integers(-qmax, qmax + 1, (M, K))
    B = rng.integers(-qmax, qmax + 1, (N, K))
    want = A.astype(np.int64) @ B.astype(np.int64).T
    got = run(kind, A, B, bn, splits, pair).cpu().numpy()
    np.testing.assert_array_equal(got.astype(np.int64), want)
    ref = hlq.hlq_debug_reference_gemm(torch.from_numpy(A.astype(np.int8)).cuda(),
                                       torch.from_numpy(B.astype(np.int8)).cuda())
    np.testing.assert_array_equal(ref.cpu().numpy(), got)


def test_tc_gemm_stream_k_tile_boundaries():
    """Stream-K runs that start and end inside tiles, several runs per tile
    and several tiles per run: one 128 x 128 tile of 300 k-blocks shared by
    every SM, and 3 x 5 tiles of 37 k-blocks whose runs cross tile edges."""
    for M, N, K in [(128, 128, 300 * 64), (384, 640, 37 * 64), (400, 272, 2064)]:
        rng = np.random.default_rng(M + N + K)
        A = rng.integers(-127, 128, (M, K))
        B = rng.integers(-127, 128, (N, K))
        want = A.astype(np.int64) @ B.astype(np.int64).T
        for kind in (1, 2):
            for bn in (128, 256):
                got = run(kind, A, B, bn, -1, 0).cpu().numpy()
                np.testing.assert_array_equal(got.astype(np.int64), want)
    assert hlq.hlq_read_device_status() == 0


def test_tc_gemm_library_plan_exact():
    """The plan the library picks for the workload shapes (tile width, K
    split), at full size, checked on sampled rows."""
    for kind, qmax, M, N, K in [(0, 7, 12608, 768, 2304), (1, 127, 2304, 768, 6304),
                                (1, 127, 256, 2304, 25088), (2, 127, 2304, 768, 6304),
                                (3, 127, 256, 2304, 25088), (2, 127, 4096, 2048, 8192),
                                (3, 127, 4096, 2048, 8192)]:
        rng = np.random.default_rng(M + N + K)
        A = rng.integers(-qmax, qmax + 1, (M, K))
        B = rng.integers(-qmax, qmax + 1, (N, K))
        got = run(kind, A, B, 0, 0).cpu().numpy().astype(np.int64)
        rows = rng.choice(M, 64, replace=False)
        np.testing.assert_array_equal(got[rows], A[rows].astype(np.int64) @ B.astype(np.int64).T)


@pytest.mark.parametrize("kind", [1, 2, 3])
def test_tc_gemm_f16_worst_case_magnitude(kind):
    """Every product 127*127 with one sign: |acc| = 16129*K, far above 2^24,
    only exact through the chunked drains (and the int32 split reduction);
    -127 and 127 are also the extreme codes of the in-GEMM widening."""
    M, N, K = 256, 256, 16384
    A = np.full((M, K), 127, np.int64)
    A[1::2] = -127
    B = np.full((N, K), 127, np.int64)
    for splits, pair in ((1, 0), (2, 0), (5, 0), (1, 1), (3, 1), (-1, 0)):
        got = run(kind, A, B, 128, splits, pair).cpu().numpy()
        assert got[0, 0] == 16129 * K and got[1, 0] == -16129 * K
        assert np.all(got[0::2] == 16129 * K) and np.all(got[1::2] == -16129 * K)


def test_tc_gemm_widening_every_code():
    """Every int8 code value (including -128, outside the codes the library
    writes) at every position of a k-block, against a one-hot operand, so
    that each widened code comes out alone: with kind 3 the codes are A
    (acc = A . I = A), with kind 2 they are B (acc = I . B^T = B^T)."""
    K = 256
    P = np.tile(np.arange(-128, 128, dtype=np.int64), (256, 1))
    for r in range(256):
        P[r] = np.roll(P[r], 3 * r + (r >> 7))
    E = np.eye(K, dtype=np.int64)
    for pair in (0, 1):
        got = run(3, P, E, 128, 1, pair).cpu().numpy()
        np.testing.assert_array_equal(got.astype(np.int64), P)
        got = run(2, E, P, 128, 1, pair).cpu().numpy()
        np.testing.assert_array_equal(got.astype(np.int64), P.T)


def test_tc_gemm_e4m3_worst_case_magnitude():
    M, N, K = 128, 256, 4096
    A = np.full((M, K), 7, np.int64)
    A[::3] = -7
    B = np.full((N, K), -7, np.int64)
    want = A[:, :1] * B[:, 0][None, :] * K
    for pair in (0, 1):
        got = run(0, A, B, 256, 1, pair).cpu().numpy()
        np.testing.assert_array_equal(got, want)
