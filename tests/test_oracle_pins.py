"""Pins of the CPU oracle against what the method and the mathematics fix.

None of these re-derives a value with the oracle's own code: each compares
the oracle with a library routine (scipy's Hadamard matrix, numpy fp64
matmul, cuRAND's host-side Philox4x32-10 generator), a closed form of the
method, exact rational arithmetic, brute force on tiny inputs, or an error
bound of the quantizer.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle
from tests.exact_ref import exact_signed_sum, round_fraction_to_f32

H_SCIPY = scipy.linalg.hadamard(16).astype(np.int64)


def gray_bitrev_sequency(k):
    """Walsh (sequency) order of Sylvester rows: row = bitrev4(gray(k))."""
    g = k ^ (k >> 1)
    return int(f"{g:04b}"[::-1], 2)


def sign_changes(row):
    return int(np.sum(row[1:] != row[:-1]))


# ------------------------------------------------------------------ Hadamard

def test_hadamard_matches_scipy_sylvester():
    H = oracle.hadamard16().astype(np.int64)
    assert np.array_equal(H, H_SCIPY)


def test_hadamard_orthogonal_up_to_16():
    H = oracle.hadamard16().astype(np.int64)
    assert np.array_equal(H @ H.T, 16 * np.eye(16, dtype=np.int64))


def test_sequency_order_gray_code_and_golden():
    sigma = oracle.sequency_order()
    assert [int(s) for s in sigma] == [gray_bitrev_sequency(k) for k in range(16)]
    golden = [int(t) for t in open(
        __file__.replace("test_oracle_pins.py", "golden/sequency16.txt")
    ).read().split("#")[0].split()]
    assert [int(s) for s in sigma] == golden
    for k in range(16):
        assert sign_changes(H_SCIPY[sigma[k]]) == k
    # rank 8 keeps exactly the even Sylvester rows
    assert sorted(int(s) for s in sigma[:8]) == [0, 2, 4, 6, 8, 10, 12, 14]


# ------------------------------------------------------------ exact sums

def _adversarial_vectors(rng):
    out = []
    for spread in (0, 5, 12, 13, 20, 25, 26, 41, 42, 60, 100, 200):
        mant = rng.standard_normal(16)
        exps = rng.integers(-spread // 2 - 1, spread // 2 + 1, 16)
        exps[0], exps[1] = -spread // 2, spread - spread // 2
        out.append((mant * np.exp2(exps.astype(np.float64))).astype(np.float32))
    # cancellation: big values that cancel, leaving tiny ones
    v = np.zeros(16, np.float32)
    v[0], v[1], v[2] = 2.0 ** 40, 2.0 ** 40, np.float32(1e-30)
    out.append(v)
    # subnormals
    out.append((rng.standard_normal(16) * 1e-40).astype(np.float32))
    v = np.zeros(16, np.float32)
    v[3] = np.float32(1.4e-45)
    v[5] = np.float32(-2.8e-45)
    out.append(v)
    # exact ties at fp32 rounding: 1 + 2^-24 (+ tiny) patterns
    v = np.zeros(16, np.float32)
    v[0], v[1] = 1.0, 2.0 ** -24
    out.append(v)
    v = v.copy()
    v[2] = 2.0 ** -60
    out.append(v)
    v = np.zeros(16, np.float32)
    v[0], v[1] = 1.0 + 2.0 ** -23, 2.0 ** -24
    out.append(v)
    # all zero, signed zeros
    out.append(np.zeros(16, np.float32))
    out.append(-np.zeros(16, np.float32))
    # large magnitudes
    out.append((rng.standard_normal(16) * 1e37).astype(np.float32))
    return out


def test_exact_sum_brute_force_fractions():
    rng = np.random.default_rng(7)
    H = oracle.hadamard16()
    vecs = _adversarial_vectors(rng) + [
        rng.standard_normal(16).astype(np.float32) for _ in range(20)]
    for v in vecs:
        for i in range(16):
            for hrow in (H[i], -H[i]):
                got = oracle.exact_sum_f32(hrow, v)
                want = exact_signed_sum(hrow, v)
                assert got == want or (got == 0 and want == 0), (v, i, got, want)


def test_round_to_f32_ties_to_even():
    # 1 + 2^-24 is a tie between 1 and 1+2^-23: even mantissa is 1
    H1 = np.ones(2, np.int32)
    assert oracle.exact_sum_f32(H1, np.array([1.0, 2.0 ** -24], np.float32)) == 1.0
    # 1+2^-23 + 2^-24 ties between 1+2^-23 (odd) and 1+2^-22 (even)
    got = oracle.exact_sum_f32(H1, np.array([1.0 + 2.0 ** -23, 2.0 ** -24], np.float32))
    assert got == np.float32(1.0 + 2.0 ** -22)
    # just above a tie rounds up
    H3 = np.ones(3, np.int32)
    got = oracle.exact_sum_f32(H3, np.array([1.0, 2.0 ** -24, 2.0 ** -70], np.float32))
    assert got == np.float32(1.0 + 2.0 ** -23)


# ------------------------------------------------------------ transforms

def _blockdiag_H(n):
    return np.kron(np.eye(n // 16, dtype=np.int64), H_SCIPY)


def test_hq_transform_equals_fp64_matmul_when_exact():
    # bf16-like values with a small exponent spread: fp64 sums are exact,
    # so RN_f32(fp64 matmul) is the exactly rounded sum.
    rng = np.random.default_rng(1)
    g = (rng.standard_normal((8, 64)) * 0.01).astype(np.float32)
    g = np.round(g * 2 ** 12) / 2 ** 12
    g = g.astype(np.float32)
    D = _blockdiag_H(64)
    want = (g.astype(np.float64) @ D.T).astype(np.float32)
    assert np.array_equal(oracle.hq_transform(g, 0), want)
    w = g.T.copy()                              # [64, 8], blocks along rows
    want_w = (D @ w.astype(np.float64)).astype(np.float32)
    assert np.array_equal(oracle.hq_transform(w, 1), want_w)


def test_hq_transform_brute_force_adversarial():
    rng = np.random.default_rng(3)
    vecs = _adversarial_vectors(rng)
    g = np.stack(vecs[:4]).astype(np.float32)        # [4, 16]
    Y = oracle.hq_transform(np.concatenate([g, g[::-1]], 1), 0)
    for r in range(4):
        for i in range(16):
            assert Y[r, i] == exact_signed_sum(H_SCIPY[i], g[r])
            assert Y[r, 16 + i] == exact_signed_sum(H_SCIPY[i], g[3 - r])
    Yw = oracle.hq_transform(np.ascontiguousarray(g.T), 1)   # [16, 4]
    for c in range(4):
        for i in range(16):
            assert Yw[i, c] == exact_signed_sum(H_SCIPY[i], g[c])


def test_hla_transform_matches_selection_matrix():
    rng = np.random.default_rng(2)
    T, C = 64, 24
    x = np.round(rng.standard_normal((T, C)) * 2 ** 10) / 2 ** 10
    x = x.astype(np.float32)
    for rank in (1, 2, 4, 8, 16):
        rows = [gray_bitrev_sequency(k) for k in range(rank)]
        P = np.zeros((T // 16 * rank, T), dtype=np.int64)
        for b in range(T // 16):
            for k in range(rank):
                P[b * rank + k, 16 * b:16 * b + 16] = H_SCIPY[rows[k]]
        want = (P @ x.astype(np.float64)).T.astype(np.float32)   # [C, T']
        assert np.array_equal(oracle.hla_transform(x, rank), want), rank


def test_hla_transform_brute_force_adversarial():
    rng = np.random.default_rng(4)
    vecs = _adversarial_vectors(rng)[:6]
    x = np.stack(vecs, axis=1).astype(np.float32)     # [16, 6]
    out = oracle.hla_transform(x, 8)                   # [6, 8]
    for c in range(6):
        for k in range(8):
            want = exact_signed_sum(H_SCIPY[gray_bitrev_sequency(k)], x[:, c])
            assert out[c, k] == want


# ------------------------------------------- closed forms, quantization off

def test_hq_quant_off_reproduces_gy_w():
    """H orthogonal up to 16: (1/16) (g_y D^T)(D w) = g_y w."""
    rng = np.random.default_rng(5)
    T, Cin, Cout = 48, 32, 64
    gy = rng.standard_normal((T, Cout))
    w = rng.standard_normal((Cout, Cin))
    Y = oracle.hq_transform_f64(gy, 0)
    Wt = oracle.hq_transform_f64(w, 1)
    got = Y @ Wt / 16.0
    want = gy @ w
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want)) * Cout


def test_hla_full_rank_quant_off_reproduces_gyT_x():
    rng = np.random.default_rng(6)
    T, Cin, Cout = 64, 24, 40
    gy = rng.standard_normal((T, Cout))
    x = rng.standard_normal((T, Cin))
    G = oracle.hla_transform_f64(gy, 16)
    X = oracle.hla_transform_f64(x, 16)
    got = G @ X.T / 16.0
    want = gy.T @ x
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want)) * T


@pytest.mark.parametrize("rank", [1, 2, 4, 8])
def test_hla_low_rank_quant_off_group_sum_closed_form(rank):
    """Lowest-sequency rows span the vectors constant on runs of 16/rank
    tokens, so (1/16) Gbar^T Xbar = (rank/16) sum_runs S_g S_x^T."""
    rng = np.random.default_rng(10 + rank)
    T, Cin, Cout = 96, 20, 28
    gy = rng.standard_normal((T, Cout))
    x = rng.standard_normal((T, Cin))
    G = oracle.hla_transform_f64(gy, rank)
    X = oracle.hla_transform_f64(x, rank)
    got = G @ X.T / 16.0
    L = 16 // rank
    Sg = gy.reshape(T // L, L, Cout).sum(1)
    Sx = x.reshape(T // L, L, Cin).sum(1)
    want = (rank / 16.0) * (Sg.T @ Sx)
    assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want)) * T


def test_hla_rank8_exact_on_equal_token_pairs():
    rng = np.random.default_rng(9)
    T, Cin, Cout = 64, 12, 20
    gy = np.repeat(rng.standard_normal((T // 2, Cout)), 2, axis=0)
    x = np.repeat(rng.standard_normal((T // 2, Cin)), 2, axis=0)
    G = oracle.hla_transform_f64(gy, 8)
    X = oracle.hla_transform_f64(x, 8)
    assert np.allclose(G @ X.T / 16.0, gy.T @ x, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ quantizers

def test_amax_matches_numpy():
    rng = np.random.default_rng(23)
    cases = [rng.standard_normal(1000).astype(np.float32),
             np.array([-3.0, 2.0, -0.0], np.float32),            # max held by a negative
             np.array([-0.0, 0.0], np.float32),
             np.array([1e-45, -2e-45, 0.0], np.float32),          # subnormals
             np.array([np.finfo(np.float32).max, -np.finfo(np.float32).max], np.float32),
             np.zeros(0, np.float32)]
    for v in cases:
        want = np.float32(np.max(np.abs(v))) if v.size else np.float32(0)
        got = oracle.amax(v)
        assert got == want and not np.signbit(got), v


def test_scale_rule_and_zero_tensor():
    Y = np.array([[0.0, -3.5, 1.0, 2.0]], np.float32)
    q, s = oracle.hq_quantize(Y, oracle.PER_TENSOR, oracle.RNE, 0, 0)
    assert s[0] == np.float32(3.5) / np.float32(7.0)
    assert list(q[0]) == [0, -7, 2, 4]
    q, s = oracle.hq_quantize(np.zeros((3, 16), np.float32), oracle.PER_TOKEN,
                              oracle.SR, 0, 0)
    assert np.all(q == 0) and np.all(s == 0)


def test_rne_error_bound_and_ties():
    rng = np.random.default_rng(11)
    Y = rng.standard_normal((64, 128)).astype(np.float32)
    for gran in (oracle.PER_TENSOR, oracle.PER_TOKEN):
        q, s = oracle.hq_quantize(Y, gran, oracle.RNE, 0, 0)
        sc = s[:, None] if gran == oracle.PER_TOKEN else s[0]
        x = Y / sc                                   # fp32 division, as defined
        assert np.all(np.abs(q) <= 7)
        inside = np.abs(x) <= 7
        assert np.all(np.abs(q[inside] - x[inside]) <= 0.5)
        assert np.all(q[~inside] == np.sign(x[~inside]) * 7)
    # exact ties: amax 7 -> s = 1, values k + 0.5 go to the even neighbour
    Y = np.array([[7.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5]], np.float32)
    q, _ = oracle.hq_quantize(Y, oracle.PER_TENSOR, oracle.RNE, 0, 0)
    assert list(q[0]) == [7, 0, 2, 2, 0, -2, -2, 4]
    v = np.array([127.0, 0.5, 1.5, -2.5, 126.5, -126.5], np.float32)
    q8, s8 = oracle.int8_quantize(v)
    assert s8 == 1.0 and list(q8) == [127, 0, 2, -2, 126, -126]


def test_int8_rne_bound():
    rng = np.random.default_rng(12)
    v = (rng.standard_t(3, 5000) * 1e-3).astype(np.float32)
    q, s = oracle.int8_quantize(v)
    assert s == np.float32(np.max(np.abs(v))) / np.float32(127.0)
    x = v / s
    assert np.all(np.abs(q) <= 127)
    ok = np.abs(x) <= 127
    assert np.all(np.abs(q[ok] - x[ok]) <= 0.5)


def test_int4_acbp_rne_bound_ties_and_int8_equivalence():
    """The int4 storage form of the stored activation: RNE with qmax 7
    (HLQ TL;DR, int4 activation compression).  Error <= s/2 off the clamp,
    exact ties to even, scale RN(amax/7), and qmax 127 is the int8 path."""
    rng = np.random.default_rng(21)
    v = rng.standard_normal(4000).astype(np.float32)
    q, s = oracle.rne_quantize(v, 7)
    assert s == np.float32(np.max(np.abs(v))) / np.float32(7.0)
    x = v / s
    assert np.all(np.abs(q) <= 7)
    ok = np.abs(x) <= 7
    assert np.all(np.abs(q[ok] - x[ok]) <= 0.5)
    assert np.all(q[~ok] == np.sign(x[~ok]) * 7)
    t = np.array([7.0, 0.5, 1.5, 2.5, -0.5, -3.5, 6.5, -6.5], np.float32)
    q, s = oracle.rne_quantize(t, 7)
    assert s == 1.0 and list(q) == [7, 0, 2, 2, 0, -4, 6, -6]
    q127, s127 = oracle.rne_quantize(v, 127)
    q8, s8 = oracle.int8_quantize(v)
    assert s127 == s8 and np.array_equal(q127, q8)
    with pytest.raises(ValueError):
        oracle.rne_quantize(v, 15)


def test_int4_acbp_lossless_gw():
    """With every HLA coefficient of x an integer multiple of amax/7, the
    int4 stored activation loses nothing: g_w equals g_y^T x."""
    rng = np.random.default_rng(22)
    T, Cin, Cout = 64, 20, 24
    gy = np.repeat(rng.integers(-3, 4, (T // 2, Cout)), 2, 0).astype(np.float64)
    x = np.repeat(rng.integers(-1, 2, (T // 2, Cin)), 2, 0).astype(np.float64)
    gy[:16, 0] = 127 / 16.0 * 2
    x[:16, 0] = 7 / 16.0 * 2          # amax of the HLA of x: 7 * 2^-2
    gy = (gy * 2.0 ** -7).astype(np.float32)
    x = (x * 2.0 ** -2).astype(np.float32)
    q, s = oracle.compress_activation(x, 8, bits=4)
    assert np.all(np.abs(q) <= 7)
    Xb = oracle.hla_transform(x, 8)
    assert np.array_equal(q.astype(np.float64) * s, Xb)
    r = oracle.gw_path(gy, q, s, 8)
    want = gy.astype(np.float64).T @ x.astype(np.float64)
    assert np.allclose(r["g_w"], want, rtol=1e-12, atol=1e-15)


def test_lqs_mse_bounds_and_known_choices():
    """Layer-wise quantizer selection: MSE of RNE codes is bounded by s^2/4
    per element (no value clamps with RNE when s = RN(amax/7) rounds up, and
    a clamped value errs by at most s/2 + ulp); values on the code grid give
    zero error; a token a few times larger than the rest makes the
    per-tensor scale too coarse for the others (per-token chosen), while a
    huge one dominates both means (its own error is the same either way);
    identical tokens make both equal (per-tensor kept)."""
    rng = np.random.default_rng(31)
    g = rng.standard_normal((64, 128)).astype(np.float32)
    Y = oracle.hq_transform(g, axis=0)
    for gran in (oracle.PER_TENSOR, oracle.PER_TOKEN):
        _, s = oracle.hq_quantize(Y, gran, oracle.RNE, 0, 0)
        s2 = (np.asarray(s, np.float64) ** 2).mean() if gran == oracle.PER_TOKEN else float(s[0]) ** 2
        m = oracle.hq_mse(Y, gran)
        assert 0 < m <= s2 / 4 * (1 + 1e-6)
    # on the grid: Y = k * s exactly for every element -> zero error
    grid = np.tile(np.arange(-7, 8, dtype=np.float32), (4, 1)) * np.float32(0.25)
    assert oracle.hq_mse(grid, oracle.PER_TENSOR) == 0.0
    g2 = rng.standard_normal((64, 128)).astype(np.float32)
    g2[5] *= 4.0
    choice, mt, mk = oracle.lqs_select(g2)
    assert choice == oracle.PER_TOKEN and mt > 1.5 * mk
    g2[5] *= 250.0
    choice, mt, mk = oracle.lqs_select(g2)
    assert choice == oracle.PER_TENSOR and mk <= mt <= 1.5 * mk
    # identical tokens: per-token scales all equal the per-tensor one
    g3 = np.tile(rng.standard_normal((1, 128)).astype(np.float32), (32, 1))
    choice, mt, mk = oracle.lqs_select(g3)
    assert mt == mk and choice == oracle.PER_TENSOR
    choice, mt, mk = oracle.lqs_select(np.zeros((16, 32), np.float32))
    assert mt == mk == 0.0 and choice == oracle.PER_TENSOR


def test_gw_hq_ablation_transform_orientation_and_lossless_case():
    """The along-tokens HQ of the g_w ablation: with quantization off,
    (1/16) (H g_y)^T (H x) over 16-token blocks equals g_y^T x (Hadamard
    orthogonality along the contraction dim); and with block-constant
    inputs on a 2^-4 grid (coefficient 0 = 16 v, all others 0, amax 7, s = 1)
    the int4 path is lossless."""
    rng = np.random.default_rng(41)
    T, Cin, Cout = 64, 24, 40
    gy = rng.standard_normal((T, Cout))
    x = rng.standard_normal((T, Cin))
    Yg = oracle.hq_transform_f64(gy, axis=1)
    Yx = oracle.hq_transform_f64(x, axis=1)
    assert np.allclose(Yg.T @ Yx / 16.0, gy.T @ x, rtol=1e-12, atol=1e-12)
    kg = np.repeat(rng.integers(-7, 8, (T // 16, Cout)), 16, 0)
    kx = np.repeat(rng.integers(-7, 8, (T // 16, Cin)), 16, 0)
    kg[:16, 0] = 7
    kx[:16, 0] = -7
    g32 = (kg * 2.0 ** -4).astype(np.float32)
    x32 = (kx * 2.0 ** -4).astype(np.float32)
    for rnd in (oracle.RNE, oracle.SR):
        r = oracle.gw_hq_path(g32, x32, rnd=rnd, seed=9)
        assert r["s_g"][0] == 1.0 and r["s_x"][0] == 1.0
        want = g32.astype(np.float64).T @ x32.astype(np.float64)
        assert np.allclose(r["g_w"], want, rtol=1e-12, atol=1e-15)


def test_clamp_when_scale_rounds_down():
    # amax/7 rounded to fp32 can be below the true quotient, so amax/s > 7
    for amax in np.float32([1.0, 3.0, 5.0, 0.1, 1e-3, 123.456]):
        s = amax / np.float32(7)
        Y = np.array([[amax, -amax]], np.float32)
        q, _ = oracle.hq_quantize(Y, oracle.PER_TENSOR, oracle.SR, 1, 0)
        assert list(q[0]) == [7, -7]
    # Past the maximum by one ulp at most, SR reaches 8 only with probability
    # ~2^-21; a subnormal maximum goes much further: RN(10·2^-149 / 7) is
    # s = 2^-149, so the maximum lands at x = 10 and only the clamp brings
    # it back to 7 (127 for the int8 rule: RN(190·2^-149 / 127) = 2^-149).
    tiny = np.float32(2.0 ** -149)
    for rnd in (oracle.RNE, oracle.SR):
        Y = np.array([[10 * tiny, -10 * tiny, 3 * tiny]], np.float32)
        q, s = oracle.hq_quantize(Y, oracle.PER_TENSOR, rnd, 1, 0)
        assert s[0] == tiny and list(q[0]) == [7, -7, 3]
        q, s = oracle.hq_quantize(Y, oracle.PER_TOKEN, rnd, 1, 0)
        assert s[0] == tiny and list(q[0]) == [7, -7, 3]
    v = np.array([190 * tiny, -190 * tiny, 5 * tiny], np.float32)
    q8, s8 = oracle.int8_quantize(v)
    assert s8 == tiny and list(q8) == [127, -127, 5]
    q4, s4 = oracle.rne_quantize(v[:2] / np.float32(19), 7)
    assert s4 == tiny and list(q4) == [7, -7]


def test_scaling_divides_by_the_scale():
    """x = RN(v / s) by IEEE division, not v times a rounded reciprocal:
    with s = 7·2^-10 (1/s is inexact) and v = 6.5·s, v / s is the exact tie
    6.5, whose even neighbour is 6, while v·RN(1/s) rounds to 6.5000005,
    which goes to 7."""
    s = np.float32(7 * 2.0 ** -10)
    for qmax in (7, 127):
        v = np.array([qmax * s, 6.5 * s, -6.5 * s, 2.5 * s], np.float32)
        q, sc = oracle.rne_quantize(v, qmax)
        assert sc == s and list(q) == [qmax, 6, -6, 2]
    Y = np.array([[7 * s, 6.5 * s, -6.5 * s, 2.5 * s]], np.float32)
    for gran in (oracle.PER_TENSOR, oracle.PER_TOKEN):
        q, sc = oracle.hq_quantize(Y, gran, oracle.RNE, 0, 0)
        assert sc[0] == s and list(q[0]) == [7, 6, -6, 2]


def test_sr_error_bound_and_determinism():
    rng = np.random.default_rng(13)
    Y = rng.standard_normal((32, 64)).astype(np.float32)
    q1, s = oracle.hq_quantize(Y, oracle.PER_TOKEN, oracle.SR, 123, 0)
    q2, _ = oracle.hq_quantize(Y, oracle.PER_TOKEN, oracle.SR, 123, 0)
    q3, _ = oracle.hq_quantize(Y, oracle.PER_TOKEN, oracle.SR, 124, 0)
    assert np.array_equal(q1, q2) and not np.array_equal(q1, q3)
    x = Y / s[:, None]
    assert np.all(np.abs(q1 - x) < 1.0 + 1e-6)
    assert np.all((q1 == np.floor(x)) | (q1 == np.floor(x) + 1) | (np.abs(x) > 7))


def test_sr_unbiased_over_seeds():
    rng = np.random.default_rng(14)
    Y = rng.uniform(-7, 7, size=(1, 32)).astype(np.float32)
    Y[0, 0] = 7.0                                     # amax 7 -> s = 1
    n = 2048
    acc = np.zeros(32)
    for seed in range(n):
        q, s = oracle.hq_quantize(Y, oracle.PER_TENSOR, oracle.SR, seed, 0)
        assert s[0] == 1.0
        acc += q[0]
    mean = acc / n
    frac = Y[0] - np.floor(Y[0])
    sigma = np.sqrt(frac * (1 - frac) / n) + 1e-9
    assert np.all(np.abs(mean - Y[0]) <= 4.5 * sigma + 1e-9)


def test_sr_uses_element_index_and_stream():
    """Values at k + 1/2 round up exactly when the element's Philox word has
    its top bit clear: ties the code of element (r, c) to word r*cols + c."""
    rows, cols = 4, 32
    Y = np.full((rows, cols), 0.5, np.float32)
    Y[0, 0] = 7.0
    for stream in (0, 1):
        q, s = oracle.hq_quantize(Y, oracle.PER_TENSOR, oracle.SR, 99, stream)
        for r in range(rows):
            for c in range(cols):
                if (r, c) == (0, 0):
                    continue
                word = oracle.philox_word(99, stream, r * cols + c)
                assert q[r, c] == (1 if (word >> 8) < (1 << 23) else 0)


def test_sampled_rows_use_full_tensor_indices():
    """Rows quantized on their own (the full-size parity tests' form), with
    their row numbers in the full tensor: a value at k + 1/2 rounds up
    exactly when Philox word row*cols + c of the stream has its top bit
    clear, for row numbers far apart (one row repeated); the scale is
    RN(amax/7) of the row, or of the tensor maximum passed in."""
    cols = 32
    ids = np.array([123456, 3, 1000, 3], np.int64)
    Y = np.full((len(ids), cols), 0.5, np.float32)
    Y[1, 7] = -3.5                                  # row amax 3.5 -> s = 0.5
    for stream in (0, 1):
        q, s = oracle.hq_quantize_rows(Y, ids, oracle.PER_TENSOR, oracle.SR, 99,
                                       stream, tensor_amax=7.0)
        assert list(s) == [1.0]
        for i, row in enumerate(ids):
            for c in range(cols):
                if (i, c) == (1, 7):
                    assert q[i, c] in (-3, -4)
                    continue
                word = oracle.philox_word(99, stream, int(row) * cols + c)
                assert q[i, c] == (1 if (word >> 8) < (1 << 23) else 0)
        assert np.array_equal(np.delete(q[1], 7), np.delete(q[3], 7))
    q, s = oracle.hq_quantize_rows(Y, ids, oracle.PER_TOKEN, oracle.RNE, 0, 0)
    assert list(s) == [np.float32(0.5) / np.float32(7), np.float32(3.5) / np.float32(7),
                       np.float32(0.5) / np.float32(7), np.float32(0.5) / np.float32(7)]
    assert np.all(q[[0, 2, 3]] == 7) and q[1, 7] == -7
    assert np.all(np.delete(q[1], 7) == 1)          # 0.5 / 0.5 = 1 exactly


def test_path_row_samples_equal_full_rows():
    """Every path's ``rows`` sample equals those rows of the full result,
    and the sampled quantizer reproduces the full tensor's codes."""
    rng = np.random.default_rng(22)
    T, Cin, Cout = 64, 32, 48
    gy = (rng.standard_normal((T, Cout)) * 1e-3).astype(np.float32)
    w = (rng.standard_normal((Cout, Cin)) * 0.02).astype(np.float32)
    x = rng.standard_normal((T, Cin)).astype(np.float32)
    tok = np.array([63, 0, 17, 17])
    for gran in (oracle.PER_TOKEN, oracle.PER_TENSOR):
        full = oracle.gx_path(gy, w, gran_gy=gran, seed=4)
        part = oracle.gx_path(gy, w, gran_gy=gran, seed=4, rows=tok)
        assert np.array_equal(part["acc"], full["acc"][tok])
        assert np.array_equal(part["g_x"], full["g_x"][tok])
        Y = full["Y"]
        q, s = oracle.hq_quantize_rows(Y[tok], tok, gran, oracle.SR, 4,
                                       oracle.STREAM_GY,
                                       tensor_amax=float(np.max(np.abs(Y))))
        assert np.array_equal(q, full["qY"][tok])
        assert np.array_equal(s, full["s_gy"][tok] if gran == oracle.PER_TOKEN
                              else full["s_gy"])
    full = oracle.gx_hla_path(gy, w, 8)
    part = oracle.gx_hla_path(gy, w, 8, rows=tok)
    assert np.array_equal(part["acc"], full["acc"][tok])
    assert np.array_equal(part["g_x"], full["g_x"][tok])
    out = np.array([47, 1, 30])
    for per_channel in (False, True):
        xq, sx = oracle.compress_activation(x, 8, per_channel=per_channel)
        full = oracle.gw_path(gy, xq, sx, 8)
        part = oracle.gw_path(gy, xq, sx, 8, rows=out)
        assert np.array_equal(part["acc"], full["acc"][out])
        assert np.array_equal(part["g_w"], full["g_w"][out])
    full = oracle.gw_hq_path(gy, x, seed=5)
    part = oracle.gw_hq_path(gy, x, seed=5, rows=out)
    assert np.array_equal(part["acc"], full["acc"][out])
    assert np.array_equal(part["g_w"], full["g_w"][out])


# ------------------------------------------------------------ Philox

def test_philox_uniformity_and_counter_sensitivity():
    words = np.array([oracle.philox_word(5, 0, e) for e in range(40000)],
                     dtype=np.uint64)
    u = (words >> 8).astype(np.float64) / 2 ** 24
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / len(u))
    hist = np.bincount((words >> 28).astype(np.int64), minlength=16)
    expected = len(words) / 16
    chi2 = np.sum((hist - expected) ** 2 / expected)
    assert chi2 < 45.0                         # 15 dof, p ~ 1e-4
    assert oracle.philox_word(5, 0, 0) != oracle.philox_word(5, 1, 0)
    assert oracle.philox_word(5, 0, 0) != oracle.philox_word(6, 0, 0)
    assert oracle.philox_word(5, 0, 1 << 34) != oracle.philox_word(5, 0, 0)
    # word e%4 of one block
    blk = oracle.philox4x32_10([3, 0, 0, 0], [5, 0])
    assert [oracle.philox_word(5, 0, 12 + i) for i in range(4)] == list(blk)


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161         # curandRngType_t, curand.h


def _curand_host_philox():
    """cuRAND's host-side Philox4x32-10 generator (it runs on the CPU), or
    None where libcurand is not installed."""
    import ctypes
    import ctypes.util
    import glob
    import os
    names = []
    for root in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"),
                 "/usr/local/cuda"):
        if root:
            names += sorted(glob.glob(os.path.join(root, "lib64", "libcurand.so*")))
            names += sorted(glob.glob(os.path.join(root, "targets", "*", "lib",
                                                   "libcurand.so*")))
    found = ctypes.util.find_library("curand")
    if found:
        names.append(found)
    for name in names:
        try:
            lib = ctypes.CDLL(name)
        except OSError:
            continue
        gen = ctypes.c_void_p()
        if lib.curandCreateGeneratorHost(ctypes.byref(gen),
                                         CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0:
            return lib, gen
    return None


def test_philox_matches_curand_host_generator():
    """Oracle Philox words equal cuRAND's Philox4x32-10 stream.

    cuRAND's default ordering emits block k (four words) of Philox4x32-10
    under key (seed lo, seed hi) at counter (k >> 16 as a 64-bit number in
    words 0-1, k mod 65536 in word 2, 0): that is the oracle's word
    e = 4·(k >> 16) + j of stream k mod 65536.  The cases cover both key
    halves, the stream word, counter word 0, and the carry from counter word
    0 into word 1 (k = 2^48 - 1 -> 2^48).  A wrong multiplier, Weyl constant,
    round count or output permutation in the oracle fails every word."""
    import ctypes
    found = _curand_host_philox()
    if found is None:
        pytest.skip("libcurand not installed")
    lib, gen = found

    def curand_words(seed, offset, n):
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        buf = np.zeros(n, np.uint32)
        assert lib.curandGenerate(gen, buf.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(n)) == 0
        return buf

    def oracle_words(seed, offset, n):
        out = np.zeros(n, np.uint32)
        for i in range(n):
            k, j = divmod(offset + i, 4)
            out[i] = oracle.philox_word(seed, k & 0xFFFF, 4 * (k >> 16) + j)
        return out

    try:
        for seed in (0, 0x299F31D0A4093822, 0xFFFFFFFFFFFFFFFF):
            for offset, n in ((0, 4 * 1024),                 # streams 0..1023, e < 4
                              (4 * 65536 - 16, 64),          # e 0..3 -> 4..7
                              (4 * 65536 * 37 + 4 * 9000, 32),
                              (4 * ((1 << 48) - 2), 16)):    # counter word 0 -> word 1
                got = oracle_words(seed, offset, n)
                want = curand_words(seed, offset, n)
                assert np.array_equal(got, want), (hex(seed), offset)
    finally:
        lib.curandDestroyGenerator(gen)


# ------------------------------------------------------------ GEMM, packing

def test_gemm_brute_force():
    rng = np.random.default_rng(15)
    A = rng.integers(-127, 128, (5, 37)).astype(np.int8)
    B = rng.integers(-127, 128, (7, 37)).astype(np.int8)
    C = oracle.gemm_i64(A, B)
    for m in range(5):
        for n in range(7):
            assert C[m, n] == sum(int(A[m, k]) * int(B[n, k]) for k in range(37))


def test_gemm_exhaustive_int4_range():
    vals = np.arange(-7, 8, dtype=np.int8)
    A = np.array([[a] * 16 for a in vals], dtype=np.int8)          # [15, 16]
    B = np.array([[b] * 16 for b in vals], dtype=np.int8)
    C = oracle.gemm_i64(A, B)
    assert np.array_equal(C, 16 * np.outer(vals.astype(np.int64),
                                           vals.astype(np.int64)))


def test_pack_int4_layout():
    codes = np.array([[1, -1, 7, -7, 0, 3]], np.int8)
    p = oracle.pack_int4(codes)
    assert list(p[0]) == [0xF1, 0x97, 0x30]


def test_dequant_matches_fp64():
    rng = np.random.default_rng(16)
    acc = rng.integers(-10 ** 6, 10 ** 6, (6, 5))
    s_gy = rng.uniform(0.1, 2, 6).astype(np.float32)
    got = oracle.dequant_gx(acc, s_gy, oracle.PER_TOKEN, np.float32(0.25))
    want = acc * s_gy.astype(np.float64)[:, None] * 0.25 / 16
    assert np.allclose(got, want, rtol=1e-15, atol=0)
    got = oracle.dequant_gw(acc, np.float32(0.5), np.float32(3.0))
    assert np.allclose(got, acc * 1.5 / 16, rtol=1e-15, atol=0)


# --------------------------------------------------- whole paths, lossless

def _lossless_hq_operand(rng, rows, n16, s0):
    """Data whose Hadamard transform is exactly integer codes times s0."""
    codes = rng.integers(-7, 8, (rows, 16 * n16))
    codes[:, 0] = 7                                   # amax = 7*s0 per row
    D = np.kron(np.eye(n16, dtype=np.int64), H_SCIPY)
    v = codes @ D / 16.0 * s0                         # D^{-1} = D/16 (symmetric)
    return v.astype(np.float32), codes


def test_gx_path_lossless_equals_gy_w():
    rng = np.random.default_rng(17)
    T, Cin, Cout = 32, 48, 64
    gy, _ = _lossless_hq_operand(rng, T, Cout // 16, 2.0 ** -6)
    wT, _ = _lossless_hq_operand(rng, Cin, Cout // 16, 2.0 ** -3)
    w = np.ascontiguousarray(wT.T)                    # [Cout, Cin]
    for gran in (oracle.PER_TOKEN, oracle.PER_TENSOR):
        for rnd in (oracle.RNE, oracle.SR):
            r = oracle.gx_path(gy, w, gran_gy=gran, rnd=rnd, seed=3)
            want = gy.astype(np.float64) @ w.astype(np.float64)
            assert np.allclose(r["g_x"], want, rtol=1e-12, atol=1e-15)


def _with_coefficients(C, axis):
    """Data whose exact 16-block Hadamard transform is C: along columns
    (axis 0, as for g_y in the g_x path) or along rows (axis 1, as for w and
    for the along-token transforms).  D is symmetric and D^-1 = D/16."""
    if axis == 0:
        D = np.kron(np.eye(C.shape[1] // 16, dtype=np.int64), H_SCIPY)
        return (C @ D / 16.0).astype(np.float32)
    D = np.kron(np.eye(C.shape[0] // 16, dtype=np.int64), H_SCIPY)
    return (D @ C / 16.0).astype(np.float32)


def _sr_half(seed, stream, e):
    """SR code of a value at exactly 1/2 with scale 1: 1 when the Philox
    word's top 24 bits give u < 1/2."""
    return 1 if (oracle.philox_word(seed, stream, e) >> 8) < (1 << 23) else 0


def test_path_streams_scales_and_element_indices():
    """Which Philox stream, element index and scale each quantized operand
    of the HQ paths takes: g_y stream 0 at t·Cout + c, one scale per token
    or per tensor; w stream 1 at o·Cin + i of the transformed [Cout, Cin]
    tensor, one scale per tensor; the g_w ablation's g_y and x streams 2 and
    3 at t·C + c of their along-token transforms, one scale each.  Each
    operand is built so that its exact transform is 1/2 everywhere but for a
    7, so every other code shows the word it drew."""
    seed = 31
    T, Cin, Cout = 32, 16, 32
    Cg = np.full((T, Cout), 0.5)
    Cg[:, 0] = 7.0
    Cg[1, 0] = 0.5                                   # token 1 has no 7
    Cw = np.full((Cout, Cin), 0.5)
    Cw[0, 0] = 7.0
    gy = _with_coefficients(Cg, 0)
    w = _with_coefficients(Cw, 1)
    for gran in (oracle.PER_TOKEN, oracle.PER_TENSOR):
        r = oracle.gx_path(gy, w, gran_gy=gran, rnd=oracle.SR, seed=seed)
        assert np.array_equal(r["Y"], Cg.astype(np.float32))
        assert list(r["s_w"]) == [1.0]
        for o in range(Cout):
            for i in range(Cin):
                want = 7 if (o, i) == (0, 0) else _sr_half(seed, 1, o * Cin + i)
                assert r["qW"][i, o] == want, (o, i)
        if gran == oracle.PER_TOKEN:
            assert r["s_gy"][1] == np.float32(0.5) / np.float32(7)
            assert np.all(r["qY"][1] == 7)           # its own scale: 1/2 -> 7
            assert np.all(np.delete(r["s_gy"], 1) == 1.0)
        else:
            assert list(r["s_gy"]) == [1.0]
        for t in range(T):
            if gran == oracle.PER_TOKEN and t == 1:
                continue
            for c in range(Cout):
                want = 7 if Cg[t, c] == 7 else _sr_half(seed, 0, t * Cout + c)
                assert r["qY"][t, c] == want, (t, c)
    Cg2 = np.full((T, Cout), 0.5)
    Cg2[0, 0] = 7.0
    Cx2 = np.full((T, Cin), 0.5)
    Cx2[3, 5] = -7.0
    r = oracle.gw_hq_path(_with_coefficients(Cg2, 1), _with_coefficients(Cx2, 1),
                          rnd=oracle.SR, seed=seed)
    assert list(r["s_g"]) == [1.0] and list(r["s_x"]) == [1.0]
    for t in range(T):
        for c in range(Cout):
            want = 7 if (t, c) == (0, 0) else _sr_half(seed, 2, t * Cout + c)
            assert r["qG"][c, t] == want, (t, c)
        for c in range(Cin):
            want = -7 if (t, c) == (3, 5) else _sr_half(seed, 3, t * Cin + c)
            assert r["qX"][c, t] == want, (t, c)


def test_gw_path_lossless_equals_gyT_x():
    rng = np.random.default_rng(18)
    T, Cin, Cout = 64, 20, 24
    # token pairs equal -> only the kept (even) Hadamard rows are non-zero;
    # values on a power-of-two grid with |Xbar| hitting 127*s exactly.
    gy = np.repeat(rng.integers(-3, 4, (T // 2, Cout)), 2, 0).astype(np.float64)
    x = np.repeat(rng.integers(-3, 4, (T // 2, Cin)), 2, 0).astype(np.float64)
    gy[:16, 0] = 127 / 16.0 * 2
    x[:16, 0] = 127 / 16.0 * 2
    gy = (gy * 2.0 ** -7).astype(np.float32)
    x = (x * 2.0 ** -2).astype(np.float32)
    q, s = oracle.compress_activation(x, 8)
    r = oracle.gw_path(gy, q, s, 8)
    # lossless only if every coefficient is an integer multiple of its scale
    assert np.array_equal(r["qG"].astype(np.float64) * r["s_g"], r["Gb"])
    want = gy.astype(np.float64).T @ x.astype(np.float64)
    assert np.allclose(r["g_w"], want, rtol=1e-12, atol=1e-15)


def _in_kept_span(K, rank, s):
    """[T, C] data whose rank-`rank` HLA coefficients are exactly K·s
    (K [C, T·rank/16] integer codes): per 16-token block, the combination
    (1/16)·Σ_k K[:, rank·b + k]·H[σ(k)] of the kept Walsh rows, which are
    orthogonal with squared norm 16."""
    C, Tp = K.shape
    T = Tp // rank * 16
    rows = np.array([H_SCIPY[gray_bitrev_sequency(k)] for k in range(rank)])
    out = np.zeros((T, C))
    for b in range(T // 16):
        out[16 * b:16 * b + 16] = rows.T @ K[:, rank * b:rank * b + rank].T / 16.0
    return (out * s).astype(np.float32)


@pytest.mark.parametrize("rank", [1, 2, 4, 8, 16])
def test_gw_path_lossless_every_rank(rank):
    """Data in the span of the kept Walsh rows loses nothing at rank r:
    with codes whose maximum is 127 and power-of-two scales, the int8 codes
    are the constructed ones and g_w equals g_yᵀx exactly (Parseval over the
    kept rows: Σ_t g_t x_t = (1/16) Σ_k G_k X_k per block)."""
    rng = np.random.default_rng(60 + rank)
    T, Cin, Cout = 64, 12, 20
    Tp = T * rank // 16
    Kg = rng.integers(-127, 128, (Cout, Tp))
    Kx = rng.integers(-127, 128, (Cin, Tp))
    Kg[0, 0], Kx[1, -1] = 127, -127
    gy = _in_kept_span(Kg, rank, 2.0 ** -7)
    x = _in_kept_span(Kx, rank, 2.0 ** -3)
    q, s = oracle.compress_activation(x, rank)
    assert s == np.float32(2.0 ** -3) and np.array_equal(q, Kx)
    r = oracle.gw_path(gy, q, s, rank)
    assert r["s_g"] == np.float32(2.0 ** -7) and np.array_equal(r["qG"], Kg)
    want = gy.astype(np.float64).T @ x.astype(np.float64)
    assert np.allclose(r["g_w"], want, rtol=1e-12, atol=1e-15)


# ----------------------------------------- per-channel scales of the ACBP

def _per_channel_lossless_x(rng, T, Cin, exps):
    """x whose HLA (rank 8) coefficients in channel c are integer multiples
    of 2^(e_c - 1) with maximum exactly 127 * 2^(e_c - 1): token pairs equal
    (only the kept even Sylvester rows are non-zero) and a spike block."""
    x = np.repeat(rng.integers(-3, 4, (T // 2, Cin)), 2, 0).astype(np.float64)
    x[:16, :] = 127 / 16.0 * 2
    return (x * 2.0 ** (np.asarray(exps, dtype=np.float64)[None, :] - 2)).astype(np.float32)


def test_per_channel_acbp_lossless_gw_with_outlier_channels():
    """Channels of very different magnitude (outlier channels 2^6 larger):
    one scale per channel keeps every channel on its own code grid, so the
    stored activation is lossless and g_w equals g_y^T x; one scale for the
    whole tensor is not (the small channels lose their low bits).  Cin !=
    Cout, so a scale applied along the wrong axis of g_w fails."""
    rng = np.random.default_rng(23)
    T, Cin, Cout = 64, 20, 24
    exps = np.zeros(Cin, dtype=np.int64)
    exps[[3, 11]] = 6
    exps[[5, 17]] = -3
    x = _per_channel_lossless_x(rng, T, Cin, exps)
    gy = np.repeat(rng.integers(-3, 4, (T // 2, Cout)), 2, 0).astype(np.float64)
    gy[:16, 0] = 127 / 16.0 * 2
    gy = (gy * 2.0 ** -7).astype(np.float32)
    q, s = oracle.compress_activation(x, 8, per_channel=True)
    assert s.shape == (Cin,)
    assert np.array_equal(s.astype(np.float64), 2.0 ** (exps - 1.0))
    Xb = oracle.hla_transform(x, 8)
    assert np.array_equal(q.astype(np.float64) * s.astype(np.float64)[:, None], Xb)
    want = gy.astype(np.float64).T @ x.astype(np.float64)
    r = oracle.gw_path(gy, q, s, 8)
    assert np.allclose(r["g_w"], want, rtol=1e-12, atol=1e-15)
    qt, st = oracle.compress_activation(x, 8)
    rt = oracle.gw_path(gy, qt, st, 8)
    small = exps < 0
    assert not np.allclose(rt["g_w"][:, small], want[:, small], rtol=1e-6, atol=0)


@pytest.mark.parametrize("bits", [8, 4])
def test_per_channel_equal_maxima_reduce_to_per_tensor(bits):
    """When every channel's largest coefficient is the same number, the
    per-channel scales all equal the per-tensor scale and the codes and g_w
    are those of the per-tensor quantizer, bit for bit."""
    rng = np.random.default_rng(24)
    T, Cin, Cout = 64, 32, 16
    x = rng.standard_normal((T, Cin)).astype(np.float32)
    x[:16, :] = 40.0          # block 0: DC coefficient 640 in every channel
    gy = rng.standard_normal((T, Cout)).astype(np.float32)
    qc, sc = oracle.compress_activation(x, 8, bits=bits, per_channel=True)
    qt, st = oracle.compress_activation(x, 8, bits=bits)
    assert np.all(sc == st)
    assert np.array_equal(qc, qt)
    rc = oracle.gw_path(gy, qc, sc, 8)
    rt = oracle.gw_path(gy, qt, st, 8)
    assert np.array_equal(rc["acc"], rt["acc"])
    assert np.array_equal(rc["g_w"], rt["g_w"])


@pytest.mark.parametrize("bits", [8, 4])
def test_per_channel_rne_bound_per_row(bits):
    """Outlier channels (1 % of channels x50): each channel's scale is
    RN(amax_c / qmax) of its own coefficients, its largest code is +-qmax,
    and every code is within half a step of its coefficient (own scale),
    which is never coarser than the per-tensor step."""
    rng = np.random.default_rng(25)
    T, Cin = 128, 200
    x = rng.standard_normal((T, Cin))
    x[:, rng.choice(Cin, 2, replace=False)] *= 50.0
    x = x.astype(np.float32)
    qmax = 127 if bits == 8 else 7
    q, s = oracle.compress_activation(x, 8, bits=bits, per_channel=True)
    _, st = oracle.compress_activation(x, 8, bits=bits)
    Xb = oracle.hla_transform(x, 8).astype(np.float64)
    amax_c = np.max(np.abs(Xb), axis=1)
    assert np.array_equal(s, (amax_c / qmax).astype(np.float32))
    assert np.all(np.max(np.abs(q.astype(np.int64)), axis=1) == qmax)
    err = np.abs(q.astype(np.float64) * s.astype(np.float64)[:, None] - Xb)
    ulp = np.spacing(amax_c.astype(np.float32)).astype(np.float64)
    assert np.all(err <= s.astype(np.float64)[:, None] / 2 + ulp[:, None])
    assert np.all(s <= st)


# ------------------------------------- ablation: HLA on the g_x contraction

@pytest.mark.parametrize("rank", [1, 2, 4, 8])
def test_gx_hla_ablation_lossless_equals_gy_w(rank):
    """g_y constant on groups of 16/rank consecutive output channels lies in
    the span of the rank lowest-sequency Walsh rows, so the low-rank product
    over Cout is exact; with every kept coefficient on its int8 grid (spike
    blocks set both maxima to 127 * s) g_x equals g_y . w.  Keeping other
    Walsh rows (e.g. the first rank rows in Sylvester order) breaks it, and
    T, Cin, Cout all differ, so a transposed operand fails too."""
    rng = np.random.default_rng(26)
    T, Cin, Cout = 48, 40, 64
    L = 16 // rank
    gy = np.repeat(rng.integers(-3, 4, (T, Cout // L)), L, 1).astype(np.float64)
    gy[0, :16] = 127 / 16.0 * 2              # DC coefficient 127 * 2 of block 0
    w = rng.integers(-3, 4, (Cout, Cin)).astype(np.float64)
    w[:16, 0] = 127 / 16.0                   # DC coefficient 127
    gy = (gy * 2.0 ** -7).astype(np.float32)
    w = (w * 2.0 ** -2).astype(np.float32)
    r = oracle.gx_hla_path(gy, w, rank)
    assert r["qG"].shape == (T, Cout // 16 * rank) and r["qW"].shape == (Cin, Cout // 16 * rank)
    assert np.array_equal(r["qG"].astype(np.float64) * r["s_g"], r["Gb"])
    assert np.array_equal(r["qW"].astype(np.float64) * r["s_w"], r["Wb"])
    want = gy.astype(np.float64) @ w.astype(np.float64)
    assert np.allclose(r["g_x"], want, rtol=1e-12, atol=1e-15)
    if rank < 16:   # the same data but generic within the groups is not exact
        gy2 = gy.copy()
        gy2[:, 1::2] += np.float32(2.0 ** -7)
        r2 = oracle.gx_hla_path(gy2, w, rank)
        want2 = gy2.astype(np.float64) @ w.astype(np.float64)
        assert not np.allclose(r2["g_x"], want2, rtol=1e-9, atol=0)


def test_gx_hla_ablation_full_rank_quant_off_is_gy_w():
    """Rank 16 keeps every Walsh row: the exactly rounded transforms of both
    operands, multiplied in fp64 and divided by 16, give g_y . w to fp32
    rounding of the coefficients (H16 H16^T = 16 I)."""
    rng = np.random.default_rng(27)
    T, Cin, Cout = 32, 24, 48
    gy = rng.standard_normal((T, Cout)).astype(np.float32)
    w = rng.standard_normal((Cout, Cin)).astype(np.float32)
    r = oracle.gx_hla_path(gy, w, 16)
    got = r["Gb"].astype(np.float64) @ r["Wb"].astype(np.float64).T / 16.0
    want = gy.astype(np.float64) @ w.astype(np.float64)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-5)
    # and the permutation of the kept rows is the same on both operands:
    # Sylvester order of g_y's rows against sequency order of w's would not
    # reproduce the product
    H = H_SCIPY.astype(np.float64)
    Gs = (gy.astype(np.float64).reshape(T, Cout // 16, 16) @ H.T).reshape(T, Cout)
    bad = Gs @ r["Wb"].astype(np.float64).T / 16.0
    assert not np.allclose(bad, want, rtol=1e-3, atol=1e-3)
