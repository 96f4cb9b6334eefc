"""Pins for the CPU oracle (no GPU needed).

The oracle is only trusted because these checks tie it to things other than
itself: the binary16 format definition and numpy's independent codec, closed
forms of the operator (identity B, all-ones, one-hot rows, negative alpha), a
hand-worked example, and exact rational brute force on tiny inputs.  Each
check is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, a transposed operand, scale and ReLU swapped, a wrong rounding rule, a
row-sampling index error) fails at least one of them.

Operator: "Tutorial14: 使用TileLang语言编写attention算子", section 3 (formula)
and section 2 (scale first, then max with 0; fp16 in and out).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# binary16 codec
# ----------------------------------------------------------------------------

def test_decode_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_decode(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan_ours = np.isnan(ours)
    assert np.array_equal(nan_ours, np.isnan(ref))
    assert np.array_equal(ours[~nan_ours].view(np.uint64), ref[~nan_ours].view(np.uint64))


def test_decode_from_definition():
    # a few patterns worked from the field definition
    assert oracle.f16_decode([0x3C00])[0] == 1.0
    assert oracle.f16_decode([0x0001])[0] == 2.0 ** -24
    assert oracle.f16_decode([0x03FF])[0] == 1023 * 2.0 ** -24
    assert oracle.f16_decode([0x0400])[0] == 2.0 ** -14
    assert oracle.f16_decode([0x7BFF])[0] == 65504.0
    assert oracle.f16_decode([0xC000])[0] == -2.0
    assert np.isinf(oracle.f16_decode([0x7C00])[0])
    assert np.isnan(oracle.f16_decode([0x7E00])[0])


def _golden_codec():
    rows = []
    with open(os.path.join(GOLDEN, "binary16_codec.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((float(parts[0]), int(parts[1], 16)))
    return rows


@pytest.mark.parametrize("value,bits", _golden_codec())
def test_encode_golden_table(value, bits):
    assert int(oracle.f16_encode([value])[0]) == bits


def test_encode_random_matches_numpy():
    rng = np.random.default_rng(7)
    n = 1_000_000
    mag = np.exp2(rng.uniform(-26.0, 16.5, n))
    x = mag * rng.choice([-1.0, 1.0], n)
    ours = oracle.f16_encode(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_every_tie_goes_to_even():
    # the midpoint of every pair of adjacent finite positive halves is exact in
    # binary64; round-to-nearest-even must pick the pattern with an even LSB
    lo_bits = np.arange(0, 0x7BFF, dtype=np.uint32).astype(np.uint16)
    lo = lo_bits.view(np.float16).astype(np.float64)
    hi = (lo_bits + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2.0
    want = np.where(lo_bits % 2 == 0, lo_bits, lo_bits + 1).astype(np.uint16)
    assert np.array_equal(oracle.f16_encode(mid), want)
    assert np.array_equal(oracle.f16_encode(-mid), want | 0x8000)
    # nudged off the tie, the nearer neighbour wins
    assert np.array_equal(oracle.f16_encode(np.nextafter(mid, 0)), lo_bits)
    assert np.array_equal(oracle.f16_encode(np.nextafter(mid, np.inf)), lo_bits + 1)


def test_encode_round_trip_all_finite():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    assert np.array_equal(oracle.f16_encode(vals[finite]), bits[finite])


# ----------------------------------------------------------------------------
# exact reference for tiny cases: rationals, written independently of the C code
# ----------------------------------------------------------------------------

def _f16_bits_from_fraction(q: Fraction) -> int:
    """Round an exact rational to binary16 (ties to even), using exact arithmetic."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (-24 if e < -14 else e - 10)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if e < -14:
        return sign | fl
    if fl == 2048:
        fl = 1024
        e += 1
    if e > 15:
        return sign | 0x7C00
    return sign | ((e + 15) << 10) | (fl - 1024)


def test_fraction_encoder_agrees_with_numpy():
    # pins the test's own exact encoder before it is used as a reference
    rng = np.random.default_rng(3)
    x = np.exp2(rng.uniform(-25.0, 15.9, 5000)) * rng.choice([-1.0, 1.0], 5000)
    ref = x.astype(np.float16).view(np.uint16)
    got = np.array([_f16_bits_from_fraction(Fraction(float(v))) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _exact_reference(A16, B16, alpha):
    """C and pre-ReLU value by exact rational arithmetic, in plain Python loops."""
    M, K = A16.shape
    N = B16.shape[1]
    al = Fraction(float(np.float32(alpha)))
    C = np.zeros((M, N), dtype=np.uint16)
    Z = np.zeros((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(A16[i, k])) * Fraction(float(B16[k, j]))
            z = al * s
            Z[i, j] = z
            C[i, j] = _f16_bits_from_fraction(z if z > 0 else Fraction(0))
    return C, Z


def _rand16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


BRUTE_SHAPES = [(1, 1, 1), (1, 1, 5), (3, 5, 2), (2, 3, 7), (7, 3, 11), (5, 17, 1),
                (17, 13, 16), (4, 9, 17)]


@pytest.mark.parametrize("M,N,K", BRUTE_SHAPES)
@pytest.mark.parametrize("alpha", [0.5, 1.0, -0.75, 0.3])
def test_brute_force_exact(M, N, K, alpha):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A = _rand16(rng, (M, K))
    B = _rand16(rng, (K, N))
    C, Z = oracle.gemm_scale_relu(A, B, alpha, return_pre=True)
    Cx, Zx = _exact_reference(A, B, alpha)
    assert np.array_equal(C.view(np.uint16), Cx)
    for i in range(M):
        for j in range(N):
            assert Z[i, j] == pytest.approx(float(Zx[i, j]), rel=1e-14, abs=1e-300)


@pytest.mark.parametrize("M,N,K", [(3, 4, 5), (6, 2, 9)])
def test_brute_force_fsum(M, N, K):
    # a second independent route: math.fsum of the exact products, then numpy's codec
    rng = np.random.default_rng(11 + M + N + K)
    A = _rand16(rng, (M, K))
    B = _rand16(rng, (K, N))
    alpha = 0.5
    C = oracle.gemm_scale_relu(A, B, alpha)
    for i in range(M):
        for j in range(N):
            s = math.fsum(float(A[i, k]) * float(B[k, j]) for k in range(K))
            y = max(alpha * s, 0.0)
            assert C[i, j].view(np.uint16) == np.float16(y).view(np.uint16)


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(64, 64), (130, 72), (5, 3)])
@pytest.mark.parametrize("alpha", [0.5, 1.0, 0.3, -0.7])
def test_identity_b(M, K, alpha):
    rng = np.random.default_rng(M + K)
    A = _rand16(rng, (M, K))
    B = np.eye(K, dtype=np.float16)
    C = oracle.gemm_scale_relu(A, B, alpha)
    want = np.maximum(float(np.float32(alpha)) * A.astype(np.float64), 0.0).astype(np.float16)
    assert np.array_equal(C.view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("K,alpha,expect", [
    (1000, 0.5, 500.0), (3000, 1.0, 3000.0), (2049, 1.0, 2048.0), (2051, 1.0, 2052.0),
    (4098, 1.0, 4096.0), (4102, 1.0, 4104.0), (1, 1.0, 1.0), (7, 0.5, 3.5)])
def test_all_ones(K, alpha, expect):
    M, N = 3, 5
    A = np.ones((M, K), dtype=np.float16)
    B = np.ones((K, N), dtype=np.float16)
    C, Z = oracle.gemm_scale_relu(A, B, alpha, return_pre=True)
    assert np.all(C == np.float16(expect))
    assert np.all(Z == alpha * K)


def test_one_hot_rows_select_rows_of_b():
    # row i of A is the unit vector e_{k_i}: row i of C must be ReLU(alpha * B[k_i, :]);
    # a transposed A or B, or a k/n index mix-up, breaks this on a non-square shape
    rng = np.random.default_rng(5)
    M, N, K = 6, 11, 9
    ks = [0, 8, 3, 3, 5, 1]
    A = np.zeros((M, K), dtype=np.float16)
    for i, k in enumerate(ks):
        A[i, k] = 1
    B = _rand16(rng, (K, N))
    alpha = 0.5
    C = oracle.gemm_scale_relu(A, B, alpha)
    for i, k in enumerate(ks):
        want = np.maximum(alpha * B[k].astype(np.float64), 0.0).astype(np.float16)
        assert np.array_equal(C[i].view(np.uint16), want.view(np.uint16))


def test_one_hot_columns_select_columns_of_a():
    rng = np.random.default_rng(6)
    M, N, K = 7, 4, 10
    ks = [9, 0, 4, 4]
    A = _rand16(rng, (M, K))
    B = np.zeros((K, N), dtype=np.float16)
    for j, k in enumerate(ks):
        B[k, j] = 1
    C = oracle.gemm_scale_relu(A, B, 1.0)
    for j, k in enumerate(ks):
        want = np.maximum(A[:, k].astype(np.float64), 0.0).astype(np.float16)
        assert np.array_equal(C[:, j].view(np.uint16), want.view(np.uint16))


def test_negative_alpha_on_nonnegative_inputs_gives_zeros():
    rng = np.random.default_rng(8)
    A = np.abs(_rand16(rng, (33, 40)))
    B = np.abs(_rand16(rng, (40, 21)))
    C, Z = oracle.gemm_scale_relu(A, B, -0.5, return_pre=True)
    assert np.all(C.view(np.uint16) == 0)      # +0 exactly, no -0
    assert np.all(Z <= 0)


def test_negative_alpha_flips_sign_before_relu():
    # A >= 0 and B <= 0: the sum is <= 0, so ReLU(alpha * sum) with alpha < 0 is
    # |alpha| * |sum|, which a ReLU-before-scale oracle would zero out
    rng = np.random.default_rng(9)
    A = np.abs(_rand16(rng, (4, 6)))
    B = -np.abs(_rand16(rng, (6, 5)))
    C = oracle.gemm_scale_relu(A, B, -0.5)
    Cpos = oracle.gemm_scale_relu(A, -B, 0.5)
    assert np.array_equal(C.view(np.uint16), Cpos.view(np.uint16))
    assert np.all(C > 0)


def test_hand_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    A = np.array(g["A"], dtype=np.float16)
    B = np.array(g["B"], dtype=np.float16)
    for case in g["cases"]:
        C, Z = oracle.gemm_scale_relu(A, B, case["alpha"], return_pre=True)
        assert np.array_equal(C.astype(np.float64), np.array(case["C"]))
        assert np.array_equal(Z, np.array(case["pre"]))


# ----------------------------------------------------------------------------
# sizes, sampling, degenerate cases
# ----------------------------------------------------------------------------

def test_row_sampling_matches_full_rows():
    rng = np.random.default_rng(10)
    A = _rand16(rng, (70, 37))
    B = _rand16(rng, (37, 29))
    full, zf = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
    rows = [69, 0, 13, 13, 42]
    part, zp = oracle.gemm_scale_relu(A, B, 0.5, rows=rows, return_pre=True)
    assert np.array_equal(part.view(np.uint16), full[rows].view(np.uint16))
    assert np.array_equal(zp, zf[rows])


def test_row_out_of_range_rejected():
    A = np.ones((4, 3), np.float16)
    B = np.ones((3, 2), np.float16)
    with pytest.raises(ValueError):
        oracle.gemm_scale_relu(A, B, 1.0, rows=[4])


def test_k_zero_gives_zeros():
    A = np.zeros((5, 0), np.float16)
    B = np.zeros((0, 7), np.float16)
    C = oracle.gemm_scale_relu(A, B, 0.5)
    assert C.shape == (5, 7) and np.all(C.view(np.uint16) == 0)


def test_empty_outputs():
    assert oracle.gemm_scale_relu(np.zeros((0, 4), np.float16), np.zeros((4, 3), np.float16), 1.0).shape == (0, 3)
    assert oracle.gemm_scale_relu(np.zeros((2, 4), np.float16), np.zeros((4, 0), np.float16), 1.0).shape == (2, 0)


def test_c_equals_encoded_relu_of_pre():
    rng = np.random.default_rng(12)
    A = _rand16(rng, (40, 64))
    B = _rand16(rng, (64, 48))
    C, Z = oracle.gemm_scale_relu(A, B, 0.37, return_pre=True)
    want = np.maximum(Z, 0.0).astype(np.float16)
    assert np.array_equal(C.view(np.uint16), want.view(np.uint16))
    assert np.any(Z < 0) and np.any(Z > 0)


def test_overflow_to_inf_and_subnormal_output():
    # sums past the binary16 range saturate to +inf; tiny results stay subnormal
    A = np.full((1, 4), 255.0, np.float16)
    B = np.full((4, 2), 255.0, np.float16)
    C = oracle.gemm_scale_relu(A, B, 1.0)          # 4 * 65025 = 260100 > 65504
    assert np.all(np.isinf(C)) and np.all(C > 0)
    A = np.full((1, 1), 2.0 ** -12, np.float16)
    B = np.full((1, 1), 2.0 ** -12, np.float16)
    C = oracle.gemm_scale_relu(A, B, 1.0)          # 2^-24: the smallest subnormal
    assert C.view(np.uint16)[0, 0] == 0x0001


def test_threads_do_not_change_results():
    rng = np.random.default_rng(13)
    A = _rand16(rng, (64, 96))
    B = _rand16(rng, (96, 80))
    n0 = oracle.max_threads()
    try:
        oracle.set_num_threads(1)
        c1 = oracle.gemm_scale_relu(A, B, 0.5)
        oracle.set_num_threads(max(2, n0))
        c2 = oracle.gemm_scale_relu(A, B, 0.5)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(c1.view(np.uint16), c2.view(np.uint16))


# ----------------------------------------------------------------------------
# further epilogues: alpha * sum (plain GEMM) and GELU(sum + bias)
# (aikraft.ru TileLang tutorial survey: make_matmul and make_matmul_bias_gelu sections)
# ----------------------------------------------------------------------------

def test_epilogue_kind0_is_the_fused_operator():
    rng = np.random.default_rng(20)
    A = _rand16(rng, (23, 41))
    B = _rand16(rng, (41, 19))
    for alpha in (0.5, -1.25):
        c0 = oracle.gemm_epilogue(A, B, alpha, oracle.EPI_SCALE_RELU)
        c1 = oracle.gemm_scale_relu(A, B, alpha)
        assert np.array_equal(c0.view(np.uint16), c1.view(np.uint16))


@pytest.mark.parametrize("alpha", [1.0, 0.5, -0.75])
def test_scale_identity_b_keeps_negatives(alpha):
    rng = np.random.default_rng(21)
    A = _rand16(rng, (37, 24))
    C = oracle.gemm_epilogue(A, np.eye(24, dtype=np.float16), alpha, oracle.EPI_SCALE)
    want = (float(np.float32(alpha)) * A.astype(np.float64)).astype(np.float16)
    assert np.array_equal(C.view(np.uint16), want.view(np.uint16))
    assert np.any(C < 0)


@pytest.mark.parametrize("M,N,K", [(3, 5, 2), (7, 3, 11), (4, 9, 17)])
def test_scale_brute_force_exact(M, N, K):
    rng = np.random.default_rng(M * 31 + N + K)
    A = _rand16(rng, (M, K))
    B = _rand16(rng, (K, N))
    alpha = -0.3
    C = oracle.gemm_epilogue(A, B, alpha, oracle.EPI_SCALE)
    al = Fraction(float(np.float32(alpha)))
    for i in range(M):
        for j in range(N):
            s = sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)),
                    Fraction(0))
            assert C.view(np.uint16)[i, j] == _f16_bits_from_fraction(al * s)


def _torch_gelu_tanh(x):
    import torch
    return torch.nn.functional.gelu(torch.from_numpy(np.asarray(x, np.float64)),
                                    approximate="tanh").numpy()


def test_gelu_identity_b_matches_torch_gelu():
    # identity B makes the sum exactly A, so Y = GELU(A + bias) in fp64; torch's own
    # tanh-form GELU is an independent implementation of the same function
    rng = np.random.default_rng(22)
    K = 48
    A = (rng.standard_normal((40, K)) * 3).astype(np.float16)
    bias = (rng.standard_normal(K) * 2).astype(np.float16)
    C, Y = oracle.gemm_epilogue(A, np.eye(K, dtype=np.float16), kind=oracle.EPI_BIAS_GELU,
                                bias=bias, return_pre=True)
    x = A.astype(np.float64) + bias.astype(np.float64)[None, :]
    ref = _torch_gelu_tanh(x)
    # absolute floor 1e-14: torch's 0.5x(1 + tanh u) cancels to ~1e-16 absolute for x < -7
    # (far below binary16's smallest subnormal, 6e-8), where the oracle's form does not
    assert np.allclose(Y, ref, rtol=1e-13, atol=1e-14)
    assert np.array_equal(C.view(np.uint16), Y.astype(np.float16).view(np.uint16))
    assert np.any(x < -7)                     # the far negative tail is exercised too


def test_gelu_odd_part_identity_and_limits():
    # tanh-form GELU satisfies GELU(-x) = GELU(x) - x; GELU(0) = 0; GELU(x) -> x, GELU(-x) -> 0
    vals = np.array([0.0, 0.25, 1.0, 2.5, 7.0, 12.0], dtype=np.float16)
    K = vals.shape[0]
    A = np.stack([vals, -vals]).astype(np.float16)            # rows x and -x
    zero_bias = np.zeros(K, np.float16)
    _, Y = oracle.gemm_epilogue(A, np.eye(K, dtype=np.float16), kind=oracle.EPI_BIAS_GELU,
                                bias=zero_bias, return_pre=True)
    x = vals.astype(np.float64)
    assert np.allclose(Y[1], Y[0] - x, rtol=0, atol=1e-12)
    assert Y[0, 0] == 0.0
    assert abs(Y[0, -1] - 12.0) < 1e-12 and abs(Y[1, -1]) < 1e-12


def test_gelu_all_ones_with_bias():
    # sum = K exactly; Y = GELU(K + bias[n])
    K, N = 6, 4
    bias = np.array([-8.0, -6.0, -1.5, 0.5], np.float16)
    C, Y = oracle.gemm_epilogue(np.ones((3, K), np.float16), np.ones((K, N), np.float16),
                                kind=oracle.EPI_BIAS_GELU, bias=bias, return_pre=True)
    ref = _torch_gelu_tanh(K + bias.astype(np.float64))
    assert np.allclose(Y, ref[None, :], rtol=1e-13, atol=1e-14)


def test_gelu_k_zero_is_gelu_of_bias():
    bias = np.array([-3.0, -0.5, 0.0, 0.5, 3.0, 9.0, -9.0, 1.0], np.float16)
    C, Y = oracle.gemm_epilogue(np.zeros((2, 0), np.float16), np.zeros((0, 8), np.float16),
                                kind=oracle.EPI_BIAS_GELU, bias=bias, return_pre=True)
    assert np.allclose(Y, _torch_gelu_tanh(bias.astype(np.float64))[None, :], rtol=1e-13, atol=1e-14)
