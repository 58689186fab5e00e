"""Pins for the CPU oracle: each check ties it to something other than itself
(closed forms, textbook values, exhaustive decoding, a library routine on
exactly representable data, exact rational brute force on tiny inputs)."""
from fractions import Fraction

import numpy as np
import pytest

import golden_values
import oracle
from dense_gemm_tmem_gb300 import inputs


def f64(x):
    return np.asarray(x, dtype=np.float64)


def test_f16_decode_exhaustive():
    """Every binary16 code decodes to numpy's widening of the same code
    (sign of zero included; NaN codes decode to NaN)."""
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    # a few hand-checked values: 1.0, -2.0, largest normal, smallest subnormal
    assert oracle.f16_to_f64(0x3C00) == 1.0
    assert oracle.f16_to_f64(0xC000) == -2.0
    assert oracle.f16_to_f64(0x7BFF) == 65504.0
    assert oracle.f16_to_f64(0x0001) == 2.0 ** -24


@pytest.mark.parametrize("dt", [np.float16, np.float32])
def test_textbook_2x2(dt):
    A = np.array([[1, 2], [3, 4]], dtype=dt)
    B = np.array([[5, 6], [7, 8]], dtype=dt)
    C = oracle.gemm(A, B)
    assert np.array_equal(C, [[19, 22], [43, 50]])
    C = oracle.gemm(A, B, bias=np.array([1, -1], dtype=np.float32))
    assert np.array_equal(C, [[20, 21], [44, 49]])
    # BA differs from AB: catches swapped operands
    assert np.array_equal(oracle.gemm(B, A), [[23, 34], [31, 46]])


def _frac_matmul(A, B, bias):
    M, K = A.shape
    N = B.shape[1]
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                     for k in range(K)), Fraction(0))
            if bias is not None:
                s += Fraction(float(bias[j]))
            row.append(s)
        out.append(row)
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 4), (3, 5, 7), (4, 1, 9)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_tiny_exact_rational(M, N, K, with_bias):
    """Exact rational brute force on tiny fp16 inputs: the binary64 oracle must
    be within one rounding of the exact value per term."""
    A = inputs.draw((M, K), 11 + M, "uniform", inputs.F16)
    B = inputs.draw((K, N), 12 + N, "uniform", inputs.F16)
    bias = inputs.draw((N,), 13 + K, "uniform", inputs.F32) if with_bias else None
    C = oracle.gemm(A, B, bias)
    exact = _frac_matmul(A, B, bias)
    for i in range(M):
        for j in range(N):
            scale = sum(abs(float(A[i, k]) * float(B[k, j])) for k in range(K))
            scale += abs(float(bias[j])) if bias is not None else 0.0
            err = abs(Fraction(C[i, j]) - exact[i][j])
            assert err <= Fraction(2.0 ** -50) * Fraction(scale + 1e-300)


def test_identity_and_negated_identity():
    n = 37
    eye = np.eye(n, dtype=np.float16)
    B = inputs.draw((n, 23), 5, "uniform", inputs.F16)
    assert np.array_equal(oracle.gemm(eye, B), B.astype(np.float64))
    assert np.array_equal(oracle.gemm(-eye, B), -B.astype(np.float64))
    A = inputs.draw((19, n), 6, "uniform", inputs.F16)
    assert np.array_equal(oracle.gemm(A, eye), A.astype(np.float64))


def test_permutation_rows_and_columns():
    """P·B permutes B's rows; B·P permutes its columns (catches index swaps)."""
    rng = np.random.default_rng(3)
    n = 64
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float16)
    P[np.arange(n), perm] = 1
    B = inputs.draw((n, 40), 7, "uniform", inputs.F16)
    assert np.array_equal(oracle.gemm(P, B), B[perm].astype(np.float64))
    A = inputs.draw((33, n), 8, "uniform", inputs.F16)
    # (A·P)[i, j] = A[i, k] with perm[k] = j
    inv = np.argsort(perm)
    assert np.array_equal(oracle.gemm(A, P), A[:, inv].astype(np.float64))


def test_rank_one_closed_form():
    """A[i,k] = u_i, B[k,j] = v_j  =>  C[i,j] = K*u_i*v_j + bias_j."""
    M, N, K = 17, 29, 300
    u = np.arange(-8, 9, dtype=np.float64)[:M]
    v = np.arange(-14, 15, dtype=np.float64)[:N] / 4
    A = np.repeat(u[:, None], K, axis=1).astype(np.float16)
    B = np.repeat(v[None, :], K, axis=0).astype(np.float16)
    bias = np.linspace(-3, 3, N).astype(np.float32)
    C = oracle.gemm(A, B, bias)
    expect = K * np.outer(u, v) + bias.astype(np.float64)[None, :]
    assert np.array_equal(C, expect)


def test_all_ones_gives_k():
    M, N, K = 9, 11, 1000
    A = np.ones((M, K), np.float16)
    B = np.ones((K, N), np.float16)
    assert np.array_equal(oracle.gemm(A, B), np.full((M, N), float(K)))
    bias = np.arange(N, dtype=np.float32) - 5
    expect = np.broadcast_to(K + bias.astype(np.float64)[None, :], (M, N))
    assert np.array_equal(oracle.gemm(A, B, bias), expect)


@pytest.mark.parametrize("dt", [inputs.F16, inputs.F32])
def test_integer_inputs_match_integer_matmul(dt):
    """Integer-valued data: every partial sum is an exact integer, so the
    oracle must equal numpy's int64 matrix product exactly."""
    M, N, K = 70, 90, 513
    lo, hi = inputs.int_range(dt)
    A = inputs.draw((M, K), 21, "int", dt, lo, hi)
    B = inputs.draw((K, N), 22, "int", dt, lo, hi)
    bias = inputs.draw((N,), 23, "int", inputs.F32, -2, 2)
    ref = A.astype(np.int64) @ B.astype(np.int64) + bias.astype(np.int64)[None, :]
    assert np.array_equal(oracle.gemm(A, B, bias), ref.astype(np.float64))


def test_fp32_inputs_against_library_matmul():
    """Random fp32 data: binary64 accumulation agrees with numpy's float64
    product to within the float64 rounding bound."""
    M, N, K = 31, 47, 257
    A = inputs.draw((M, K), 31, "uniform", inputs.F32)
    B = inputs.draw((K, N), 32, "uniform", inputs.F32)
    C = oracle.gemm(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    bound = K * 2.0 ** -52 * (np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64))
    assert np.all(np.abs(C - ref) <= bound)


@pytest.mark.parametrize("a_major", [0, 1])
@pytest.mark.parametrize("b_major", [0, 1])
def test_layouts_read_transposed_storage(a_major, b_major):
    """Column-major storage is the transposed array; all four layout pairs give
    the same numbers as row-major storage of the same matrices."""
    M, N, K = 23, 41, 67
    A = inputs.draw((M, K), 41, "uniform", inputs.F16)
    B = inputs.draw((K, N), 42, "uniform", inputs.F16)
    ref = oracle.gemm(A, B)
    As = A if a_major == 0 else np.ascontiguousarray(A.T)
    Bs = B if b_major == 0 else np.ascontiguousarray(B.T)
    C = oracle.gemm(As, Bs, a_major=a_major, b_major=b_major)
    assert np.array_equal(C, ref)


def test_rows_subset_and_threads_bitwise():
    M, N, K = 64, 48, 200
    A = inputs.draw((M, K), 51, "normal", inputs.F16)
    B = inputs.draw((N, K), 52, "normal", inputs.F16)
    bias = inputs.draw((N,), 53, "normal", inputs.F32)
    full1 = oracle.gemm(A, B, bias, b_major=1, threads=1)
    full8 = oracle.gemm(A, B, bias, b_major=1, threads=8)
    assert np.array_equal(full1, full8)
    rows = [0, 5, 63, 17, 17]
    sub = oracle.gemm_rows(A, B, bias, b_major=1, rows=rows, threads=3)
    assert np.array_equal(sub, full1[rows])


def test_degenerate_shapes():
    A = np.zeros((3, 0), np.float16)
    B = np.zeros((0, 4), np.float16)
    assert np.array_equal(oracle.gemm(A, B), np.zeros((3, 4)))
    bias = np.array([1.5, -2, 0, 7], np.float32)
    assert np.array_equal(oracle.gemm(A, B, bias), np.tile(bias.astype(np.float64), (3, 1)))
    assert oracle.gemm(np.zeros((0, 5), np.float16), np.zeros((5, 4), np.float16)).shape == (0, 4)
    assert oracle.gemm(np.zeros((3, 5), np.float16), np.zeros((5, 0), np.float16)).shape == (3, 0)


def test_bad_arguments():
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((3, 5), np.float16), np.zeros((4, 2), np.float16))
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((3, 5), np.float16), np.zeros((5, 2), np.float16),
                    bias=np.zeros(3, np.float32))
    with pytest.raises(ValueError):
        oracle.gemm_rows(np.zeros((3, 5), np.float16), np.zeros((5, 2), np.float16),
                         rows=[3])
    with pytest.raises(TypeError):
        oracle.gemm(np.zeros((3, 5), np.float64), np.zeros((5, 2), np.float64))


@pytest.mark.parametrize("dt", [np.float16, np.float32])
@pytest.mark.parametrize("b_major", [0, 1])
def test_golden_block_sum(dt, b_major):
    """The pages' worked reduction (0 + 1 + ... + 255 = 32640, printed in
    tests/golden/block_sum_arange256.txt) as a 1 x K by K x 1 product, in
    both operand orders and both storage orders of B."""
    gv = golden_values.load("block_sum_arange256.txt")
    K, want = int(gv["K"]), gv["C"]
    row = np.arange(K, dtype=dt).reshape(1, K)
    ones = np.ones((K, 1), dtype=dt)
    Bs = ones.T.copy() if b_major else ones  # column-major B is stored (N, K)
    assert oracle.gemm(row, Bs, b_major=b_major)[0, 0] == want
    # the same sum with the ramp in B and the ones in A
    ramp = row.T.copy()
    Bs = ramp.T.copy() if b_major else ramp
    assert oracle.gemm(ones.T.copy(), Bs, b_major=b_major)[0, 0] == want
    # a bias of -want cancels it exactly; a dropped bias would not
    got = oracle.gemm(row, ones, bias=np.array([-want], dtype=np.float32))
    assert got[0, 0] == 0.0
