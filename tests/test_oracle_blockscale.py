"""Pins for the block-scaled operand oracle (oracle/blockscale.py): brute force on tiny
shapes, the reduction to the plain GEMM, uniform scales factoring out, and a single
tile's scale acting only on that tile's partial sums."""
import itertools

import numpy as np
import pytest

import oracle
import synthetic
from oracle import blockscale as BS


def test_brute_force_tiny():
    rng = np.random.default_rng(1)
    M, N, K, br, bk = 3, 2, 5, 2, 2
    a, b = rng.normal(size=(M, K)), rng.normal(size=(N, K))
    sA, sB = rng.uniform(0.5, 2, size=(2, 3)), rng.uniform(0.5, 2, size=(1, 3))
    want = np.zeros((M, N))
    for i, j, k in itertools.product(range(M), range(N), range(K)):
        want[i, j] += a[i, k] * sA[i // br, k // bk] * b[j, k] * sB[j // br, k // bk]
    assert np.allclose(BS.gemm_block_scaled(a, b, sA, sB, block=(br, bk)), want, rtol=1e-14, atol=1e-14)


def test_unit_scales_are_the_plain_gemm():
    M, N, K = 40, 24, 96
    A = synthetic.e4m3_bytes(synthetic.draw("int:8", 31, M * K).reshape(M, K).astype(np.float32))
    B = synthetic.e4m3_bytes(synthetic.draw("int:8", 32, N * K).reshape(N, K).astype(np.float32))
    a, b = oracle.decode(A, "e4m3"), oracle.decode(B, "e4m3")
    for block in ((1, 32), (32, 32), (16, 16)):
        br, bk = block
        ones_a = np.ones((-(-M // br), -(-K // bk)))
        ones_b = np.ones((-(-N // br), -(-K // bk)))
        z, _ = oracle.gemm(A, B, "e4m3")
        assert np.array_equal(BS.gemm_block_scaled(a, b, ones_a, ones_b, block), z)


def test_uniform_scales_factor_out_and_one_tile_acts_locally():
    rng = np.random.default_rng(2)
    M, N, K = 33, 17, 70          # ragged against 32 x 32 tiles
    a = rng.integers(-8, 9, size=(M, K)).astype(np.float64)
    b = rng.integers(-8, 9, size=(N, K)).astype(np.float64)
    shA, shB = (2, 3), (1, 3)
    plain = a @ b.T
    C = BS.gemm_block_scaled(a, b, np.full(shA, 4.0), np.full(shB, 0.25), block=(32, 32))
    assert np.array_equal(C, plain)                # 4 * 0.25 = 1, exact on integers
    sA = np.ones(shA)
    sA[1, 2] = 8.0                                 # rows 32.., K 64..69
    C = BS.gemm_block_scaled(a, b, sA, np.ones(shB), block=(32, 32))
    part = a[32:, 64:] @ b[:, 64:].T
    assert np.array_equal(C[:32], plain[:32])
    assert np.array_equal(C[32:], plain[32:] + 7.0 * part)


def test_scale_shapes_must_tile_the_operands():
    a, b = np.zeros((5, 64)), np.zeros((3, 64))
    with pytest.raises(ValueError):
        BS.gemm_block_scaled(a, b, np.ones((5, 3)), np.ones((3, 2)), block=(1, 32))


def test_row_subset_equals_the_full_result_rows():
    # the rows option evaluates the same definition for a subset of C's rows, ragged row
    # blocks included: exactly the full result's rows where the arithmetic is exact (small
    # integers, power-of-two scales), and within FP64 rounding otherwise (the library matrix
    # product sums in an order that depends on the shapes)
    rng = np.random.default_rng(3)
    M, N, K = 70, 20, 96
    rows = np.array([0, 1, 31, 32, 33, 63, 64, 69])
    for br, bk in ((1, 32), (32, 32), (16, 64)):
        shA, shB = (-(-M // br), -(-K // bk)), (-(-N // br), -(-K // bk))
        a = rng.integers(-8, 9, size=(M, K)).astype(np.float64)
        b = rng.integers(-8, 9, size=(N, K)).astype(np.float64)
        sA, sB = 2.0 ** rng.integers(-3, 4, size=shA), 2.0 ** rng.integers(-3, 4, size=shB)
        full = BS.gemm_block_scaled(a, b, sA, sB, (br, bk))
        assert np.array_equal(BS.gemm_block_scaled(a, b, sA, sB, (br, bk), rows=rows), full[rows])
        a, b = rng.normal(size=(M, K)), rng.normal(size=(N, K))
        sA, sB = rng.uniform(0.5, 2, size=shA), rng.uniform(0.5, 2, size=shB)
        full = BS.gemm_block_scaled(a, b, sA, sB, (br, bk))
        assert np.allclose(BS.gemm_block_scaled(a, b, sA, sB, (br, bk), rows=rows), full[rows], rtol=1e-13, atol=1e-13)
    with pytest.raises(ValueError):
        BS.gemm_block_scaled(a, b, np.ones((2, 3)), np.ones((1, 3)), (1, 32), rows=[0])


def test_brute_force_tiny_with_separate_row_blocks_for_b():
    rng = np.random.default_rng(4)
    M, N, K, br, br_b, bk = 3, 5, 6, 1, 4, 4
    a, b = rng.normal(size=(M, K)), rng.normal(size=(N, K))
    sA, sB = rng.uniform(0.5, 2, size=(3, 2)), rng.uniform(0.5, 2, size=(2, 2))
    want = np.zeros((M, N))
    for i, j, k in itertools.product(range(M), range(N), range(K)):
        want[i, j] += a[i, k] * sA[i // br, k // bk] * b[j, k] * sB[j // br_b, k // bk]
    got = BS.gemm_block_scaled(a, b, sA, sB, block=(br, bk), block_rows_b=br_b)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-14)
    rows = np.array([0, 2])
    assert np.allclose(BS.gemm_block_scaled(a, b, sA, sB, (br, bk), rows=rows, block_rows_b=br_b), want[rows],
                       rtol=1e-14, atol=1e-14)
    # B's row blocks equal to A's: the one-shape form
    sB2 = rng.uniform(0.5, 2, size=(5, 2))
    assert np.array_equal(BS.gemm_block_scaled(a, b, sA, sB2, (1, bk), block_rows_b=1),
                          BS.gemm_block_scaled(a, b, sA, sB2, (1, bk)))
    with pytest.raises(ValueError):   # sB must tile B by br_b
        BS.gemm_block_scaled(a, b, sA, sB, block=(br, bk))
