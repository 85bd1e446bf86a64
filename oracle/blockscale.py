"""Oracle for block-scaled operands: C = sum_k (sA * a)(sB * b) with one scale per tile.

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the product library; it
shares no code with the CUDA path.

Source: "H100 . WGMMA Part 2" (runguoli.com H100 course notes, Lesson 7), section 11:
besides one scale per tensor and one per row or column, FP8 operands can carry one
scale per small tile of the matrix (block-wise scaling, MXFP8 / microscaling; the
page's examples are 16 x 16 and 32 x 32 tiles).

Reading (listed in the design notes): each operand, stored K-major (A: M x K, B: N x K),
is cut into br x bk tiles of (rows x K); tile (r, t) of A holds the elements A[i][k] with
i // br = r and k // bk = t and is multiplied by sA[r][t] (likewise B with sB), so

    C[i][j] = sum_k  dec(A[i][k]) sA[i // br][k // bk] * dec(B[j][k]) sB[j // br][k // bk].

br = 1, bk = 32 is the microscaling layout (one scale per 32 consecutive K elements of
a row); br = bk = 32 the page's 32 x 32 tiles.  The scales are FP64 values here (the
formats' power-of-two scales are a special case).  The sum is taken in FP64 by a
matrix product of the scaled, decoded operands.

The page gives one tile shape per matrix; the two operands may take different ones
(reading: B's tiles may have their own row count br_b, sharing bk, so that k-block
boundaries coincide), e.g. 1 x 128 tiles of A with 128 x 128 tiles of B:

    C[i][j] = sum_k  dec(A[i][k]) sA[i // br][k // bk] * dec(B[j][k]) sB[j // br_b][k // bk].
"""
from __future__ import annotations

import numpy as np


def expand(s: np.ndarray, rows: int, K: int, br: int, bk: int) -> np.ndarray:
    """The rows x K matrix whose (i, k) entry is s[i // br][k // bk]."""
    s = np.asarray(s, dtype=np.float64)
    if s.shape != (-(-rows // br), -(-K // bk)):
        raise ValueError(f"scale shape {s.shape} does not tile {rows} x {K} by {br} x {bk}")
    return np.repeat(np.repeat(s, br, axis=0), bk, axis=1)[:rows, :K]


def gemm_block_scaled(a: np.ndarray, b: np.ndarray, sA: np.ndarray, sB: np.ndarray, block=(1, 32), rows=None,
                      block_rows_b=None):
    """C (M x N, FP64) from decoded operands a (M x K) and b (N x K) and their tile
    scales sA (ceil(M / br) x ceil(K / bk)) and sB (ceil(N / br_b) x ceil(K / bk)),
    br_b = block_rows_b (default br).  rows: only these rows of C (the same definition
    evaluated for a subset of i)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    br, bk = block
    br_b = br if block_rows_b is None else block_rows_b
    (M, K), (N, K2) = a.shape, b.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    if rows is None:
        return (a * expand(sA, M, K, br, bk)) @ (b * expand(sB, N, K, br_b, bk)).T
    rows = np.asarray(rows, dtype=np.int64)
    s = np.asarray(sA, dtype=np.float64)
    if s.shape != (-(-M // br), -(-K // bk)):
        raise ValueError(f"scale shape {s.shape} does not tile {M} x {K} by {br} x {bk}")
    sa_rows = np.repeat(s[rows // br], bk, axis=1)[:, :K]
    return (a[rows] * sa_rows) @ (b * expand(sB, N, K, br_b, bk)).T
