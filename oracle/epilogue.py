"""Oracle for the extended fused epilogue, in FP64, in the pages' order.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product library.  It shares no code
with the CUDA path.

Sources (page title, section):
  * "H100 . Kernel Design" (runguoli.com H100 course notes, Lesson 8), section
    12.1, the list of epilogue operations: alpha*Acc and alpha*Acc + beta*C,
    per-row / per-column bias, activations ReLU / GELU / SiLU, aux tensor store,
    amax tracking on the FP8 path, per-row / per-column scale fusion; and
    section 12.2, their order:
      1. load the tile's inputs (Acc, optional C, bias, scales)
      2. Z = alpha*Acc + beta*C   (Z = alpha*Acc without C)
      3. Z += row or column bias
      4. Y = activation(Z)
      5. output scale / quantisation, gathering amax where needed
      6. materialise D and the optional aux output (here: Z, before the activation)
      7. final type conversion and store.
  * "H100 . WGMMA Part 2" (Lesson 7), sections 10-11: e4m3 saturates at 448
    (clamping keeps the sign); scaling factors are tensor-wise, vector-wise
    (one per row or column) or block-wise.

Readings where the pages leave a step open (each is listed in the design notes):
  * the vector-wise scales are dequantisation factors of the operands: one per
    row of A (length M) and one per row of B, i.e. per column of the output
    (length N); like the tensor-wise scales they multiply the accumulator
    before beta*C and the bias are added;
  * GELU is the exact form x * Phi(x), Phi the standard normal CDF (the pages
    name GELU without a formula); SiLU is x * sigmoid(x);
  * amax is max |Y| over the whole output, Y after the activation and before the
    output scale (the value the next step's quantisation scale is derived from);
  * the output scale d multiplies Y before the cast: D = cast(d * Y); the FP8
    cast rounds to nearest even and saturates to +-448 (section 10's clamping
    mode; the pages' conversion is cvt.rn.satfinite);
  * the aux output holds Z, the pre-activation value (section 12.3, the
    training template "AuxOut = Z").
"""
from __future__ import annotations

import math
from bisect import bisect_left
from dataclasses import dataclass
from functools import lru_cache

import numpy as np

ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU = 0, 1, 2, 3
BIAS_NONE, BIAS_COL, BIAS_ROW = 0, 1, 2
E4M3_MAX = 448.0


# --------------------------------------------------------------- activations

def _phi(x: float) -> float:
    """Standard normal CDF in FP64; erfc keeps the left tail accurate."""
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def gelu(z: np.ndarray) -> np.ndarray:
    """GELU(x) = x * Phi(x)."""
    z = np.asarray(z, dtype=np.float64)
    flat = z.ravel()
    return np.array([x * _phi(x) for x in flat], dtype=np.float64).reshape(z.shape)


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x), written so neither side overflows."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    e = np.exp(z[~pos])
    out[~pos] = z[~pos] * e / (1.0 + e)
    return out


def activation(z: np.ndarray, act: int) -> np.ndarray:
    if act == ACT_NONE:
        return np.asarray(z, dtype=np.float64).copy()
    if act == ACT_RELU:
        return np.maximum(z, 0.0)
    if act == ACT_GELU:
        return gelu(z)
    if act == ACT_SILU:
        return silu(z)
    raise ValueError(act)


# largest slope |act'(x)| over the reals: the error of Z passes into Y at most this much
LIPSCHITZ = {ACT_NONE: 1.0, ACT_RELU: 1.0, ACT_GELU: 1.1290, ACT_SILU: 1.0999}


# --------------------------------------------------------------- FP8 output cast

def _e4m3_value(code: int) -> float:
    """Value of a non-negative e4m3 code 0..0x7E from the format: 4 exponent bits
    (bias 7), 3 mantissa bits, subnormals at exponent field 0."""
    e, m = (code >> 3) & 0xF, code & 7
    if e == 0:
        return m * 2.0 ** -9
    return (1.0 + m / 8.0) * 2.0 ** (e - 7)


@lru_cache(maxsize=1)
def _e4m3_grid():
    return tuple(_e4m3_value(c) for c in range(0x7F))   # 0x7F is NaN


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """FP64 -> e4m3 codes: round to nearest, ties to the even code, saturating
    to the largest finite magnitude 448 with the sign kept."""
    grid = _e4m3_grid()
    xs = np.asarray(x, dtype=np.float64)
    out = np.empty(xs.shape, dtype=np.uint8)
    flat_in, flat_out = xs.ravel(), out.reshape(-1)
    for idx, v in enumerate(flat_in):
        if math.isnan(v):
            raise ValueError("NaN has no saturating e4m3 encoding here")
        a = abs(v)
        if a >= E4M3_MAX:
            code = 0x7E
        else:
            hi = bisect_left(grid, a)           # grid[hi-1] < a <= grid[hi]
            if grid[hi] == a:
                code = hi
            else:
                lo = hi - 1
                dl, dh = a - grid[lo], grid[hi] - a
                code = lo if dl < dh else hi if dh < dl else (lo if lo % 2 == 0 else hi)
        flat_out[idx] = code | (0x80 if math.copysign(1.0, v) < 0 else 0)
    return out


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    grid = _e4m3_grid()
    c = np.asarray(codes, dtype=np.uint8)
    mag = np.array([grid[int(v) & 0x7F] if (int(v) & 0x7F) != 0x7F else np.nan for v in c.ravel()])
    sign = np.where((c.ravel() & 0x80) != 0, -1.0, 1.0)
    return (sign * mag).reshape(c.shape)


# --------------------------------------------------------------- the epilogue

@dataclass
class Epilogue:
    """What the fused epilogue does; defaults reduce it to D = Acc."""
    alpha: float = 1.0
    beta: float = 0.0
    scales: tuple | None = None          # tensor-wise (sA, sB)
    row_scale: np.ndarray | None = None  # FP32[M] (per row of A)
    col_scale: np.ndarray | None = None  # FP32[N] (per row of B = column of D)
    c_in: np.ndarray | None = None       # FP64 values of C, M x N
    bias: np.ndarray | None = None
    bias_mode: int = BIAS_NONE
    act: int = ACT_NONE
    d_scale: float = 1.0


def apply(acc: np.ndarray, absdot: np.ndarray, e: Epilogue, rows=None):
    """Steps 2-5 of the pages' order on the raw FP64 accumulator `acc` (rows x N).

    Returns (Z, Y, D_pre, bound_z) where Z is the pre-activation value, Y the
    activation, D_pre = d * Y before the cast, and bound_z = |total scale| *
    sum_k |a||b| (the magnitude the accumulation error is relative to).
    `rows` selects which rows of the full problem acc holds (default all).
    """
    acc = np.asarray(acc, dtype=np.float64)
    nr, N = acc.shape
    ridx = np.arange(nr) if rows is None else np.asarray(rows, dtype=np.int64)
    s = float(e.alpha)
    if e.scales is not None:
        s *= float(e.scales[0]) * float(e.scales[1])
    scale = np.full((nr, N), s, dtype=np.float64)
    if e.row_scale is not None:
        scale *= np.asarray(e.row_scale, dtype=np.float64)[ridx][:, None]
    if e.col_scale is not None:
        scale *= np.asarray(e.col_scale, dtype=np.float64)[None, :]
    Z = scale * acc                                       # alpha * Acc, all scales folded in
    if e.c_in is not None and e.beta != 0.0:
        Z = Z + float(e.beta) * np.asarray(e.c_in, dtype=np.float64)[ridx]   # + beta * C
    if e.bias_mode == BIAS_COL:
        Z = Z + np.asarray(e.bias, dtype=np.float64)[None, :]
    elif e.bias_mode == BIAS_ROW:
        Z = Z + np.asarray(e.bias, dtype=np.float64)[ridx][:, None]
    Y = activation(Z, e.act)
    D_pre = float(e.d_scale) * Y
    return Z, Y, D_pre, np.abs(scale) * np.asarray(absdot, dtype=np.float64)


# ------------------------------------------------- block scale factor generation
#
# "H100 . Kernel Design" section 12.1 lists block scale factor generation among the
# epilogue operations, and "H100 . WGMMA Part 2" section 11 describes block-wise scaling
# (MXFP8, microscaling): the matrix is cut into small tiles (its examples: 16 x 16 or
# 32 x 32), one scale per tile.  Reading (listed in the design notes): the output Y is cut
# into br x bc tiles (32 x 32 by default, ragged at the edges); each tile gets a
# power-of-two scale X = 2^E, E = floor(log2(amax)) - 8 with amax = max |Y| over the tile
# (8 = the exponent of e4m3's largest power of two, as the microscaling format derives its
# shared exponent), E = 0 for an all-zero tile; the tile's codes are e4m3(Y / X), rounded
# to nearest even and saturated to +-448.  X is exact, so Y / X is too.

def block_scale_e4m3(Y: np.ndarray, block=(32, 32)):
    """(codes, E): e4m3 codes of Y (its shape) and the int exponents E of each tile's
    scale 2^E, shape (ceil(rows / br), ceil(cols / bc))."""
    Y = np.asarray(Y, dtype=np.float64)
    br, bc = block
    R, C = Y.shape
    E = np.zeros((-(-R // br), -(-C // bc)), dtype=np.int64)
    codes = np.zeros(Y.shape, dtype=np.uint8)
    for i in range(E.shape[0]):
        for j in range(E.shape[1]):
            t = Y[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
            m = float(np.max(np.abs(t)))
            e = math.floor(math.log2(m)) - 8 if m > 0 else 0
            E[i, j] = e
            codes[i * br:(i + 1) * br, j * bc:(j + 1) * bc] = encode_e4m3(t / 2.0 ** e)
    return codes, E


def amax(Y: np.ndarray) -> float:
    """max |Y| over the output (0 for an empty output)."""
    return float(np.max(np.abs(Y))) if np.size(Y) else 0.0
