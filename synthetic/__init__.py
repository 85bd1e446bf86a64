"""Seeded synthetic GEMM inputs, shared by the tests, the bench and the oracle.

This module draws random numbers and encodes them into the storage formats the
GEMM consumes (BF16 bit patterns, FP8-e4m3 bytes plus a per-tensor FP32 scale,
FP32 bias vectors).  It holds none of the GEMM's own arithmetic: no products,
no sums, no epilogue, no tile schedule.  Both the CUDA path and the oracle read
the bytes produced here, so the encoding choices below fix the inputs, not the
method.

Random stream: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Element i of a stream seeded with s is
mix(s + (i + 1) * 0x9E3779B97F4A7C15 mod 2^64), turned into a 53-bit uniform
double in [0, 1).  Normals come from Box-Muller on consecutive uniform pairs.

Encodings:
  * BF16: the FP64 draw is rounded to FP32 (round-to-nearest-even), then to
    BF16 (round-to-nearest-even on the FP32 bit pattern).
  * FP8-e4m3 with a tensor-wise scale (the "tensor-wise" option of the FP8
    scaling factors in the H100 course notes, WGMMA Part 2, section 11):
    x32 = FP32(draw); s = FP32(amax(|x32|) / 448); q = e4m3(x32 / s) with
    round-to-nearest-even and saturation to +-448 (the satfinite behaviour the
    same notes describe in section 13).  e4m3 has no infinities; the bytes
    0x7F / 0xFF (NaN) are never produced.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

E4M3_MAX = 448.0
E5M2_MAX = 57344.0


def splitmix64(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """uint64 outputs number offset .. offset+count-1 of the splitmix64 stream."""
    idx = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, count: int) -> np.ndarray:
    """53-bit uniform doubles in [0, 1)."""
    return (splitmix64(seed, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(seed: int, count: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    return lo + (hi - lo) * uniform01(seed, count)


def normal(seed: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """Box-Muller: element 2j = r cos(t), element 2j+1 = r sin(t)."""
    pairs = (count + 1) // 2
    u = uniform01(seed, 2 * pairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))  # log(1 - u1), u1 < 1 so never log(0)
    t = (2.0 * np.pi) * u2
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:count] * sigma


def draw(dist: str, seed: int, count: int) -> np.ndarray:
    """dist: 'uniform' (U[-1,1]), 'normal' (N(0,1)) or 'normal:<sigma>'."""
    if dist == "uniform":
        return uniform(seed, count)
    if dist == "normal":
        return normal(seed, count)
    if dist.startswith("normal:"):
        return normal(seed, count, float(dist.split(":", 1)[1]))
    if dist.startswith("int:"):
        # small integers in [-r, r], used for exactness cases
        r = int(dist.split(":", 1)[1])
        return np.floor(uniform01(seed, count) * (2 * r + 1)) - r
    raise ValueError(f"unknown distribution {dist!r}")


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP64 -> FP32 (RNE) -> BF16 bit pattern (RNE), as uint16."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (f >> np.uint64(16)) & np.uint64(1)
    rounded = (f + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def _fp8_bytes(x32: np.ndarray, mbits: int, ebias: int, vmax: float) -> np.ndarray:
    """FP32 values -> FP8 codes with `mbits` mantissa bits and exponent bias `ebias`,
    round-to-nearest-even, saturating to +-vmax (the largest finite value)."""
    v = np.asarray(x32, dtype=np.float32).astype(np.float64)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    a = np.minimum(np.abs(v), vmax)
    emin = 1 - ebias                       # exponent of the smallest normal
    # exponent of a (for a in the normal range); frexp gives a = f * 2^e, f in [0.5, 1)
    _, e = np.frexp(a)
    e = e.astype(np.int64) - 1  # a = 1.xxx * 2^e
    e = np.maximum(e, emin)     # below 2^emin the spacing stays 2^(emin - mbits) (subnormals)
    step = np.ldexp(1.0, (e - mbits).astype(np.int32))
    q = np.rint(a / step) * step  # np.rint rounds half to even
    q = np.minimum(q, vmax)
    # back to a code
    _, e2 = np.frexp(q)
    e2 = e2.astype(np.int64) - 1
    normal_ = q >= 2.0 ** emin
    exp_field = np.where(normal_, e2 + ebias, 0)
    mant = np.where(normal_, q / np.ldexp(1.0, e2.astype(np.int32)) - 1.0, q / 2.0 ** (emin - mbits))
    mant = np.where(normal_, mant * (1 << mbits), mant)
    code = (exp_field.astype(np.int64) << mbits) | np.rint(mant).astype(np.int64)
    code = np.where(q == 0, 0, code)
    code = code | (sign.astype(np.int64) << 7)
    return code.astype(np.uint8)


def e4m3_bytes(x32: np.ndarray) -> np.ndarray:
    """FP32 values -> e4m3 bytes, round-to-nearest-even, saturating to +-448.

    e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field
    0 is subnormal (value m * 2^-9); the all-ones pattern S.1111.111 is NaN.
    """
    return _fp8_bytes(x32, 3, 7, E4M3_MAX)


def e5m2_bytes(x32: np.ndarray) -> np.ndarray:
    """FP32 values -> e5m2 bytes, round-to-nearest-even, saturating to +-57344.

    e5m2: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits; exponent field
    0 is subnormal (value m * 2^-16); exponent field 31 holds infinity and NaN,
    which saturation never produces.
    """
    return _fp8_bytes(x32, 2, 15, E5M2_MAX)


def _fp8_quantise(x: np.ndarray, encode, vmax: float):
    x32 = np.asarray(x, dtype=np.float32)
    amax = float(np.max(np.abs(x32))) if x32.size else 0.0
    scale = np.float32(amax) / np.float32(vmax) if amax > 0 else np.float32(1.0)
    scale = np.float32(scale)
    return encode(x32 / scale), scale


def e4m3_quantise(x: np.ndarray):
    """Tensor-wise FP8 quantisation: returns (bytes, scale) with x ~ scale * decode(bytes)."""
    return _fp8_quantise(x, e4m3_bytes, E4M3_MAX)


def e5m2_quantise(x: np.ndarray):
    """Tensor-wise e5m2 quantisation: returns (bytes, scale) with x ~ scale * decode(bytes)."""
    return _fp8_quantise(x, e5m2_bytes, E5M2_MAX)


# input element types: A's and B's format ("e4m3_e5m2" = A e4m3, B e5m2)
DTYPES = ("bf16", "e4m3", "e5m2", "e4m3_e5m2", "e5m2_e4m3")


def operand_types(dtype: str):
    """(format of A, format of B) for a dtype name."""
    if dtype not in DTYPES:
        raise ValueError(dtype)
    if "_" in dtype:
        a, b = dtype.split("_")
        return a, b
    return dtype, dtype


# Seeds per matrix: A = 1000 + c, B = 2000 + c, bias = 3000 + c, the epilogue's addend
# matrix (beta * C) = 4000 + c, c = config number.
SEED_A, SEED_B, SEED_BIAS, SEED_C = 1000, 2000, 3000, 4000


def make_group_rows(groups: int, total: int, case: int, spread: float = 0.5):
    """Seeded row counts of `groups` groups adding up to `total`: each group's share is
    (1 - spread) / groups + spread * w_g / sum(w), w_g uniform in [0, 1) (seed 5000 + c),
    rounded down, and the remainder goes to the last group."""
    w = uniform01(5000 + case, groups)
    share = (1.0 - spread) / groups + spread * w / w.sum()
    rows = np.floor(share * total).astype(np.int64)
    rows[-1] += total - rows.sum()
    return [int(r) for r in rows]


def make_group_shapes(groups: int, case: int, m_range=(256, 4096), n_choices=(1024, 2048, 4096, 8192),
                      k_choices=(1024, 2048, 4096, 8192)):
    """Seeded (M_g, N_g, K_g) of `groups` GEMMs of different shapes (seed 6000 + c):
    M_g uniform in m_range rounded to 8, N_g and K_g drawn from the choices."""
    r = splitmix64(6000 + case, 3 * groups)
    out = []
    for g in range(groups):
        m = m_range[0] + int(r[3 * g] % np.uint64(m_range[1] - m_range[0] + 1))
        out.append((m - m % 8, int(n_choices[int(r[3 * g + 1] % np.uint64(len(n_choices)))]),
                    int(k_choices[int(r[3 * g + 2] % np.uint64(len(k_choices)))])))
    return out


def make_addend(M: int, N: int, dist: str, case: int, dtype: str = "bf16"):
    """Seeded M x N addend matrix for beta * C: (array to upload, its FP64 values).
    dtype 'bf16' gives BF16 bit patterns (uint16), 'f32' FP32 values."""
    x = draw(dist, SEED_C + case, M * N).reshape(M, N)
    if dtype == "bf16":
        bits = bf16_bits(x)
        return bits, (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f32":
        x32 = x.astype(np.float32)
        return x32, x32.astype(np.float64)
    raise ValueError(dtype)


class GemmInputs:
    """Host-side input bundle: A (M x K), B (N x K), both K-contiguous."""

    def __init__(self, M, N, K, dtype, A, B, scales, bias):
        self.M, self.N, self.K, self.dtype = M, N, K, dtype
        self.A, self.B = A, B          # uint16 (BF16 bits) or uint8 (e4m3), shape (M,K) / (N,K)
        self.scales = scales           # float32[2] (sA, sB) or None
        self.bias = bias               # float32[N] or None


def make_gemm_inputs(M: int, N: int, K: int, dtype: str = "bf16", dist: str = "uniform",
                     case: int = 1, bias_dist: str | None = None, fp8_scaled: bool = True) -> GemmInputs:
    """Seeded inputs for one GEMM case.  dtype one of DTYPES.  With fp8_scaled=False the e4m3
    bytes encode the drawn values directly (no tensor-wise scale; scales is None)."""
    xa = draw(dist, SEED_A + case, M * K).reshape(M, K)
    xb = draw(dist, SEED_B + case, N * K).reshape(N, K)
    bias = None
    if bias_dist is not None:
        bias = draw(bias_dist, SEED_BIAS + case, N).astype(np.float32)
    if dtype == "bf16":
        return GemmInputs(M, N, K, dtype, bf16_bits(xa), bf16_bits(xb), None, bias)
    fa, fb = operand_types(dtype)
    enc = {"e4m3": (e4m3_bytes, e4m3_quantise), "e5m2": (e5m2_bytes, e5m2_quantise)}
    if not fp8_scaled:
        return GemmInputs(M, N, K, dtype, enc[fa][0](xa.astype(np.float32)), enc[fb][0](xb.astype(np.float32)),
                          None, bias)
    qa, sa = enc[fa][1](xa)
    qb, sb = enc[fb][1](xb)
    return GemmInputs(M, N, K, dtype, qa, qb, np.array([sa, sb], dtype=np.float32), bias)
