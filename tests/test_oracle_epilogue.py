"""Pins for the extended-epilogue oracle (oracle/epilogue.py): library routines
for the activations and the FP8 cast, closed forms, a hand-worked example of
the whole order, and linearity identities that fail on a dropped or misplaced
term."""
import math
import os

import numpy as np
import torch

import oracle
import synthetic
from oracle import epilogue as E

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- activations

def test_gelu_vs_torch_and_closed_forms():
    x = np.concatenate([synthetic.normal(21, 4000) * 3.0, np.array([0.0, 1.0, -1.0, 8.0, -8.0, 40.0, -40.0])])
    g = E.gelu(x)
    # torch evaluates 0.5 x (1 + erf(x / sqrt 2)), which cancels in the left tail: compare
    # where that form is accurate, and everywhere against x * ndtr(x) (scipy's normal CDF)
    mid = np.abs(x) < 5
    ref = torch.nn.functional.gelu(torch.from_numpy(x)).numpy()
    assert np.allclose(g[mid], ref[mid], rtol=1e-14, atol=2e-15)
    special = __import__("pytest").importorskip("scipy.special")
    assert np.allclose(g, x * special.ndtr(x), rtol=1e-13, atol=1e-300)
    # Phi(1) from a normal table: 0.8413447460685429
    assert abs(E.gelu(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    # Phi(x) + Phi(-x) = 1  =>  gelu(x) - gelu(-x) = x
    assert np.allclose(E.gelu(x) - E.gelu(-x), x, rtol=1e-13, atol=1e-13)
    assert E.gelu(np.array([0.0]))[0] == 0.0


def test_silu_vs_torch_and_closed_forms():
    x = np.concatenate([synthetic.normal(22, 4000) * 5.0, np.array([0.0, 50.0, -50.0, 800.0, -800.0])])
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    s = E.silu(x)
    assert np.allclose(s, ref, rtol=1e-14, atol=1e-300)
    # sigmoid(ln 3) = 3/4
    assert abs(E.silu(np.array([math.log(3.0)]))[0] - 0.75 * math.log(3.0)) < 1e-15
    # sigmoid(x) + sigmoid(-x) = 1  =>  silu(x) - silu(-x) = x
    assert np.allclose(E.silu(x) - E.silu(-x), x, rtol=1e-13, atol=1e-13)
    assert E.silu(np.array([-800.0]))[0] == 0.0 and np.isfinite(s).all()


def test_lipschitz_constants_bound_the_slopes():
    x = np.linspace(-12, 12, 200001)
    for act in (E.ACT_GELU, E.ACT_SILU):
        y = E.activation(x, act)
        slope = np.abs(np.diff(y) / np.diff(x)).max()
        assert slope <= E.LIPSCHITZ[act] and slope > E.LIPSCHITZ[act] - 1e-3


def test_relu_and_identity():
    x = np.array([-2.0, -0.0, 0.0, 3.5])
    assert np.array_equal(E.activation(x, E.ACT_RELU), [0.0, 0.0, 0.0, 3.5])
    assert np.array_equal(E.activation(x, E.ACT_NONE), x)


# ---------------------------------------------------------------- FP8 output cast

def test_encode_e4m3_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.decode(codes, "e4m3")               # the C oracle's decode, not this module's
    assert np.array_equal(E.encode_e4m3(vals), codes)
    assert np.array_equal(E.decode_e4m3(codes), vals) or np.allclose(E.decode_e4m3(codes), vals)


def test_encode_e4m3_vs_torch_in_range():
    x = synthetic.normal(23, 20000) * np.exp(synthetic.uniform(24, 20000) * 6)
    x = x[np.abs(x) < 440.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(E.encode_e4m3(x), ref)


def test_encode_e4m3_ties_and_saturation_by_hand():
    # 1 + 1/16 is halfway between 1 (0x38) and 1.125 (0x39): even code 0x38
    # 1 + 3/16 is halfway between 1.125 (0x39) and 1.25 (0x3A): even code 0x3A
    # 2^-10 is halfway between 0 and the smallest subnormal 2^-9: 0
    # 3 * 2^-10 is halfway between 2^-9 (0x01) and 2^-8 (0x02): 0x02
    cases = [(1 + 1 / 16, 0x38), (1 + 3 / 16, 0x3A), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
             (-(1 + 1 / 16), 0xB8), (460.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (-0.0, 0x80)]
    for x, want in cases:
        assert E.encode_e4m3(np.array([x]))[0] == want, (x, want)


def test_encode_e4m3_saturation_matches_page():
    # the page's clamping rows (values above 448 clamp to +-448, sign kept)
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_facts.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and "=" not in line:
                rows.append(line.split())
    assert rows
    for _, x, want in rows:
        code = E.encode_e4m3(np.array([float(x)]))
        assert oracle.decode(code, "e4m3")[0] == float(want)


# ---------------------------------------------------------------- the order

def _acc(A_vals, B_vals):
    """Raw FP64 accumulator and sum |a||b| from the C oracle (alpha 1, nothing else)."""
    A = synthetic.bf16_bits(np.asarray(A_vals, dtype=np.float64))
    B = synthetic.bf16_bits(np.asarray(B_vals, dtype=np.float64))
    return oracle.gemm(A, B, "bf16")


def test_hand_worked_order_row_bias_relu_fp8():
    # acc = A B^T with B = I, so acc = A = [[1, 2], [3, 4]]
    acc, ad = _acc([[1, 2], [3, 4]], [[1, 0], [0, 1]])
    assert np.array_equal(acc, [[1, 2], [3, 4]])
    e = E.Epilogue(alpha=2.0, row_scale=np.array([1.0, 0.5]), col_scale=np.array([1.0, 2.0]),
                   beta=-1.0, c_in=np.array([[1.0, 1.0], [10.0, 0.0]]),
                   bias=np.array([0.5, -1.0]), bias_mode=E.BIAS_ROW, act=E.ACT_RELU, d_scale=0.5)
    Z, Y, D, bz = E.apply(acc, ad, e)
    # scale = 2 * [[1, 2], [0.5, 1]] -> alpha Acc = [[2, 8], [3, 8]]; - C -> [[1, 7], [-7, 8]];
    # + row bias [0.5, -1] -> [[1.5, 7.5], [-8, 7]]; ReLU -> [[1.5, 7.5], [0, 7]]; * 0.5
    assert np.array_equal(Z, [[1.5, 7.5], [-8.0, 7.0]])
    assert np.array_equal(Y, [[1.5, 7.5], [0.0, 7.0]])
    assert E.amax(Y) == 7.5
    assert np.array_equal(D, [[0.75, 3.75], [0.0, 3.5]])
    # 0.75 = 1.5 * 2^-1 (e 6, m 4), 3.75 = 1.875 * 2 (e 8, m 7), 3.5 = 1.75 * 2 (e 8, m 6)
    assert np.array_equal(E.encode_e4m3(D), [[0x34, 0x47], [0x00, 0x46]])
    assert np.array_equal(bz, [[2.0, 8.0], [3.0, 8.0]])


def test_hand_worked_column_bias_and_silu_order():
    acc, ad = _acc([[1, 2], [3, 4]], [[1, 0], [0, 1]])
    e = E.Epilogue(alpha=1.0, bias=np.array([0.5, -1.0]), bias_mode=E.BIAS_COL, act=E.ACT_SILU)
    Z, Y, _, _ = E.apply(acc, ad, e)
    assert np.array_equal(Z, [[1.5, 1.0], [3.5, 3.0]])        # bias per column
    assert np.allclose(Y, Z / (1 + np.exp(-Z)), rtol=1e-15)     # activation after the bias


def test_output_scale_follows_the_activation():
    # D = d * GELU(Z), not GELU(d * Z): at Z = 1 with d = 4 that is 4 Phi(1) = 3.3653789842741716
    acc, ad = _acc([[1]], [[1]])
    _, Y, D, _ = E.apply(acc, ad, E.Epilogue(act=E.ACT_GELU, d_scale=4.0))
    assert abs(D[0, 0] - 3.3653789842741716) < 1e-15 and abs(Y[0, 0] - 0.8413447460685429) < 1e-15


def test_beta_only_and_identity_defaults():
    A = synthetic.bf16_bits(synthetic.uniform(31, 6 * 40).reshape(6, 40))
    B = synthetic.bf16_bits(synthetic.uniform(32, 5 * 40).reshape(5, 40))
    acc, ad = oracle.gemm(A, B, "bf16")
    Z, Y, D, _ = E.apply(acc, ad, E.Epilogue())
    assert np.array_equal(Z, acc) and np.array_equal(D, acc)
    C = synthetic.uniform(33, 30).reshape(6, 5)
    Z, _, _, _ = E.apply(acc, ad, E.Epilogue(alpha=0.0, beta=1.5, c_in=C))
    assert np.array_equal(Z, 1.5 * C)


def test_vector_scales_equal_scaled_operands():
    """alpha * r_i * c_j * sum_k a_ik b_jk == sum_k (r_i a_ik)(c_j b_jk): with power-of-two
    scales and small integers every value is exact, so the two agree bit for bit."""
    M, N, K = 7, 9, 24
    a = np.round(synthetic.uniform(41, M * K) * 8).reshape(M, K)
    b = np.round(synthetic.uniform(42, N * K) * 8).reshape(N, K)
    r = 2.0 ** np.round(synthetic.uniform(43, M) * 3)
    c = 2.0 ** np.round(synthetic.uniform(44, N) * 3)
    acc, ad = _acc(a, b)
    Z, _, _, bz = E.apply(acc, ad, E.Epilogue(alpha=0.25, row_scale=r, col_scale=c))
    acc2, ad2 = _acc(a * r[:, None], b * c[:, None])
    assert np.array_equal(Z, 0.25 * acc2)
    assert np.array_equal(bz, 0.25 * ad2)


def test_tensor_scales_fold_like_the_basic_epilogue():
    A = synthetic.e4m3_bytes(synthetic.normal(51, 8 * 64).astype(np.float32).reshape(8, 64))
    B = synthetic.e4m3_bytes(synthetic.normal(52, 6 * 64).astype(np.float32).reshape(6, 64))
    bias = synthetic.normal(53, 6).astype(np.float32)
    z_basic, ad_basic = oracle.gemm(A, B, "e4m3", alpha=0.5, scales=(0.25, 2.0), bias=bias, relu=True)
    acc, ad = oracle.gemm(A, B, "e4m3")
    _, Y, _, bz = E.apply(acc, ad, E.Epilogue(alpha=0.5, scales=(0.25, 2.0), bias=bias,
                                              bias_mode=E.BIAS_COL, act=E.ACT_RELU))
    assert np.allclose(Y, z_basic, rtol=1e-15, atol=0) and np.allclose(bz, ad_basic, rtol=1e-15)


def test_rows_selection_matches_full():
    A = synthetic.bf16_bits(synthetic.uniform(61, 12 * 32).reshape(12, 32))
    B = synthetic.bf16_bits(synthetic.uniform(62, 5 * 32).reshape(5, 32))
    C = synthetic.uniform(63, 60).reshape(12, 5)
    r = synthetic.uniform(64, 12) + 2
    bias = synthetic.uniform(65, 12)
    e = E.Epilogue(alpha=1.5, beta=0.5, c_in=C, row_scale=r, bias=bias, bias_mode=E.BIAS_ROW, act=E.ACT_GELU)
    acc, ad = oracle.gemm(A, B, "bf16")
    full = E.apply(acc, ad, e)
    rows = np.array([11, 3, 0])
    acc_r, ad_r = oracle.gemm(A, B, "bf16", rows=rows)
    part = E.apply(acc_r, ad_r, e, rows=rows)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p)


def test_amax():
    assert E.amax(np.zeros((0, 4))) == 0.0
    assert E.amax(np.array([[-3.0, 2.0], [1.0, 0.5]])) == 3.0


# ------------------------------------------------- block scale factor generation

E_ = E   # the module (E names the tiles' exponents below)

def test_block_scales_hand_worked():
    # one 2 x 2 tile: amax 300 -> E = floor(log2 300) - 8 = 0, X = 1; 300 lies between
    # the e4m3 values 288 and 320 and rounds to 288; -1, 0.5 and 2 are exact
    codes, E = E_.block_scale_e4m3(np.array([[300.0, -1.0], [0.5, 2.0]]), block=(2, 2))
    assert E.tolist() == [[0]]
    assert E_.decode_e4m3(codes).tolist() == [[288.0, -1.0], [0.5, 2.0]]
    # amax 1000 -> E = 9 - 8 = 1, X = 2: 1000 / 2 = 500 saturates to 448; 3 / 2 = 1.5 exact
    codes, E = E_.block_scale_e4m3(np.array([[1000.0, 3.0]]), block=(1, 2))
    assert E.tolist() == [[1]] and E_.decode_e4m3(codes).tolist() == [[448.0, 1.5]]
    # tiny values: amax 0.01 -> floor(log2 0.01) = -7, E = -15, X = 2^-15; 0.01 * 2^15 = 327.68 -> 320
    codes, E = E_.block_scale_e4m3(np.array([[0.01]]), block=(1, 1))
    assert E.tolist() == [[-15]] and E_.decode_e4m3(codes).tolist() == [[320.0]]
    # an all-zero tile keeps X = 1 and zero codes
    codes, E = E_.block_scale_e4m3(np.zeros((3, 3)), block=(2, 2))
    assert (E == 0).all() and (codes == 0).all()


def test_block_scales_tiles_ragged_and_independent():
    rng = np.random.default_rng(5)
    Y = rng.normal(size=(70, 45)) * np.exp(rng.normal(size=(70, 45)) * 3)
    codes, E = E_.block_scale_e4m3(Y)
    assert E.shape == (3, 2) and codes.shape == Y.shape
    Yd = E_.decode_e4m3(codes)
    for i in range(3):
        for j in range(2):
            sl = (slice(32 * i, 32 * i + 32), slice(32 * j, 32 * j + 32))
            m = np.abs(Y[sl]).max()
            # the tile's largest magnitude lands in [256, 512) of the scaled range; none exceeds 448
            assert 256 <= m / 2.0 ** E[i, j] < 512
            assert np.abs(Yd[sl]).max() <= 448
            # reconstruction within half an e4m3 step (3 mantissa bits: 2^-4 relative), or the
            # saturation at 448 X, or the smallest subnormal step for tiny values
            X = 2.0 ** E[i, j]
            err = np.abs(Yd[sl] * X - Y[sl])
            tol = np.maximum(np.abs(Y[sl]) * 2.0 ** -4, 2.0 ** -10 * X)
            sat = np.abs(Y[sl]) >= 448 * X
            assert (err[~sat] <= tol[~sat]).all()
            assert (np.abs(Yd[sl][sat]) == 448).all()
    # changing one tile leaves the others' codes and scales alone
    Y2 = Y.copy()
    Y2[:32, :32] *= 1000.0
    codes2, E2 = E_.block_scale_e4m3(Y2)
    assert (E2[0, 0] == E[0, 0] + 9 or E2[0, 0] == E[0, 0] + 10)
    mask = np.ones(Y.shape, dtype=bool)
    mask[:32, :32] = False
    assert np.array_equal(codes2[mask], codes[mask]) and (E2.ravel()[1:] == E.ravel()[1:]).all()


def test_block_scales_follow_powers_of_two():
    rng = np.random.default_rng(6)
    Y = rng.normal(size=(40, 40))
    codes, E = E_.block_scale_e4m3(Y, block=(16, 16))
    for k in (-5, 3, 11):
        c2, e2 = E_.block_scale_e4m3(Y * 2.0 ** k, block=(16, 16))
        assert np.array_equal(c2, codes) and np.array_equal(e2, E + k)
