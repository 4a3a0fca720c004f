"""Pins for the oracle: facts that come from the page and from mathematics, not from the oracle.

Page: "INT8 Convrot Safetensors" (stable-diffusion.cpp docs).
  - H4 is the printed matrix / 2 ("How INT8 convrot works").
  - R_G is its normalized Kronecker power, block-diagonal over contiguous
    groups, orthogonal and symmetric ("How INT8 convrot works").
  - X_rot W_rot^T = X W^T before quantization ("How INT8 convrot works").
  - s = max|rot|/127, Q = clamp(round(rot/s), -127, 127) ("Weight
    quantization", "Runtime activation quantization").
  - A = sum Q_x Q_w in signed 32-bit; Y = A s_x s_w + b ("Runtime activation
    quantization").

Each mistake one could plausibly make in the oracle fails at least one test:
a wrong H4 entry (printed matrix, closed form, orthogonality), a wrong digit
stride or group offset in the fast transform (dense vs fast on several groups,
block-diagonal library build), max instead of max-abs (negative-max row),
the wrong rounding mode (rounding pin), a transposed GEMM operand (brute force
on non-square shapes), a wrong scale index or a dropped bias (error bound of Y
against the exact X W^T + b).
"""

import json
import os

import numpy as np
import pytest
import scipy.linalg

import oracle

GS = [4, 16, 64, 256, 1024]


def closed_form_R(G):
    """R_G[i, j] = 2^-n * (-1)^(#{digit positions p : i_p + j_p = 3}).

    Derivation: H4[a, b] = +-1/2 with a minus sign exactly where a + b = 3 (the
    anti-diagonal of the printed matrix), and an entry of a Kronecker power is
    the product of the factors' entries picked by the base-4 digits.
    """
    n = int(round(np.log(G) / np.log(4)))
    idx = np.arange(G)
    minus = np.zeros((G, G), np.int64)
    for p in range(n):
        di = (idx // 4**p) % 4
        minus += (di[:, None] + di[None, :]) == 3
    return np.where(minus % 2 == 1, -1.0, 1.0) / 2.0**n


def test_h4_is_the_printed_matrix(golden_dir):
    rows = [list(map(float, ln.split())) for ln in open(os.path.join(golden_dir, "h4_printed.txt"))
            if ln.strip() and not ln.startswith("#")]
    np.testing.assert_array_equal(oracle.h4(), np.array(rows) / 2.0)


def test_h4_regular_symmetric_orthogonal():
    H = oracle.h4()
    np.testing.assert_array_equal(H, H.T)
    np.testing.assert_allclose(H @ H.T, np.eye(4), rtol=0, atol=1e-15)
    # "regular" Hadamard: every row has the same sum (here 1)
    np.testing.assert_array_equal(H.sum(axis=1), np.ones(4))


@pytest.mark.parametrize("G", GS)
def test_rotation_matches_closed_form(G):
    np.testing.assert_array_equal(oracle.rotation_matrix(G), closed_form_R(G))


@pytest.mark.parametrize("G", GS)
def test_rotation_orthogonal_symmetric_involution(G):
    R = oracle.rotation_matrix(G)
    np.testing.assert_array_equal(R, R.T)
    np.testing.assert_allclose(R @ R.T, np.eye(G), rtol=0, atol=1e-12)
    np.testing.assert_allclose(R @ R, np.eye(G), rtol=0, atol=1e-12)
    np.testing.assert_allclose(R.sum(axis=1), np.ones(G), rtol=0, atol=1e-12)


@pytest.mark.parametrize("G", [1, 2, 3, 8, 12, 32, 128, 0, -4])
def test_rejects_non_power_of_four(G):
    assert oracle.log4(G) == -1
    with pytest.raises(ValueError):
        oracle.rotation_matrix(G) if G > 0 else oracle.rotate_fast(np.zeros((1, 4), np.float32), G)


def test_rejects_group_not_dividing_k():
    with pytest.raises(ValueError):
        oracle.pack_rows(np.zeros((2, 24), np.float32), 16)


@pytest.mark.parametrize("G", GS)
def test_fast_equals_dense_on_several_groups(G):
    rng = np.random.default_rng(G)
    k = 3 * G if G <= 256 else 2 * G
    X = rng.standard_normal((5, k)).astype(np.float32)
    X[:, 1] *= 50  # an outlier channel
    np.testing.assert_allclose(oracle.rotate_fast(X, G), oracle.rotate_dense(X, G),
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("G,k", [(4, 20), (16, 64), (64, 192)])
def test_rotation_is_block_diagonal_library_build(G, k):
    """X R with R = scipy block_diag of the closed-form R_G, one block per group."""
    rng = np.random.default_rng(k)
    X = rng.standard_normal((3, k)).astype(np.float32)
    R = scipy.linalg.block_diag(*([closed_form_R(G)] * (k // G)))
    np.testing.assert_allclose(oracle.rotate_fast(X, G), X.astype(np.float64) @ R,
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("G", [4096, 16384, 65536])
def test_rotation_large_g_one_hot_rows(G):
    """For G = 4096 and up (dense R too big to test wholesale): rotating e_j gives
    row j of R, the closed form read off the printed H4's sign pattern."""
    n = int(round(np.log(G) / np.log(4)))
    js = [0, 1, 3, G - 1, 1234, G // 2 + 77]
    X = np.zeros((len(js), G), np.float32)
    for r, j in enumerate(js):
        X[r, j] = 1.0
    rot = oracle.rotate_fast(X, G)
    idx = np.arange(G)
    for r, j in enumerate(js):
        minus = np.zeros(G, np.int64)
        for p in range(n):
            minus += ((idx // 4**p) % 4 + (j // 4**p) % 4) == 3
        np.testing.assert_array_equal(rot[r], np.where(minus % 2, -1.0, 1.0) / 2.0**n)


@pytest.mark.parametrize("G", [16384, 65536])
def test_rotation_large_g_is_an_involution(G):
    """R_G is symmetric and orthogonal, so rotating twice gives the input back."""
    rng = np.random.default_rng(G)
    X = rng.standard_normal((2, 2 * G)).astype(np.float32)
    twice = oracle.rotate_fast(oracle.rotate_fast(X, G).astype(np.float32), G)
    np.testing.assert_allclose(twice, X.astype(np.float64), rtol=0, atol=1e-5)


@pytest.mark.parametrize("G", [4, 64, 256])
def test_rotation_identity_preserves_linear(G):
    """X_rot W_rot^T == X W^T in fp64 (no quantization)."""
    rng = np.random.default_rng(7)
    k = 2 * G if G < 256 else 512
    X = rng.standard_normal((6, k)).astype(np.float32)
    W = (0.02 * rng.standard_normal((9, k))).astype(np.float32)
    lhs = oracle.rotate_fast(X, G) @ oracle.rotate_fast(W, G).T
    rhs = X.astype(np.float64) @ W.astype(np.float64).T
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * np.max(np.abs(rhs))


def _hand():
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    return json.load(open(os.path.join(here, "hand_worked_rows.json")))


@pytest.mark.parametrize("case", _hand()["rows"], ids=lambda c: c["why"][:40])
def test_hand_worked_rows(case):
    x = np.array([case["x"]], np.float32)
    rot = oracle.rotate_fast(x, case["G"])
    np.testing.assert_array_equal(rot[0], np.array(case["x_rot"], np.float64))
    np.testing.assert_array_equal(oracle.rotate_dense(x, case["G"])[0], rot[0])
    Q, s, v = oracle.pack_rows(x, case["G"])
    num, den = case["scale_over"]
    assert s[0] == np.float32(num / den)
    np.testing.assert_array_equal(Q[0], np.array(case["Q"], np.int8))


def test_worked_linear():
    c = _hand()["linear"]
    x = np.array([c["x"]], np.float32)
    w = np.array([c["w"]], np.float32)
    out = oracle.linear(x, w, np.array([c["b"]], np.float32), c["G"])
    assert int(out["A"][0, 0]) == c["A"]
    assert abs(float(out["Y64"][0, 0]) - c["Y"]) <= c["Y_tol"]
    # the reconstruction approximates the exact x.w + b
    assert abs(float(out["Y64"][0, 0]) - (c["exact_xw"] + c["b"])) < 0.2


def test_quantize_properties():
    rng = np.random.default_rng(11)
    rot = rng.standard_normal((50, 256)) * rng.uniform(0.01, 100, size=(50, 1))
    rot[3] = 0.0
    Q, s, v = oracle.quantize_rows(rot, ldq=384)
    assert Q.shape == (50, 384) and np.all(Q[:, 256:] == 0)
    assert np.all(np.abs(Q) <= 127)
    nz = np.arange(50) != 3
    assert np.all(np.abs(Q[nz, :256]).max(axis=1) == 127)  # the max code is reached
    assert s[3] == 0 and np.all(Q[3] == 0)
    # scale is max|rot|/127 rounded to fp32
    np.testing.assert_array_equal(s[nz], (np.abs(rot[nz]).max(axis=1) / 127).astype(np.float32))
    # codes are within half a step of the pre-round value, and |Q s - rot| <= s/2 (+ fp32 scale rounding)
    assert np.all(np.abs(Q[:, :256] - v) <= 0.5)
    err = np.abs(Q[:, :256] * s[:, None].astype(np.float64) - rot)
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-6) + 1e-7 * np.abs(rot))
    # sign is kept wherever the code is non-zero
    assert np.all(np.sign(Q[:, :256])[Q[:, :256] != 0] == np.sign(rot)[Q[:, :256] != 0])


def test_half_away_not_half_even():
    rot = np.array([[254.0, 0.5, -0.5, 2.5, -2.5, 1.5, -1.5, 0.49999999]])
    Q, s, _ = oracle.quantize_rows(rot)
    assert s[0] == 2.0
    np.testing.assert_array_equal(Q[0], [127, 0, 0, 1, -1, 1, -1, 0])
    rot2 = rot * 2  # now v = rot2 / 4 = rot / 2 again with s = 4
    Q2, s2, _ = oracle.quantize_rows(rot2)
    np.testing.assert_array_equal(Q2[0], Q[0])


def test_gemm_brute_force_non_square():
    rng = np.random.default_rng(3)
    m, n, k = 5, 7, 13
    Qx = rng.integers(-127, 128, size=(m, k + 3), dtype=np.int8)
    Qw = rng.integers(-127, 128, size=(n, k + 5), dtype=np.int8)
    A = oracle.gemm_i32(Qx, Qw, k)
    for r in range(m):
        for o in range(n):
            assert A[r, o] == sum(int(Qx[r, i]) * int(Qw[o, i]) for i in range(k))
    np.testing.assert_array_equal(A, Qx[:, :k].astype(np.int64) @ Qw[:, :k].astype(np.int64).T)


def test_gemm_saturation_and_int32_range():
    k = 12288
    Qx = np.full((2, k), 127, np.int8)
    Qx[1] = -127
    Qw = np.full((3, k), 127, np.int8)
    Qw[1, ::2] = -127  # alternating signs cancel exactly
    Qw[2] = -127
    A = oracle.gemm_i32(Qx, Qw, k)
    np.testing.assert_array_equal(A, [[16129 * k, 0, -16129 * k], [-16129 * k, 0, 16129 * k]])
    assert oracle.gemm_i32(np.full((1, 133144), 127, np.int8),
                           np.full((1, 133144), 127, np.int8), 133144)[0, 0] == 2147479576
    with pytest.raises(OverflowError):
        oracle.gemm_i32(np.full((1, 133145), 127, np.int8), np.full((1, 133145), 127, np.int8),
                        133145)


@pytest.mark.parametrize("G", [4, 16, 256])
def test_linear_within_quantization_error_bound(G):
    """|Y - (X W^T + b)| is bounded by the rounding of both operands.

    With xr = X R, wr = W R, dx = s_x/2, dw = s_w/2 (|Q s - rot| <= s/2):
      |Qx sx . Qw sw - xr . wr| <= sum_i |xr_i| dw + |wr_i| dx + dx dw,
    and xr . wr = x . w exactly (R orthogonal). A wrong scale index, a
    transposed operand or a dropped bias breaks this bound.
    """
    rng = np.random.default_rng(G + 100)
    m, n, k = 7, 5, 2 * max(G, 64)
    X = rng.standard_normal((m, k)).astype(np.float32)
    X[:, 3] *= 50
    X[2] *= 20  # rows with very different scales
    W = (0.02 * rng.standard_normal((n, k))).astype(np.float32)
    W[1] *= 30
    b = rng.standard_normal(n).astype(np.float32)
    out = oracle.linear(X, W, b, G)
    exact = X.astype(np.float64) @ W.astype(np.float64).T + b
    xr, wr = oracle.rotate_fast(X, G), oracle.rotate_fast(W, G)
    dx, dw = out["sx"].astype(np.float64) / 2, out["sw"].astype(np.float64) / 2
    bound = (np.abs(xr).sum(1)[:, None] * dw[None, :] + dx[:, None] * np.abs(wr).sum(1)[None, :]
             + k * dx[:, None] * dw[None, :])
    err = np.abs(out["Y64"] - exact)
    assert np.all(err <= bound * (1 + 1e-6) + 1e-9)
    # the bound has teeth: a dropped bias or scales taken from the wrong row break it
    assert np.any(np.abs(out["Y64"] - b - exact) > bound)
    wrong_row = out["A"] * out["sx"][::-1, None].astype(np.float64) * out["sw"][None, :] + b
    assert np.any(np.abs(wrong_row - exact) > bound)


def test_pack_rows_zero_pads_and_composes():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((4, 64)).astype(np.float32)
    Q, s, v = oracle.pack_rows(X, 16, ldq=128)
    assert Q.shape == (4, 128) and np.all(Q[:, 64:] == 0)
    Q2, s2, v2 = oracle.quantize_rows(oracle.rotate_dense(X, 16))
    np.testing.assert_array_equal(Q[:, :64], Q2)
    np.testing.assert_array_equal(s, s2)


def test_strided_input_rows():
    rng = np.random.default_rng(9)
    big = rng.standard_normal((3, 100)).astype(np.float32)
    X = big[:, :64]  # leading dimension 100
    np.testing.assert_array_equal(oracle.rotate_fast(X, 16),
                                  oracle.rotate_fast(np.ascontiguousarray(X), 16))


# ---- GELU after the up projection (the DiT MLP; not part of the page's linear)

def test_gelu_odd_part_is_identity():
    """GELU(x) - GELU(-x) = x for both forms: x Phi(x) + x Phi(-x) = x, and the
    tanh form keeps the same symmetry (tanh is odd)."""
    x = np.linspace(-8, 8, 1601)
    for act in (1, 2):
        d = oracle.activation(x, act) - oracle.activation(-x, act)
        np.testing.assert_allclose(d, x, rtol=0, atol=1e-14)


def test_gelu_erf_matches_normal_table():
    """GELU(x) = x Phi(x): Phi(1) = 0.84134, Phi(2) = 0.97725, Phi(0.5) = 0.69146
    (standard normal table, five places)."""
    x = np.array([1.0, 2.0, 0.5, -1.0])
    phi = np.array([0.84134, 0.97725, 0.69146, 1 - 0.84134])
    np.testing.assert_allclose(oracle.activation(x, 1), x * phi, rtol=0, atol=1e-5 * 2)


def test_gelu_limits_and_slope_at_zero():
    for act in (1, 2):
        g = oracle.activation(np.array([0.0, 30.0, -30.0, 1e-6]), act)
        assert g[0] == 0.0 and abs(g[1] - 30.0) < 1e-12 and abs(g[2]) < 1e-12
        assert abs(g[3] / 1e-6 - 0.5) < 1e-6  # GELU'(0) = Phi(0) = 1/2


def test_gelu_tanh_form_approximates_erf_form():
    x = np.linspace(-6, 6, 2401)
    err = np.abs(oracle.activation(x, 2) - oracle.activation(x, 1))
    assert err.max() < 1e-3 and err.max() > 1e-6  # close, and not the same function


def test_linear_with_activation_is_activation_of_linear():
    rng = np.random.default_rng(41)
    X = rng.standard_normal((5, 64)).astype(np.float32)
    W = (0.1 * rng.standard_normal((7, 64))).astype(np.float32)
    b = rng.standard_normal(7).astype(np.float32)
    base = oracle.linear(X, W, b, 16)
    for act in (1, 2):
        got = oracle.linear(X, W, b, 16, act=act)
        np.testing.assert_array_equal(got["A"], base["A"])
        np.testing.assert_allclose(got["Y64"], oracle.activation(base["Y64"], act), rtol=0, atol=0)


# ---- runtime LoRA correction (page: "Backend support", paragraph on adapters)

def test_lora_delta_rank_one_by_hand():
    """A = e_i (one row), B = e_j (one column): the correction is scale * X[:, i] in column j."""
    rng = np.random.default_rng(51)
    X = rng.standard_normal((6, 20)).astype(np.float32)
    A = np.zeros((1, 20), np.float32)
    A[0, 7] = 1.0
    B = np.zeros((5, 1), np.float32)
    B[3, 0] = 1.0
    T, D = oracle.lora_delta(X, A, B, 2.5)
    np.testing.assert_array_equal(T[:, 0], X[:, 7].astype(np.float64))
    expect = np.zeros((6, 5))
    expect[:, 3] = 2.5 * X[:, 7].astype(np.float64)
    np.testing.assert_array_equal(D, expect)


def test_lora_delta_is_the_merged_weight_update():
    """(X A^T) B^T = X (B A)^T: the correction equals what merging s B A into W
    would add, computed here in the other association order."""
    rng = np.random.default_rng(52)
    X = rng.standard_normal((9, 64)).astype(np.float32)
    A = rng.standard_normal((16, 64)).astype(np.float32)
    B = rng.standard_normal((11, 16)).astype(np.float32)
    _, D = oracle.lora_delta(X, A, B, 0.75)
    merged = X.astype(np.float64) @ (0.75 * (B.astype(np.float64) @ A.astype(np.float64))).T
    np.testing.assert_allclose(D, merged, rtol=1e-12, atol=1e-12)


def test_lora_correction_enters_before_the_activation():
    rng = np.random.default_rng(53)
    A_int = rng.integers(-1000, 1000, size=(4, 6)).astype(np.int32)
    sx = rng.uniform(0.01, 0.1, 4).astype(np.float32)
    sw = rng.uniform(0.01, 0.1, 6).astype(np.float32)
    add = rng.standard_normal((4, 6))
    _, plain = oracle.reconstruct(A_int, sx, sw, None)
    _, with_add = oracle.reconstruct(A_int, sx, sw, None, act=1, add=add)
    np.testing.assert_allclose(with_add, oracle.activation(plain + add, 1), rtol=0, atol=0)
