"""Pins of the oracle's random Hadamard transform (the NVFP4 recipe's RHT on
the weight-gradient GEMM inputs, "From BF16 to FP8/FP4 ...", sections 2.4
and 5.6): against scipy's Hadamard matrix, the exact matrix product within
the butterfly's rounding bound, its own inverse, the outlier-spreading
closed form, the GEMM identity it must preserve, and its composition with
the (separately pinned) columnwise NVFP4 copy."""
import numpy as np
import pytest

import oracle as O
import workloads as W

U = 2.0 ** -24


def sylvester16():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    return scipy_linalg.hadamard(16).astype(np.float64)


def signs(mask):
    return np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])


@pytest.mark.parametrize("mask", [0x0000, 0xFFFF, 0xA5C3, 0x0001, 0x8000])
def test_rht16_unit_vectors_give_scaled_hadamard_columns(mask):
    H = sylvester16()
    for j in range(16):
        e = np.zeros(16, np.float32)
        e[j] = 1.0
        got = O.rht16(e, mask).astype(np.float64)
        assert np.array_equal(got, H[:, j] * signs(mask)[j] / 4.0), j


@pytest.mark.parametrize("mask", [0x0000, 0x3C5A, 0xFFFF])
def test_rht16_within_the_butterfly_bound_of_the_exact_product(mask):
    """Each output is a depth-4 pairwise sum of the 16 signed inputs:
    |error| <= gamma_4 * sum|x| / 4 with gamma_4 = 4u / (1 - 4u)."""
    H = sylvester16()
    rng = np.random.default_rng(mask)
    g4 = 4 * U / (1 - 4 * U)
    worst = 0.0
    for _ in range(2000):
        v = (rng.standard_normal(16) * np.exp(rng.uniform(-20, 20, 16))).astype(np.float32)
        exact = H @ (signs(mask) * v.astype(np.float64)) / 4.0
        got = O.rht16(v, mask).astype(np.float64)
        bound = g4 * np.abs(v.astype(np.float64)).sum() / 4.0
        assert np.all(np.abs(got - exact) <= bound)
        worst = max(worst, float(np.max(np.abs(got - exact) / bound)))
    assert worst > 0.0          # the test does see rounding (it is not vacuous)


def test_rht16_is_its_own_inverse_without_signs_and_exact_on_small_integers():
    rng = np.random.default_rng(3)
    for _ in range(200):
        v = rng.integers(-1000, 1000, 16).astype(np.float32)
        once = O.rht16(v, 0)
        assert np.array_equal(O.rht16(once, 0), v)
    # with signs the inverse is D H / 4: undo the butterfly, then the signs
    v = rng.integers(-1000, 1000, 16).astype(np.float32)
    m = 0x9A63
    back = O.rht16(O.rht16(v, m), 0) * signs(m).astype(np.float32)
    assert np.array_equal(back, v)


@pytest.mark.parametrize("j,mask", [(0, 0), (7, 0x00F0), (15, 0xFFFF)])
def test_rht16_spreads_a_single_outlier_evenly(j, mask):
    """One outlier A among zeros becomes 16 values of magnitude A / 4: the
    block amax drops by 4x (the purpose of the transform)."""
    v = np.zeros(16, np.float32)
    v[j] = 1000.0
    got = O.rht16(v, mask)
    assert np.array_equal(np.abs(got), np.full(16, 250.0, np.float32))


def test_rht_cols_acts_on_16_row_groups_of_each_column():
    x = W.gen("outliers", (48, 24), 5, bf16=True)
    xf = W.bf16_bits_to_f32(x)
    xr = O.rht_cols(x, 0x5A5A)
    assert xr.shape == (48, 24) and xr.dtype == np.float32
    for g in range(3):
        for k in (0, 7, 23):
            assert np.array_equal(xr[16 * g:16 * g + 16, k], O.rht16(xf[16 * g:16 * g + 16, k], 0x5A5A))


def test_rht_preserves_the_wgrad_product():
    """(Q X)^T (Q Y) = X^T Y for the orthogonal Q = H D / 4 on each 16-row
    group: the transform leaves the weight-gradient GEMM unchanged (up to
    FP32 rounding of the transformed operands)."""
    X = W.gen("normal", (64, 8), 1, bf16=False)
    Y = W.gen("grad", (64, 12), 2, bf16=False)
    m = 0x1234
    lhs = O.rht_cols(X, m).astype(np.float64).T @ O.rht_cols(Y, m).astype(np.float64)
    rhs = X.astype(np.float64).T @ Y.astype(np.float64)
    scale = np.abs(X).astype(np.float64).T @ np.abs(Y).astype(np.float64)
    assert np.all(np.abs(lhs - rhs) <= 1e-6 * scale)


@pytest.mark.parametrize("rnd", [O.RN, O.SR])
def test_nvfp4_rht_colT_is_the_columnwise_copy_of_the_transform(rnd):
    x = W.gen("outliers", (64, 48), 9, bf16=True)
    m = 0xC3A5
    q, sb, a, sg = O.nvfp4_rht_colT(x, m, rnd, seed=11, offset=3)
    xr = O.rht_cols(x, m)
    ref = O.nvfp4(xr, O.B1x16, rnd, seed=11, offset=3, rowwise=False, colwise=True)
    assert np.array_equal(q, ref.q_colT) and np.array_equal(sb, ref.sb_colT)
    assert a == O.amax(xr) and sg == ref.s_global
    # with a given amax (sharded case) the tensor scale follows it
    q2, _, a2, sg2 = O.nvfp4_rht_colT(x, m, rnd, seed=11, offset=3, amax_in=2 * a)
    assert a2 == 2 * a and sg2 == O.nvfp4_global(2 * a)[1]


def test_rht_lowers_block_amax_on_outlier_blocks():
    """On blocks holding one large outlier the transform lowers the block
    maximum relative to the block RMS (which it preserves)."""
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((16 * 64, 1)) * 0.01).astype(np.float32)
    x[rng.integers(0, 16, 64) + 16 * np.arange(64), 0] = 10.0
    xr = O.rht_cols(x, 0xBEEF)
    b0 = np.abs(x.reshape(64, 16)).max(axis=1)
    b1 = np.abs(xr.reshape(64, 16)).max(axis=1)
    assert np.all(b1 < 0.3 * b0)


def test_rht_colT_sr_row_shards_draw_what_the_whole_tensor_draws():
    """Row bands on 16-row boundaries, each with the transformed tensor's
    global amax and counter offset offset + r0*K/16, give exactly the columns
    [r0/2, (r0 + h)/2) of the unsharded stochastic copy: the transform acts
    within 16-row groups and the draws depend on the position in x only."""
    x = W.gen("t3", (80, 48), 15, bf16=True)
    M, K = x.shape
    mask = 0x5A3C
    q, sb, A, _ = O.nvfp4_rht_colT(x, mask, O.SR, seed=17, offset=3)
    for r0, h in ((0, 16), (16, 48), (64, 16)):
        qb, sbb, _, _ = O.nvfp4_rht_colT(np.ascontiguousarray(x[r0:r0 + h]), mask, O.SR, seed=17,
                                         offset=3 + r0 * K // 16, amax_in=A)
        assert np.array_equal(qb, q[:, r0 // 2:(r0 + h) // 2])
        assert np.array_equal(sbb, sb[:, r0 // 16:(r0 + h) // 16])
