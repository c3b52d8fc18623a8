"""Pins of the oracle's fixed Hadamard rotation and its block-scaled GEMM.

The rotation is checked against an independently built Sylvester matrix
(popcount signs), exact integer products, its own inverse and the
orthogonality that makes it free inside the Wgrad product.  The GEMM is
checked against exact integer matmuls, scaling laws and symmetry.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import mx_oracle as O


def test_scale_constant_is_nearest_fp32_to_2_pow_minus_2_5():
    c = O.fwht_scale(np.float32)
    assert c.dtype == np.float32
    lo = np.nextafter(c, np.float32(0))
    hi = np.nextafter(c, np.float32(1))
    # midpoints to the neighbours bracket 2**-2.5, i.e. mid_lo**2 < 1/32 < mid_hi**2
    m_lo = (Fraction(float(lo)) + Fraction(float(c))) / 2
    m_hi = (Fraction(float(hi)) + Fraction(float(c))) / 2
    assert m_lo * m_lo < Fraction(1, 32) < m_hi * m_hi


def test_transform_of_basis_is_normalized_sylvester_matrix():
    # fwht32 of e_j is column j of H/sqrt(32), H[i,j] = (-1)**popcount(i&j)
    H = O.hadamard_matrix(32)
    eye = np.eye(32)
    cols = O.fwht32(eye, np.float64)          # row j = transform of e_j
    assert np.allclose(cols.T, H / np.sqrt(32), atol=1e-15, rtol=0)
    Hn = H / np.sqrt(32.0)
    assert np.allclose(Hn @ Hn.T, np.eye(32), atol=1e-6)
    assert np.array_equal(H @ H.T, 32 * np.eye(32, dtype=np.int64))


def test_integer_inputs_exact_against_dense_product():
    # all stage sums stay below 2**24, so the fp32 butterflies are exact; only
    # the final multiply by c rounds, once.
    rng = np.random.default_rng(1)
    x = rng.integers(-(2 ** 18), 2 ** 18, size=(64, 32))
    H = O.hadamard_matrix(32)
    exact = x @ H.T                                       # int64
    got = O.fwht32(x.astype(np.float32), np.float32)
    expect = exact.astype(np.float32) * O.fwht_scale(np.float32)
    assert np.array_equal(got, expect)


def test_fp64_transform_is_an_involution():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((100, 32))
    back = O.fwht32(O.fwht32(x, np.float64), np.float64)
    assert np.allclose(back, x, atol=1e-12, rtol=0)


def test_fp32_butterfly_order_is_fixed():
    # the oracle's fp32 result equals a scalar, loop-by-loop restatement of
    # the five stages on a few blocks: a transposed index or a reversed stage
    # order changes the rounding and fails this bitwise check
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((8, 32)) * 1e3).astype(np.float32)
    got = O.fwht32(x, np.float32)
    for r in range(8):
        a = [np.float32(v) for v in x[r]]
        h = 1
        while h < 32:
            for j in range(32):
                if j & h == 0:
                    u, w = a[j], a[j + h]
                    a[j], a[j + h] = np.float32(u + w), np.float32(u - w)
            h *= 2
        ref = np.array(a, dtype=np.float32) * np.float32(O.fwht_scale(np.float32))
        assert np.array_equal(got[r], ref)


def test_reversed_stage_order_would_differ():
    # guard for the previous test: the two orders do give different bits
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((256, 32)) * 1e3).astype(np.float32)
    a = x.copy()
    for h in (16, 8, 4, 2, 1):
        a = a.reshape(256, 32 // (2 * h), 2, h)
        lo, hi = a[..., 0, :], a[..., 1, :]
        a = np.stack([lo + hi, lo - hi], axis=-2).reshape(256, 32)
    rev = a * O.fwht_scale(np.float32)
    assert not np.array_equal(rev, O.fwht32(x, np.float32))
    assert np.allclose(rev, O.fwht32(x, np.float32), rtol=1e-5, atol=1e-2)


def test_wgrad_identity_fp64():
    # (H dY)^T (H X) = dY^T X when H acts blockwise along the token axis:
    # the rotation costs nothing in exact arithmetic
    rng = np.random.default_rng(5)
    T, n_out, n_in = 128, 48, 40
    dY = rng.standard_normal((T, n_out))
    X = rng.standard_normal((T, n_in))
    HdY = O.hadamard_rotate(dY, "col", np.float64)
    HX = O.hadamard_rotate(X, "col", np.float64)
    lhs = HdY.T @ HX
    rhs = dY.T @ X
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * np.max(np.abs(rhs)) * T


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1])
@pytest.mark.parametrize("k", [-5, 4])
def test_hadamard_quantize_power_of_two_invariance(fmt, k):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 64)).astype(np.float32)
    for axis in ("row", "col"):
        c0, s0 = O.hadamard_mx_quantize(x, axis, fmt)
        c1, s1 = O.hadamard_mx_quantize(x * np.float32(2.0 ** k), axis, fmt)
        assert np.array_equal(c0, c1)
        assert np.all(s1.astype(int) - s0.astype(int) == k)


def test_hadamard_quantize_is_rotate_then_quantize():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 96)).astype(np.float32)
    y = O.hadamard_rotate(x, "col", np.float32)
    c0, s0 = O.hadamard_mx_quantize(x, "col", O.E2M1)
    c1, s1 = O.mx_quantize(y, "col", O.E2M1)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


def test_largest_finite_rotated_block_reaches_the_scale_bound():
    """The largest finite bf16 alone in a block gives the largest finite
    rotated amax: every butterfly output is +-x, and RN(x * c) < 2^125.5, so
    the scale byte is 125 - emax + 127 (250 for E2M1), the upper bound the
    kernels' single multiplier c * 2^(127-s) relies on.  Two such inputs
    overflow a butterfly sum: scale 255 and zero codes."""
    bmax = np.frombuffer(np.uint32(0x7F7F0000).tobytes(), np.float32)[0]
    x = np.zeros((2, 32), np.float32)
    x[0, 5] = bmax
    x[1, 3] = -bmax
    for fmt, emax in ((O.E2M1, 2), (O.E4M3, 8), (O.E5M2, 15)):
        codes, s = O.hadamard_mx_quantize(x, "row", fmt)
        assert s[0, 0] == 125 - emax + 127 and s[1, 0] == s[0, 0]
        vals = O.mx_dequantize(codes, s, fmt)
        # every rotated value is +-RN(|x| * c); scaled by 2^(127 - s) it is
        # 1.9921875 * 2^(emax + 0.5), which each format rounds onto its grid
        y = np.float32(np.float64(bmax) * np.float64(O.fwht_scale()))
        q = O.round_to_element(np.float64(y) / 2.0 ** (125 - emax), fmt)
        assert np.all(np.abs(vals) == np.float32(abs(float(q)) * 2.0 ** (125 - emax)))
    y = x.copy()
    y[0, 9] = bmax
    codes, s = O.hadamard_mx_quantize(y[:1], "row", O.E2M1)
    assert s[0, 0] == 255 and not np.any(codes)


def _int_codes(rng, fmt, shape, lim):
    """Codes whose element values are small integers in [-lim, lim]."""
    table = O.decode_table(fmt)
    ints = [c for c, v in enumerate(table) if np.isfinite(v) and v == int(v) and abs(v) <= lim]
    c = rng.choice(ints, size=shape).astype(np.uint8)
    return O.pack_e2m1(c) if fmt == O.E2M1 else c


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1])
def test_gemm_equals_integer_matmul(fmt):
    rng = np.random.default_rng(8)
    M, N, K = 40, 24, 128
    A = _int_codes(rng, fmt, (M, K), 16)
    B = _int_codes(rng, fmt, (N, K), 16)
    sA = np.full((M, K // 32), 127, np.uint8)
    sB = np.full((N, K // 32), 127, np.uint8)
    C, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
    table = O.decode_table(fmt)
    ua = O.unpack_e2m1(A) if fmt == O.E2M1 else A
    ub = O.unpack_e2m1(B) if fmt == O.E2M1 else B
    ia = table[ua].astype(np.int64)
    ib = table[ub].astype(np.int64)
    assert np.array_equal(C, (ia @ ib.T).astype(np.float64))
    assert np.array_equal(S, (np.abs(ia) @ np.abs(ib).T).astype(np.float64))


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1])
def test_gemm_scale_laws_and_symmetry(fmt):
    rng = np.random.default_rng(9)
    M, N, K = 16, 20, 96
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32)
    A, sA = O.mx_quantize(x, "row", fmt)
    B, sB = O.mx_quantize(w, "row", fmt)
    C, _ = O.mx_gemm_f64(A, sA, B, sB, fmt)
    Ct, _ = O.mx_gemm_f64(B, sB, A, sA, fmt)
    assert np.array_equal(C, Ct.T)
    # raising every A scale by 3 multiplies C by 8 exactly
    C8, _ = O.mx_gemm_f64(A, sA + 3, B, sB, fmt)
    assert np.array_equal(C8, 8 * C)
    # raising one k-block's scale of one row changes only that row
    sA2 = sA.copy()
    sA2[5, 1] += 1
    C2, _ = O.mx_gemm_f64(A, sA2, B, sB, fmt)
    assert np.array_equal(np.delete(C2, 5, 0), np.delete(C, 5, 0))
    assert not np.array_equal(C2[5], C[5])


def test_gemm_rows_sampler_matches_full():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    w = rng.standard_normal((48, 128)).astype(np.float32)
    for fmt in (O.E4M3, O.E2M1):
        A, sA = O.mx_quantize(x, "row", fmt)
        B, sB = O.mx_quantize(w, "row", fmt)
        C, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
        rows = np.array([0, 7, 63])
        cols = np.array([47, 3])
        Cs, Ss = O.mx_gemm_f64_rows(A, sA, B, sB, fmt, rows, cols)
        assert np.array_equal(Cs, C[np.ix_(rows, cols)])
        assert np.array_equal(Ss, S[np.ix_(rows, cols)])


def test_rotation_lowers_wgrad_error_on_outlier_columns():
    # quality check of the method, not parity: with heavy-tailed tokens the
    # rotated MXFP4 Wgrad is closer to the exact dY^T X than the unrotated one
    rng = np.random.default_rng(12)
    T, n_out, n_in = 256, 64, 64
    dY = rng.standard_normal((T, n_out)) * np.exp(rng.standard_normal(n_out) * 2)[None, :] * 1e-3
    X = rng.standard_t(3, size=(T, n_in))
    dY = dY.astype(np.float32)
    X = X.astype(np.float32)
    exact = dY.astype(np.float64).T @ X.astype(np.float64)
    A0, sA0 = O.mx_quantize(dY, "col", O.E2M1)
    B0, sB0 = O.mx_quantize(X, "col", O.E2M1)
    A1, sA1 = O.hadamard_mx_quantize(dY, "col", O.E2M1)
    B1, sB1 = O.hadamard_mx_quantize(X, "col", O.E2M1)
    plain, _ = O.mx_gemm_f64(A0, sA0, B0, sB0, O.E2M1)
    rot, _ = O.mx_gemm_f64(A1, sA1, B1, sB1, O.E2M1)
    err0 = np.linalg.norm(plain - exact) / np.linalg.norm(exact)
    err1 = np.linalg.norm(rot - exact) / np.linalg.norm(exact)
    assert err1 < err0


@pytest.mark.parametrize("fmt,tdt", [("e4m3", "float8_e4m3fn"), ("e5m2", "float8_e5m2")])
def test_gemm_oracle_against_torch_fp8_decoding(fmt, tdt):
    # an independent decode: torch's own fp8 dtypes read the code bytes, the
    # block scales are applied as powers of two and a float64 matmul sums
    import torch
    rng = np.random.default_rng(17)
    M, N, K = 24, 40, 96
    table = O.decode_table(fmt)
    finite = np.flatnonzero(np.isfinite(table)).astype(np.uint8)
    A = rng.choice(finite, size=(M, K))
    B = rng.choice(finite, size=(N, K))
    sA = rng.integers(110, 140, size=(M, K // 32)).astype(np.uint8)
    sB = rng.integers(110, 140, size=(N, K // 32)).astype(np.uint8)
    ref, _ = O.mx_gemm_f64(A, sA, B, sB, fmt)
    dt = getattr(torch, tdt)
    a = torch.from_numpy(A).view(dt).to(torch.float64).numpy()
    b = torch.from_numpy(B).view(dt).to(torch.float64).numpy()
    a = a * np.exp2(np.repeat(sA.astype(np.float64) - 127, 32, axis=1))
    b = b * np.exp2(np.repeat(sB.astype(np.float64) - 127, 32, axis=1))
    np.testing.assert_array_equal(ref, a @ b.T)
