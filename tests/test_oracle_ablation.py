"""Pins of the ablation oracle: Philox4x32-10, stochastic rounding and the
random-sign Hadamard rotation (the approaches the AMD FP4 paper, §01, sets
against its deterministic rotation)."""

import os

import numpy as np
import pytest

from oracle import mx_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _kat():
    vals = {}
    with open(os.path.join(HERE, "golden", "philox4x32_10.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *ws = line.split()
                vals[k] = [int(w, 16) for w in ws]
    return vals


def test_philox_known_answer():
    kat = _kat()
    out = O.philox4x32_10(np.array([kat["ctr"]], np.uint32), np.array([kat["key"]], np.uint32))[0]
    assert [int(w) for w in out] == kat["out"]


def _round_inverse(y, k0, k1):
    """Inverse of one Philox4x32 round, derived from the round's algebra."""
    m0inv = pow(0xD2511F53, -1, 2 ** 32)
    m1inv = pow(0xCD9E8D57, -1, 2 ** 32)
    lo1, lo0 = y[1], y[3]
    c0 = (lo0 * m0inv) % 2 ** 32          # lo0 = M0 * c0 mod 2^32
    c2 = (lo1 * m1inv) % 2 ** 32
    hi0 = (0xD2511F53 * c0) >> 32
    hi1 = (0xCD9E8D57 * c2) >> 32
    c1 = y[0] ^ hi1 ^ k0
    c3 = y[2] ^ hi0 ^ k1
    return [c0, c1, c2, c3]


def test_philox_single_round_is_the_bijection_of_the_definition():
    # one round is philox4x32_10's first round: recover it from a 10-round
    # run with the key schedule rewound, via an independently derived inverse
    rng = np.random.default_rng(1)
    for _ in range(20):
        ctr = rng.integers(0, 2 ** 32, 4, dtype=np.uint64).astype(np.uint32)
        key = rng.integers(0, 2 ** 32, 2, dtype=np.uint64).astype(np.uint32)
        full = [int(w) for w in O.philox4x32_10(ctr[None], key[None])[0]]
        k0, k1 = int(key[0]), int(key[1])
        keys = []
        for r in range(10):
            keys.append((k0, k1))
            k0 = (k0 + 0x9E3779B9) % 2 ** 32
            k1 = (k1 + 0xBB67AE85) % 2 ** 32
        x = full
        for r in reversed(range(10)):
            x = _round_inverse(x, *keys[r])
        assert x == [int(w) for w in ctr]


def test_philox_uniform_and_balanced():
    idx = np.arange(1 << 20, dtype=np.uint64)
    r = O.element_random_bits(12345, idx)
    hist = np.bincount((r >> np.uint32(24)).astype(np.int64), minlength=256)
    expect = len(r) / 256
    chi2 = ((hist - expect) ** 2 / expect).sum()
    assert chi2 < 400           # 255 degrees of freedom; p ~ 1e-8 at 400
    bits = ((r[:, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 0.005)
    # different seeds and neighbouring indices give unrelated words
    r2 = O.element_random_bits(12346, idx[:4096])
    assert np.mean(r[:4096] == r2) < 0.01


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1, O.E5M2])
def test_stochastic_rounding_properties(fmt):
    rng = np.random.default_rng(2)
    top = O.fmt_params(fmt)["maxval"]
    v = rng.uniform(-top, top, 64)
    n = 4096
    r = ((np.arange(n) + 0.5) / n * 2 ** 32).astype(np.uint64)      # stratified bits
    sr = np.stack([O.stochastic_round_to_element(v, fmt, np.full(v.shape, ri)) for ri in r])
    lo = O.round_to_element(v, fmt)
    table = O.decode_table(fmt)
    grid = np.unique(np.abs(table[np.isfinite(table)]))
    assert np.all(np.isin(np.abs(sr), grid))                          # on the grid
    for j in range(len(v)):
        cand = np.unique(np.abs(sr[:, j]))
        assert len(cand) <= 2                                         # the two neighbours
        below = grid[grid <= abs(v[j])].max()
        above = grid[grid >= abs(v[j])].min()
        assert set(cand) <= {below, above}
        q = (above - below) if above > below else 0.0
        assert abs(np.abs(sr[:, j]).mean() - abs(v[j])) <= q / n + 1e-12   # unbiased
        assert np.all(np.diff(np.abs(sr[:, j])) <= 0)                 # rounds up for small r only
    assert np.all(np.signbit(sr) == np.signbit(v)[None, :])
    # grid values never move; beyond the top the result saturates
    assert np.array_equal(O.stochastic_round_to_element(grid, fmt, np.zeros(grid.shape)), grid)
    assert O.stochastic_round_to_element(np.array([top * 1.3]), fmt, np.array([0]))[0] == top


def test_ablation_reduces_to_the_deterministic_path():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 96)).astype(np.float32)
    for axis in ("row", "col"):
        for fmt in (O.E4M3, O.E2M1):
            a = O.mx_quantize_ablation(x, axis, fmt, True, 0, False, 0)
            b = O.hadamard_mx_quantize(x, axis, fmt)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
            a = O.mx_quantize_ablation(x, axis, fmt, False, 0, False, 0)
            b = O.mx_quantize(x, axis, fmt)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_random_sign_rotation_is_orthogonal_and_scale_free():
    rng = np.random.default_rng(4)
    mask = int(rng.integers(0, 2 ** 32))
    x = rng.standard_normal((50, 32))
    y = O.fwht32(O.apply_sign_mask(x, mask), np.float64)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    back = O.apply_sign_mask(O.fwht32(y, np.float64), mask)
    assert np.allclose(back, x, atol=1e-12)
    xf = rng.standard_normal((32, 64)).astype(np.float32)
    for stochastic in (False, True):
        c0, s0 = O.mx_quantize_ablation(xf, "col", O.E2M1, True, mask, stochastic, 7)
        c1, s1 = O.mx_quantize_ablation(xf * np.float32(8.0), "col", O.E2M1, True, mask, stochastic, 7)
        assert np.array_equal(c0, c1) and np.all(s1.astype(int) - s0.astype(int) == 3)


def test_stochastic_quantization_is_unbiased_on_average():
    # averaged over seeds, dequantized SR codes approach x; RNE does not
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((32, 64)) * 0.37).astype(np.float32)
    acc = np.zeros((32, 64))
    n = 64
    for seed in range(n):
        c, s = O.mx_quantize_ablation(x, "row", O.E2M1, False, 0, True, seed)
        acc += O.dequantize_f64(c, s, O.E2M1)
    bias_sr = np.abs(acc / n - x).mean()
    c, s = O.mx_quantize(x, "row", O.E2M1)
    bias_rne = np.abs(O.dequantize_f64(c, s, O.E2M1) - x).mean()
    assert bias_sr < 0.5 * bias_rne


def test_window_indices_match_the_full_tensor():
    # a window of a larger tensor draws the same bits as the full tensor
    rng = np.random.default_rng(6)
    x = rng.standard_normal((96, 128)).astype(np.float32)
    for axis in ("row", "col"):
        full = O.mx_quantize_ablation(x, axis, O.E4M3, True, 0x13579BDF, True, 99)
        if axis == "row":
            win = O.mx_quantize_ablation(x[32:64], axis, O.E4M3, True, 0x13579BDF, True, 99,
                                         first_row=32, total_cols=128)
            assert np.array_equal(win[0], full[0][32:64]) and np.array_equal(win[1], full[1][32:64])
        else:
            win = O.mx_quantize_ablation(x[:, 40:41], axis, O.E4M3, True, 0x13579BDF, True, 99,
                                         first_col=40, total_cols=128)
            assert np.array_equal(win[0], full[0][40:41]) and np.array_equal(win[1], full[1][40:41])


def test_error_structure_of_the_variants():
    # the contrast the AMD FP4 page (§01-§02) rests on, in the oracle at a
    # small Wgrad shape: on heavy-tailed tokens the fixed rotation lowers the
    # MXFP4 error of dY^T X; deterministic variants repeat the same error
    # every draw, stochastic rounding averages it away
    rng = np.random.default_rng(8)
    T, n_out, n_in = 512, 48, 40
    dy = (rng.standard_t(3, (T, n_out)) * 1e-3).astype(np.float32)
    x = rng.standard_t(3, (T, n_in)).astype(np.float32)
    ref = dy.astype(np.float64).T @ x.astype(np.float64)

    def err(had, mask, sr, seed):
        A, sA = O.mx_quantize_ablation(dy, "col", O.E2M1, had, mask, sr, seed)
        B, sB = O.mx_quantize_ablation(x, "col", O.E2M1, had, mask, sr, seed + 1)
        c, _ = O.mx_gemm_f64(A, sA, B, sB, O.E2M1)
        return c

    rel = lambda c: np.linalg.norm(c - ref) / np.linalg.norm(ref)
    plain = err(False, 0, False, 0)
    fixed = err(True, 0, False, 0)
    assert rel(fixed) < rel(plain)
    assert np.array_equal(err(True, 0, False, 5), fixed)        # deterministic
    draws = [err(True, 0, True, 100 + 2 * d) for d in range(8)]
    one, mean8 = rel(draws[0]), rel(np.mean(draws, axis=0))
    assert mean8 < 0.6 * one                                    # unbiased: averages down
