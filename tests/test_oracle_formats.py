"""Pins of the oracle's element formats, rounding and block quantization.

Each check ties the oracle to something other than itself: the OCP tables
typed into tests/golden, torch's independent float8_e4m3fn conversions,
brute-force nearest-code search, hand-derived blocks and algebraic
invariants of MX quantization.
"""

import math

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from tests.golden.fixtures import load_blocks, load_e2m1_packed, load_e2m1_values


def test_e4m3_decode_matches_torch_float8():
    # torch's float8_e4m3fn is an independent implementation of OCP FP8 E4M3.
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.decode_table(O.E4M3)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    # signed zeros too
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def test_e4m3_closed_forms():
    t = O.decode_table(O.E4M3)
    assert np.nanmax(t) == 448.0 == 1.75 * 2 ** 8
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9                      # smallest subnormal
    assert t[0x08] == 2.0 ** -6                      # smallest normal
    assert np.isnan(t).sum() == 2                    # only S.1111.111
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert (~np.isnan(t)).sum() == 254


def test_e2m1_table_matches_spec_golden():
    gold = load_e2m1_values()
    t = O.decode_table(O.E2M1)
    assert len(t) == 16
    for c, v in gold.items():
        assert t[c] == v and math.copysign(1, t[c]) == math.copysign(1, v), c
    assert O.fmt_params(O.E2M1)["maxval"] == t.max() == 6.0


def _brute_round(v, fmt):
    """Nearest finite code magnitude by exhaustive search; ties -> even code."""
    table = O.decode_table(fmt)
    n = len(table)
    pos = [(c, table[c]) for c in range(n // 2) if np.isfinite(table[c])]
    mags = np.array([m for _, m in pos])
    codes = np.array([c for c, _ in pos])
    out = np.empty(len(v))
    a = np.abs(v)
    for i, ai in enumerate(a):
        if ai >= mags.max():
            out[i] = mags.max()
            continue
        d = np.abs(mags - ai)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if codes[b] % 2 == 0]
        out[i] = mags[best[0]]
    return np.where(np.signbit(v), -out, out)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1, O.E5M2])
def test_rounding_brute_force(fmt):
    table = O.decode_table(fmt)
    mags = np.unique(np.abs(table[np.isfinite(table)]))
    mids = (mags[:-1] + mags[1:]) / 2
    f32 = np.float32
    cands = [mags, mids]
    for m in mids:  # one fp32 ulp either side of every midpoint
        cands.append(np.array([np.nextafter(f32(m), f32(0)), np.nextafter(f32(m), f32(np.inf))], dtype=np.float64))
    top = mags.max()
    cands.append(np.array([top * 1.01, top * 1.2, top * 1.99, 1e30]))
    # every positive bf16 bit pattern below 2*max
    bits = np.arange(0, 0x7F80, dtype=np.uint32) << 16
    bf = bits.view(np.float32).astype(np.float64)
    cands.append(bf[bf < 2 * top])
    v = np.concatenate(cands)
    v = np.concatenate([v, -v])
    got = O.round_to_element(v, fmt)
    exp = _brute_round(v, fmt)
    assert np.array_equal(got, exp)
    assert np.array_equal(np.signbit(got), np.signbit(exp))


def test_e4m3_rounding_matches_torch_cast():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even; compare codes
    # on |v| <= 448 (above that torch does not saturate).
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(200_000) * np.exp2(rng.integers(-12, 9, 200_000)),
        rng.uniform(-448, 448, 50_000),
    ]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = O.encode_element(O.round_to_element(v.astype(np.float64), O.E4M3), O.E4M3)
    assert np.array_equal(ours, ref)


def test_encode_decode_inverse():
    for fmt in (O.E4M3, O.E2M1, O.E5M2):
        t = O.decode_table(fmt)
        for c, val in enumerate(t):
            if not np.isfinite(val):
                continue
            assert O.encode_element(np.array([val]), fmt)[0] == c


@pytest.mark.parametrize("case", load_blocks(), ids=lambda c: c["name"])
def test_hand_derived_blocks(case):
    fmt = case["fmt"]
    x = np.array(case["x"], dtype=np.float32).reshape(1, 32)
    # every fixture input is exactly bf16
    xb = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(xb, x, equal_nan=True)
    codes, s = O.mx_quantize(x, "row", fmt)
    if fmt == O.E2M1:
        codes = O.unpack_e2m1(codes)
    assert int(s[0, 0]) == case["scale"]
    assert [int(c) for c in codes[0]] == case["codes"]


def test_e2m1_packed_bytes_hand_derived():
    # the packed bytes themselves, never unpacked: element 2j in the low
    # nibble (reading R5), on hand-derived blocks whose 16 bytes all differ
    # from their own nibble swap; row-wise one block per row, column-wise the
    # same blocks down the columns, stored transposed (R6)
    cases = load_e2m1_packed()
    x = np.array([c["x"] for c in cases], dtype=np.float32)            # [n, 32]
    xb = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(xb, x)                                        # exact bf16 inputs
    packed = np.array([c["packed"] for c in cases], dtype=np.uint8)     # [n, 16]
    scales = np.array([[c["scale"]] for c in cases], dtype=np.uint8)
    codes, s = O.mx_quantize(x, "row", O.E2M1)
    assert codes.dtype == np.uint8 and codes.shape == (len(cases), 16)
    np.testing.assert_array_equal(codes, packed)
    np.testing.assert_array_equal(s, scales)
    codes_c, s_c = O.mx_quantize(np.ascontiguousarray(x.T), "col", O.E2M1)
    np.testing.assert_array_equal(codes_c, packed)
    np.testing.assert_array_equal(s_c, scales)


def test_e2m1_golden_bytes_are_not_nibble_symmetric():
    # a nibble-swapped packing would fail the test above on every byte of
    # the first two blocks
    for c in load_e2m1_packed()[:2]:
        for b in c["packed"]:
            assert (b & 0xF) != (b >> 4)


def _representable_block(rng, fmt, R, C):
    """Blocks whose values are element values times 2**e, amax in the top binade."""
    table = O.decode_table(fmt)
    finite = table[np.isfinite(table)]
    vals = rng.choice(finite, size=(R, C))
    top = O.fmt_params(fmt)["maxval"]
    vals[:, ::32] = np.where(rng.random((R, C // 32)) < 0.5, top, -top)
    e = rng.integers(-40, 40, size=(R, C // 32))
    return (vals.reshape(R, C // 32, 32) * np.exp2(e)[..., None]).reshape(R, C)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1, O.E5M2])
def test_exact_round_trip(fmt):
    rng = np.random.default_rng(5)
    z = _representable_block(rng, fmt, 8, 256).astype(np.float32)
    for axis in ("row", "col"):
        # col: blocks run down the rows of z^T and come back transposed as z
        src = z if axis == "row" else np.ascontiguousarray(z.T)
        codes, s = O.mx_quantize(src, axis, fmt)
        back = O.mx_dequantize(codes, s, fmt)
        assert np.array_equal(back, z)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E2M1, O.E5M2])
@pytest.mark.parametrize("k", [-20, -3, 1, 7, 30])
def test_power_of_two_invariance(fmt, k):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((16, 128)) * 3).astype(np.float32)
    c0, s0 = O.mx_quantize(x, "row", fmt)
    c1, s1 = O.mx_quantize(x * np.float32(2.0 ** k), "row", fmt)
    assert np.array_equal(c0, c1)
    assert np.array_equal(s1.astype(int) - s0.astype(int), np.full(s0.shape, k))


def test_col_layout_is_transpose_of_row():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((64, 96)).astype(np.float32)
    for fmt in (O.E4M3, O.E2M1):
        cc, sc = O.mx_quantize(x, "col", fmt)
        cr, sr = O.mx_quantize(np.ascontiguousarray(x.T), "row", fmt)
        assert np.array_equal(cc, cr) and np.array_equal(sc, sr)
        assert cc.shape == ((96, 64) if fmt == O.E4M3 else (96, 32))
        assert sc.shape == (96, 2)


def test_dequant_bf16_and_nan_scale():
    codes = np.array([[0x38] * 32], dtype=np.uint8)      # 1.0 each
    s = np.array([[127 + 5]], dtype=np.uint8)
    assert np.all(O.mx_dequantize(codes, s, O.E4M3) == 32.0)
    s255 = np.array([[255]], dtype=np.uint8)
    assert np.all(np.isnan(O.mx_dequantize(codes, s255, O.E4M3)))
    # a value with 4 significant bits is exact in bf16
    codes2 = np.array([[0x39] * 32], dtype=np.uint8)     # 1.125
    assert np.all(O.mx_dequantize(codes2, s, O.E4M3, out="bf16") == 1.125 * 32)


def test_quantization_error_bound():
    # each element's error is at most half a grid step of its binade, or the
    # saturation loss; the relative block error stays below 2**-(mbits+1)
    # times the block's scale-normalised top value.
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 256)).astype(np.float32)
    for fmt in (O.E4M3, O.E2M1, O.E5M2):
        c, s = O.mx_quantize(x, "row", fmt)
        back = O.dequantize_f64(c, s, fmt)
        scale = np.exp2(s.astype(np.float64) - 127)
        err = np.abs(back - x).reshape(32, 8, 32) / scale[..., None]
        mb = O.fmt_params(fmt)["mbits"]
        top = O.fmt_params(fmt)["maxval"]
        # half a step of the top binade bounds every error once saturation is excluded
        bound = 2.0 ** (math.floor(math.log2(top)) - mb - 1)
        sat = (np.abs(x).reshape(32, 8, 32) / scale[..., None]) > top
        assert np.all(err[~sat] <= bound + 1e-12)


def test_e5m2_decode_matches_torch_float8():
    # torch's float8_e5m2 is an independent implementation of OCP FP8 E5M2
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    ours = O.decode_table(O.E5M2)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def test_e5m2_closed_forms():
    t = O.decode_table(O.E5M2)
    finite = t[np.isfinite(t)]
    assert finite.max() == 57344.0 == 1.75 * 2 ** 15 == t[0x7B]
    assert t[0x01] == 2.0 ** -16 and t[0x04] == 2.0 ** -14
    assert np.isinf(t[0x7C]) and np.isinf(t[0xFC]) and t[0xFC] < 0
    assert np.isnan(t).sum() == 6 and len(finite) == 248
    assert O.fmt_params(O.E5M2)["emax"] == 15


def test_e5m2_rounding_matches_torch_cast():
    rng = np.random.default_rng(13)
    v = np.concatenate([
        rng.standard_normal(200_000) * np.exp2(rng.integers(-20, 16, 200_000)),
        rng.uniform(-57344, 57344, 50_000),
    ]).astype(np.float32)
    v = v[np.abs(v) <= 57344]
    ref = torch.from_numpy(v).to(torch.float8_e5m2).view(torch.uint8).numpy()
    ours = O.encode_element(O.round_to_element(v.astype(np.float64), O.E5M2), O.E5M2)
    assert np.array_equal(ours, ref)
