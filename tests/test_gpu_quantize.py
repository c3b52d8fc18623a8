"""Parity of the CUDA quantizers and dequantizer with the CPU oracle.

Codes and scales must match bit for bit (the butterfly order and the
rounding are fixed), on tiny shapes, ragged tiles and the full-size
workloads, including the degenerate blocks (zeros, NaN, Inf, subnormal and
huge maxima).
"""

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq, synth
from tests.golden.fixtures import load_blocks, load_e2m1_packed
from tests.libutil import bf16_to_f32_np, ensure_built, to_np

pytestmark = pytest.mark.gpu

FMTS = ["e4m3", "e2m1", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _x(rows, cols, seed=0, kind="act"):
    if kind == "act":
        return synth.activation(rows, cols, seed).cuda()
    return synth.normal_with_outliers((rows, cols), seed).cuda()


def _check(x, axis, fmt, had):
    xn = bf16_to_f32_np(x)
    if had:
        codes, scales = mxq.hadamard_mx_quantize(x, axis, fmt)
    else:
        codes, scales = mxq.mx_quantize(x, axis, fmt)
    mxq.check()
    ec, es = O.quantize_any(xn, axis, fmt, had)
    np.testing.assert_array_equal(to_np(scales), es)
    np.testing.assert_array_equal(to_np(codes), ec)


ROW_SHAPES = [(1, 32), (32, 32), (33, 64), (64, 96), (128, 128), (200, 160), (257, 416)]
COL_SHAPES = [(32, 8), (32, 32), (64, 40), (96, 136), (160, 200), (288, 392)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("had", [False, True])
@pytest.mark.parametrize("shape", ROW_SHAPES)
def test_rowwise_parity(fmt, had, shape):
    _check(_x(*shape, seed=shape[0]), "row", fmt, had)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("had", [False, True])
@pytest.mark.parametrize("shape", COL_SHAPES)
def test_colwise_parity(fmt, had, shape):
    _check(_x(*shape, seed=shape[1]), "col", fmt, had)


@pytest.mark.parametrize("fr,hr,fc,hc", [
    ("e4m3", False, "e2m1", True),   # activations / output gradients in the block pass
    ("e4m3", False, "e4m3", False),  # weights
    ("e2m1", True, "e2m1", True),    # both axes rotated, E2M1
    ("e2m1", False, "e4m3", True),
    ("e5m2", False, "e5m2", False),  # E5M2 on either side, with and without the rotation
    ("e5m2", True, "e2m1", True),
    ("e4m3", False, "e5m2", True),
    ("e2m1", True, "e5m2", False),
])
@pytest.mark.parametrize("shape", [(32, 32), (96, 160), (160, 288), (384, 256)])
def test_dual_parity(fr, hr, fc, hc, shape):
    x = _x(*shape, seed=7)
    xn = bf16_to_f32_np(x)
    cr, sr, cc, sc = mxq.mx_quantize_dual(x, fr, hr, fc, hc)
    mxq.check()
    er, esr = O.quantize_any(xn, "row", fr, hr)
    ec, esc = O.quantize_any(xn, "col", fc, hc)
    np.testing.assert_array_equal(to_np(sr), esr)
    np.testing.assert_array_equal(to_np(cr), er)
    np.testing.assert_array_equal(to_np(sc), esc)
    np.testing.assert_array_equal(to_np(cc), ec)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(288, 1440), (1056, 2088), (4128, 1056)])
def test_grouped_tile_order(fmt, shape):
    # one-byte column-wise outputs visit tiles in groups of 8 tile columns;
    # these shapes have more than one group, a ragged last group and ragged
    # tile rows and columns
    x = synth.normal_with_outliers(shape, shape[0] + shape[1]).cuda()
    _check(x, "col", fmt, False)
    _check(x, "col", fmt, True)
    if shape[1] % 32 == 0:
        cr, sr, cc, sc = mxq.mx_quantize_dual(x, "e4m3", False, "e4m3", fmt == "e5m2")
        mxq.check()
        xn = bf16_to_f32_np(x)
        ec, es = O.quantize_any(xn, "col", "e4m3", fmt == "e5m2")
        np.testing.assert_array_equal(to_np(sc), es)
        np.testing.assert_array_equal(to_np(cc), ec)
        ec, es = O.quantize_any(xn, "row", "e4m3", False)
        np.testing.assert_array_equal(to_np(sr), es)
        np.testing.assert_array_equal(to_np(cr), ec)


def _special_tensor(rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-30, 30, (rows, 1)))).astype(np.float32)
    flat = x.reshape(-1)
    n = flat.size
    idx = rng.choice(n, size=n // 50, replace=False)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 3.0e38, -3.3e38, 2.0 ** -133,
                         -(2.0 ** -130), 1e-40, 448.0, 500.0, 6.0, 7.5, -5.0], dtype=np.float32)
    flat[idx] = specials[rng.integers(0, len(specials), size=idx.size)]
    x[:32, :32] = 0.0                       # an all-zero block on both axes
    x[32:64, 32:64] = -0.0
    x[64:96, :32] = 2.0 ** -130             # subnormal maxima
    xb = torch.from_numpy(x).to(torch.bfloat16)
    return xb


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("had", [False, True])
def test_special_values(fmt, had):
    x = _special_tensor(128, 256, 3 + int(had)).cuda()
    _check(x, "row", fmt, had)
    _check(x, "col", fmt, had)


@pytest.mark.parametrize("fmt", FMTS)
def test_largest_finite_rotated_blocks(fmt):
    """Blocks whose rotated amax is the largest finite one (a single input at
    the bf16 maximum, scale byte 125 - emax + 127) and blocks whose butterfly
    sums overflow (two such inputs: scale 255, zero codes), in both layouts
    and the one-pass kernel, against the oracle."""
    bmax = np.frombuffer(np.uint32(0x7F7F0000).tobytes(), np.float32)[0]
    x = np.random.default_rng(9).standard_normal((128, 128)).astype(np.float32)
    x[0, :32] = 0.0
    x[0, 7] = bmax                   # row block 0 of row 0
    x[1, 32:64] = 0.0
    x[1, 40] = -bmax                 # row block 1 of row 1
    x[2, 64:96] = 0.0
    x[2, 70] = bmax
    x[2, 90] = bmax                  # an overflowing row block
    x[32:64, 100] = 0.0
    x[40, 100] = -bmax               # column block 1 of column 100
    x[64:96, 101] = 0.0
    x[64, 101] = bmax
    x[95, 101] = bmax                # an overflowing column block
    xb = torch.from_numpy(x).to(torch.bfloat16).cuda()
    _check(xb, "row", fmt, True)
    _check(xb, "col", fmt, True)
    xn = bf16_to_f32_np(xb)
    cr, sr, cc, sc = mxq.mx_quantize_dual(xb, fmt, True, fmt, True)
    mxq.check()
    for (codes, scales), axis in (((cr, sr), "row"), ((cc, sc), "col")):
        ec, es = O.hadamard_mx_quantize(xn, axis, fmt)
        np.testing.assert_array_equal(to_np(scales), es)
        np.testing.assert_array_equal(to_np(codes), ec)
    emax = {"e4m3": 8, "e2m1": 2, "e5m2": 15}[fmt]
    assert int(to_np(sr)[0, 0]) == 125 - emax + 127 and int(to_np(sr)[2, 2]) == 255


@pytest.mark.parametrize("case", load_blocks(), ids=lambda c: c["name"])
def test_hand_derived_blocks_on_gpu(case):
    x = torch.tensor(case["x"], dtype=torch.float32).to(torch.bfloat16).reshape(1, 32).cuda()
    codes, scales = mxq.mx_quantize(x, "row", case["fmt"])
    mxq.check()
    c = to_np(codes)[0]
    if case["fmt"] == "e2m1":
        c = O.unpack_e2m1(c)
    assert int(to_np(scales)[0, 0]) == case["scale"]
    assert [int(v) for v in c] == case["codes"]


def test_e2m1_packed_bytes_hand_derived_on_gpu():
    # the kernels' packed bytes against the hand-derived golden, never
    # unpacked (element 2j in the low nibble): row-wise one block per row,
    # column-wise the same blocks down the columns (8 columns, the last ones
    # zero), and both layouts of the one-pass quantizer
    cases = load_e2m1_packed()
    n = len(cases)
    x = torch.tensor([c["x"] for c in cases], dtype=torch.float32)      # [n, 32]
    packed = np.array([c["packed"] for c in cases], dtype=np.uint8)
    scales = np.array([[c["scale"]] for c in cases], dtype=np.uint8)
    xr = x.to(torch.bfloat16).cuda()
    codes, sc = mxq.mx_quantize(xr, "row", "e2m1")
    mxq.check()
    np.testing.assert_array_equal(to_np(codes), packed)
    np.testing.assert_array_equal(to_np(sc), scales)
    xc = torch.zeros((32, 8), dtype=torch.float32)
    xc[:, :n] = x.T
    xc = xc.to(torch.bfloat16).cuda()
    codes, sc = mxq.mx_quantize(xc, "col", "e2m1")
    mxq.check()
    np.testing.assert_array_equal(to_np(codes)[:n], packed)
    np.testing.assert_array_equal(to_np(sc)[:n], scales)
    assert not to_np(codes)[n:].any() and not to_np(sc)[n:].any()
    # one-pass quantizer, E2M1 along both axes: the blocks as the first rows
    # of a 32x32 tile (row-wise output checked), then as its first columns
    # (column-wise output checked)
    xd = torch.zeros((32, 32), dtype=torch.float32)
    xd[:n, :] = x
    cr, sr, _, _ = mxq.mx_quantize_dual(xd.to(torch.bfloat16).cuda(), "e2m1", False, "e2m1", False)
    mxq.check()
    np.testing.assert_array_equal(to_np(cr)[:n], packed)
    np.testing.assert_array_equal(to_np(sr)[:n], scales)
    _, _, cc, scc = mxq.mx_quantize_dual(xd.T.contiguous().to(torch.bfloat16).cuda(), "e2m1", False,
                                         "e2m1", False)
    mxq.check()
    np.testing.assert_array_equal(to_np(cc)[:n], packed)
    np.testing.assert_array_equal(to_np(scc)[:n], scales)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("axis", ["row", "col"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_dequantize_parity(fmt, axis, out_dtype):
    x = _special_tensor(96, 160, 11).cuda()
    codes, scales = mxq.mx_quantize(x, axis, fmt)
    got = mxq.mx_dequantize(codes, scales, 96, 160, axis, fmt, out_dtype)
    mxq.check()
    out = "f32" if out_dtype == torch.float32 else "bf16"
    exp = O.mx_dequantize(to_np(codes), to_np(scales), fmt, out)
    if axis == "col":
        exp = exp.T
    np.testing.assert_array_equal(to_np(got.float()), exp)


def test_dequantize_arbitrary_scales():
    # every scale byte, including 0 (subnormal 2^-127), 254 (overflow to inf)
    # and 255 (NaN), against every E4M3 code
    codes = torch.arange(256, dtype=torch.uint8).repeat(256, 1).reshape(256, 256)
    scales = torch.arange(256, dtype=torch.uint8).repeat_interleave(8).reshape(256, 8)
    codes = codes.contiguous()
    got = mxq.mx_dequantize(codes.cuda(), scales.cuda(), 256, 256, "row", "e4m3")
    mxq.check()
    exp = O.mx_dequantize(codes.numpy(), scales.numpy(), "e4m3")
    np.testing.assert_array_equal(to_np(got), exp)
    c2 = torch.randint(0, 256, (64, 64), dtype=torch.uint8, generator=torch.Generator().manual_seed(1))
    s2 = torch.arange(256, dtype=torch.uint8)[torch.randperm(256, generator=torch.Generator().manual_seed(2))][:256].reshape(64, 4)
    got2 = mxq.mx_dequantize(c2.cuda(), s2.cuda(), 64, 128, "row", "e2m1")
    mxq.check()
    exp2 = O.mx_dequantize(c2.numpy(), s2.numpy(), "e2m1")
    np.testing.assert_array_equal(to_np(got2), exp2)
    # E5M2: every code (its infinities and NaNs included) against every scale
    got3 = mxq.mx_dequantize(codes.cuda(), scales.cuda(), 256, 256, "row", "e5m2")
    mxq.check()
    exp3 = O.mx_dequantize(codes.numpy(), scales.numpy(), "e5m2")
    np.testing.assert_array_equal(to_np(got3), exp3)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(32, 1), (64, 37), (96, 130), (160, 258), (4128, 1001),
                                   (32, 8), (160, 264), (288, 136), (4128, 1000)])
def test_dequantize_colwise_ragged(fmt, out_dtype, shape):
    # column-wise codes [cols][rows] of random bytes and random scales: odd
    # and ragged column counts (the shared-memory transpose with scalar tail
    # stores), and column counts whose output rows are 16-byte multiples (the
    # TMA path) with partial row and column tiles
    R, C = shape
    g = torch.Generator().manual_seed(R * 7 + C)
    cb = R // 2 if fmt == "e2m1" else R
    codes = torch.randint(0, 256, (C, cb), dtype=torch.uint8, generator=g)
    scales = torch.randint(90, 170, (C, R // 32), dtype=torch.uint8, generator=g)
    got = mxq.mx_dequantize(codes.cuda(), scales.cuda(), R, C, "col", fmt, out_dtype)
    mxq.check()
    out = "f32" if out_dtype == torch.float32 else "bf16"
    exp = O.mx_dequantize(codes.numpy(), scales.numpy(), fmt, out).T
    np.testing.assert_array_equal(to_np(got.float()), exp)


def test_small_round_trip_workload():
    # 256x1024 N(0,1) with 1% x100 outliers, E4M3 row-wise, then dequantize
    x = synth.quantize_dequantize_small()["x"].cuda()
    codes, scales = mxq.mx_quantize(x, "row", "e4m3")
    back = mxq.mx_dequantize(codes, scales, 256, 1024, "row", "e4m3")
    mxq.check()
    ec, es = O.mx_quantize(bf16_to_f32_np(x), "row", "e4m3")
    np.testing.assert_array_equal(to_np(codes), ec)
    np.testing.assert_array_equal(to_np(scales), es)
    np.testing.assert_array_equal(to_np(back), O.mx_dequantize(ec, es, "e4m3"))


def test_full_size_dual_hadamard_e2m1():
    # 8192x4096 activation, fused Hadamard + E2M1 along rows and columns
    x = synth.hadamard_dual_activation()["x"].cuda()
    cr, sr, cc, sc = mxq.mx_quantize_dual(x, "e2m1", True, "e2m1", True)
    mxq.check()
    xn = bf16_to_f32_np(x)
    er, esr = O.hadamard_mx_quantize(xn, "row", "e2m1")
    np.testing.assert_array_equal(to_np(sr), esr)
    np.testing.assert_array_equal(to_np(cr), er)
    del er, esr
    ec, esc = O.hadamard_mx_quantize(xn, "col", "e2m1")
    np.testing.assert_array_equal(to_np(sc), esc)
    np.testing.assert_array_equal(to_np(cc), ec)


def test_deterministic_repeat():
    x = _x(512, 768, seed=5)
    a = mxq.mx_quantize_dual(x, "e4m3", False, "e2m1", True)
    b = mxq.mx_quantize_dual(x, "e4m3", False, "e2m1", True)
    mxq.check()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_bounded_wait_reports_timeout():
    s = mxq._stream()
    assert mxq.lib().mxq_debug_expire_wait(10_000_000, s) == 0
    assert mxq.mxq_check(s) == 5  # MXQ_ERR_TIMEOUT
    assert mxq.mxq_check(s) == 0  # cleared after being reported
    # the context is still usable
    _check(_x(64, 64), "row", "e4m3", False)
