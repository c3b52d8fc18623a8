"""Scales in the tensor cores' chunk layout (MXQ_SCALES_TC).

The quantizers can write their E8M0 scales straight into the 512-byte chunk
layout the GEMM's tcgen05.cp reads, and the GEMM then reads them in place
(no re-layout pass, no workspace).  The expected chunks are built here from
the oracle's row-major scales by the layout's definition in the header:
byte (line, block) of chunk (line / 128) * (blocked / 128) + block / 4 at
(line % 32) * 16 + ((line % 128) / 32) * 4 + block % 4, zeros past the last
line.
"""

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq, synth
from tests.libutil import bf16_to_f32_np, ensure_built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def tc_from_rowmajor(s, lines, blocked):
    nb = blocked // 32
    kcs = blocked // 128
    tiles = (lines + 127) // 128
    out = np.zeros(tiles * kcs * 512, np.uint8)
    for line in range(lines):
        for b in range(nb):
            chunk = (line // 128) * kcs + b // 4
            off = (line % 32) * 16 + ((line % 128) // 32) * 4 + b % 4
            out[chunk * 512 + off] = s[line, b]
    return out


def _x(rows, cols, seed):
    return synth.activation(rows, cols, seed).cuda()


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("had", [False, True])
@pytest.mark.parametrize("axis,shape", [("row", (200, 256)), ("row", (130, 512)),
                                        ("col", (256, 200)), ("col", (512, 136))])
def test_quantize_tc_scales(fmt, had, axis, shape):
    x = _x(*shape, seed=shape[0] + shape[1])
    q = mxq.hadamard_mx_quantize if had else mxq.mx_quantize
    codes, scales = q(x, axis, fmt, scale_layout="tc")
    mxq.check()
    ec, es = O.quantize_any(bf16_to_f32_np(x), axis, fmt, had)
    lines, blocked = (shape[0], shape[1]) if axis == "row" else (shape[1], shape[0])
    np.testing.assert_array_equal(to_np(codes), ec)
    np.testing.assert_array_equal(to_np(scales), tc_from_rowmajor(es, lines, blocked))


@pytest.mark.parametrize("fr,hr,fc,hc", [("e4m3", False, "e2m1", True), ("e4m3", False, "e4m3", False)])
def test_dual_tc_scales(fr, hr, fc, hc):
    x = _x(512, 384, seed=4)    # E2M1 column blocks need rows % 256 == 0
    cr, sr, cc, sc = mxq.mx_quantize_dual(x, fr, hr, fc, hc, scale_layout="tc")
    mxq.check()
    xn = bf16_to_f32_np(x)
    er, esr = O.quantize_any(xn, "row", fr, hr)
    ec, esc = O.quantize_any(xn, "col", fc, hc)
    np.testing.assert_array_equal(to_np(cr), er)
    np.testing.assert_array_equal(to_np(cc), ec)
    np.testing.assert_array_equal(to_np(sr), tc_from_rowmajor(esr, 512, 384))
    np.testing.assert_array_equal(to_np(sc), tc_from_rowmajor(esc, 384, 512))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("shape", [(200, 264, 512), (384, 520, 1024), (64, 40, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_reads_tc_scales_in_place(fmt, shape):
    # same codes and scale bytes through both paths: bitwise equal products,
    # and both within the bound of the oracle's
    M, N, K = shape
    xa = _x(M, K, seed=M)
    xb = synth.weight(N, K, seed=N).cuda()
    A, sA = mxq.mx_quantize(xa, "row", fmt, scale_layout="tc")
    B, sB = mxq.mx_quantize(xb, "row", fmt, scale_layout="tc")
    A2, sA2 = mxq.mx_quantize(xa, "row", fmt)
    B2, sB2 = mxq.mx_quantize(xb, "row", fmt)
    c_tc = mxq.mx_gemm(A, sA, B, sB, fmt, M, N, K, scale_layout="tc")
    c_rm = mxq.mx_gemm(A2, sA2, B2, sB2, fmt, M, N, K)
    mxq.check()
    assert torch.equal(c_tc, c_rm)
    oA, osA = O.mx_quantize(bf16_to_f32_np(xa), "row", fmt)
    oB, osB = O.mx_quantize(bf16_to_f32_np(xb), "row", fmt)
    ref, S = O.mx_gemm_f64(oA, osA, oB, osB, fmt)
    assert np.all(np.abs(to_np(c_tc).astype(np.float64) - ref) <= 2e-4 * S)


def test_tc_argument_errors():
    t = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    s = mxq._stream()
    TC = mxq.SCALES_TC
    # quantizer: blocked dimension must cover whole chunks (pairs for E2M1)
    assert mxq.mxq_quantize_ex(p, 64, 96, mxq.ROWWISE, mxq.E4M3, 0, p, p, TC, s) == 1
    assert mxq.mxq_quantize_ex(p, 64, 128, mxq.ROWWISE, mxq.E2M1, 0, p, p, TC, s) == 1
    assert mxq.mxq_quantize_ex(p, 64, 128, mxq.ROWWISE, mxq.E4M3, 0, p, p + 4, TC, s) == 2
    assert mxq.mxq_quantize_ex(p, 64, 128, mxq.ROWWISE, mxq.E4M3, 0, p, p, 9, s) == 1
    # GEMM: K in whole chunks (chunk pairs for E2M1), 16-byte aligned scales
    assert mxq.mxq_gemm_ex(p, p, p, p, mxq.E4M3, 128, 128, 96, p, 0, TC, None, 0, s) == 1
    assert mxq.mxq_gemm_ex(p, p, p, p, mxq.E2M1, 128, 128, 128, p, 0, TC, None, 0, s) == 1
    assert mxq.mxq_gemm_ex(p, p + 4, p, p, mxq.E4M3, 128, 128, 128, p, 0, TC, None, 0, s) == 2
    assert mxq.mxq_gemm_ex(p, p, p, p, mxq.E4M3, 128, 128, 128, p, 0, 7, None, 0, s) == 1
    # row-major through the extended entry point still needs its workspace
    assert mxq.mxq_gemm_ex(p, p, p, p, mxq.E4M3, 128, 128, 128, p, 0, 0, None, 0, s) == 1
    mxq.check()


def test_epilogue_tc_argument_errors():
    t = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    s = mxq._stream()
    TC, RM = mxq.SCALES_TC, mxq.SCALES_ROWMAJOR
    Q = mxq.mxq_gemm_quantize_ex
    assert Q(p, p, p, p, 0, 128, 96, 128, TC, 0, p, p, TC, None, 0, s) == 1        # N % 128
    assert Q(p, p, p, p, 0, 128, 128, 128, TC, 1, p, p, TC, None, 0, s) == 1       # E2M1: N % 256
    assert Q(p, p, p, p, 0, 128, 128, 128, TC, 0, p, p + 4, TC, None, 0, s) == 2   # alignment
    assert Q(p, p, p, p, 0, 128, 128, 128, TC, 0, p, p, 5, None, 0, s) == 1        # layout
    assert Q(p, p, p, p, 0, 128, 128, 128, RM, 0, p, p, TC, None, 0, s) == 1       # needs workspace
    mxq.check()
