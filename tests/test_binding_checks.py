"""The tensor-level binding's buffer checks (CPU): every wrapper accepts the
buffers it allocates itself and correctly sized caller buffers, and rejects
host tensors, wrong dtypes, non-contiguous and undersized buffers before
any launch.

The library's entry points are replaced by recorders here (no GPU), and
the device check is stubbed so that host tensors stand in for device ones;
the real library still answers the host-only size queries."""

import pytest
import torch

from precision_mx_quantize_gb300 import mxq
from tests.libutil import ensure_built

RAW = ["mxq_quantize", "mxq_hadamard_quantize", "mxq_quantize_dual", "mxq_quantize_ex",
       "mxq_quantize_dual_ex", "mxq_quantize_ablation", "mxq_dequantize", "mxq_gemm",
       "mxq_gemm_ex", "mxq_gemm_quantize", "mxq_gemm_quantize_ex"]


@pytest.fixture
def fake_device(monkeypatch):
    ensure_built()
    calls = []
    for name in RAW:
        monkeypatch.setattr(mxq, name, lambda *a, _n=name: calls.append(_n) or 0)
    monkeypatch.setattr(mxq, "_stream", lambda device=None: 0)
    monkeypatch.setattr(mxq, "_on_gpu", lambda t: True)
    return calls


def _x(r, c):
    return torch.zeros(r, c, dtype=torch.bfloat16)


QUANT_CASES = [(r, c, axis, fmt) for (r, c) in [(64, 96), (256, 512), (33, 64)]
               for axis in ("row", "col") for fmt in ("e4m3", "e2m1", "e5m2")
               if (axis == "row" and c % 32 == 0) or (axis == "col" and r % 32 == 0)]


@pytest.mark.parametrize("case", QUANT_CASES, ids=str)
def test_quantizers_accept_their_own_and_exact_buffers(fake_device, case):
    r, c, axis, fmt = case
    x = _x(r, c)
    for q in (mxq.mx_quantize, mxq.hadamard_mx_quantize):
        codes, scales = q(x, axis, fmt)
        q(x, axis, fmt, out=(codes, scales))
        cs, ss = mxq.code_shape(r, c, axis, fmt)
        assert tuple(codes.shape) == cs and tuple(scales.shape) == ss
    mxq.mx_quantize_ablation(x, axis, fmt, True, 5, True, 7)
    mxq.mx_dequantize(codes, scales, r, c, axis, fmt, torch.float32)
    mxq.mx_dequantize(codes, scales, r, c, axis, fmt, torch.bfloat16,
                      out=torch.empty(r, c, dtype=torch.bfloat16))
    assert fake_device


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
def test_tc_scale_layouts_and_dual(fake_device, fmt):
    x = _x(512, 256)
    for axis in ("row", "col"):
        codes, scales = mxq.mx_quantize(x, axis, fmt, scale_layout="tc")
        lines, blocked = (512, 256) if axis == "row" else (256, 512)
        assert scales.numel() == mxq.mxq_scales_tc_bytes(lines, blocked)
        mxq.mx_quantize(x, axis, fmt, out=(codes, scales), scale_layout="tc")
    if fmt != "e5m2":
        for layout in ("rowmajor", "tc"):
            out = mxq.mx_quantize_dual(x, "e4m3", False, fmt, True, scale_layout=layout)
            mxq.mx_quantize_dual(x, "e4m3", False, fmt, True, out=out, scale_layout=layout)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("layout", ["rowmajor", "tc"])
def test_gemm_wrappers_accept_quantizer_outputs(fake_device, fmt, layout):
    M, N, K = 256, 384, 512
    A, sA = mxq.mx_quantize(_x(M, K), "row", fmt, scale_layout=layout)
    B, sB = mxq.mx_quantize(_x(N, K), "row", fmt, scale_layout=layout)
    for od in (torch.float32, torch.bfloat16):
        C = mxq.mx_gemm(A, sA, B, sB, fmt, M, N, K, od, scale_layout=layout)
        assert C.shape == (M, N) and C.dtype == od
        mxq.mx_gemm(A, sA, B, sB, fmt, M, N, K, od, out=C, scale_layout=layout)
    # a transposed operand from the column-wise quantizer (the dgrad B)
    Bt, sBt = mxq.mx_quantize(_x(K, N), "col", fmt, scale_layout=layout)
    mxq.mx_gemm(A, sA, Bt, sBt, fmt, M, N, K, scale_layout=layout)
    for out_fmt in ("e4m3", "e2m1", "e5m2"):
        for out_layout in ("rowmajor", "tc"):
            q = mxq.mx_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt, scale_layout=layout,
                                     out_scale_layout=out_layout)
            mxq.mx_gemm_quantize(A, sA, B, sB, fmt, M, N, K, out_fmt, out=q, scale_layout=layout,
                                 out_scale_layout=out_layout)


def test_bad_buffers_are_rejected(fake_device):
    x = _x(64, 128)
    codes, scales = mxq.mx_quantize(x, "row", "e4m3")
    c2, s2 = mxq.mx_quantize(x, "col", "e2m1")
    A, sA = mxq.mx_quantize(_x(128, 256), "row", "e4m3")
    n = len(fake_device)
    with pytest.raises(ValueError, match="codes"):
        mxq.mx_quantize(x, "row", "e4m3", out=(codes[:-1], scales))
    with pytest.raises(ValueError, match="scales"):
        mxq.mx_quantize(x, "row", "e4m3", out=(codes, scales[:-1]))
    with pytest.raises(ValueError, match="must be torch.uint8"):
        mxq.mx_quantize(x, "row", "e4m3", out=(codes.to(torch.int16), scales))
    with pytest.raises(ValueError, match="contiguous"):
        mxq.mx_quantize(_x(128, 64).t(), "row", "e4m3")
    with pytest.raises(ValueError, match="bfloat16"):
        mxq.mx_quantize(x.float(), "row", "e4m3")
    with pytest.raises(ValueError, match="2-D"):
        mxq.mx_quantize(x.reshape(-1), "row", "e4m3")
    # E2M1 codes are half the size: E4M3-sized expectations must not pass for
    # a column-wise E4M3 request on E2M1-sized buffers
    with pytest.raises(ValueError, match="codes"):
        mxq.mx_quantize(x, "col", "e4m3", out=(c2, s2))
    with pytest.raises(ValueError, match="out_dtype"):
        mxq.mx_dequantize(codes, scales, 64, 128, "row", "e4m3", torch.float16)
    with pytest.raises(ValueError, match="out"):
        mxq.mx_dequantize(codes, scales, 64, 128, "row", "e4m3", torch.float32,
                          out=torch.empty(64, 127))
    with pytest.raises(ValueError, match="codes_B"):
        mxq.mx_gemm(A, sA, A, sA, "e4m3", 128, 256, 256)
    with pytest.raises(ValueError, match="out"):
        mxq.mx_gemm(A, sA, A, sA, "e4m3", 128, 128, 256, out=torch.empty(128, 128,
                                                                          dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="no tensor-core scale layout"):
        mxq.mx_quantize(_x(64, 96), "row", "e4m3", scale_layout="tc")
    assert len(fake_device) == n        # nothing rejected reached the library


def test_host_tensors_never_reach_the_library(monkeypatch):
    ensure_built()
    calls = []
    for name in RAW:
        monkeypatch.setattr(mxq, name, lambda *a, _n=name: calls.append(_n) or 0)
    x = _x(64, 128)
    with pytest.raises(ValueError, match="CUDA device"):
        mxq.mx_quantize(x, "row", "e4m3")
    with pytest.raises(ValueError, match="CUDA device"):
        mxq.mx_quantize_dual(x)
    with pytest.raises(ValueError, match="CUDA device"):
        mxq.mx_dequantize(torch.zeros(64, 128, dtype=torch.uint8),
                          torch.zeros(64, 4, dtype=torch.uint8), 64, 128)
    with pytest.raises(ValueError, match="CUDA device"):
        z = torch.zeros(128, 128, dtype=torch.uint8)
        mxq.mx_gemm(z, torch.zeros(128, 4, dtype=torch.uint8), z,
                    torch.zeros(128, 4, dtype=torch.uint8), "e4m3", 128, 128, 128)
    assert calls == []
