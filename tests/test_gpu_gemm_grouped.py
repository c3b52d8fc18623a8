"""Grouped GEMM launch (mxq_gemm_grouped): several independent problems of one
format in one persistent grid.  Each output must be bit for bit what the
single-problem call (mxq_gemm_ex with chunk-layout scales) writes -- the tiles
and their K order are the same -- and, on small shapes, within the GEMM bound
of the fp64 oracle."""

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


def _operands(M, N, K, fmt, seed, hadamard):
    a = synth.activation(K, M, seed).cuda()          # [K tokens, M] -> column-wise along K
    b = synth.activation(K, N, seed + 1).cuda()
    if hadamard:
        A, sA = mxq.hadamard_mx_quantize(a, "col", fmt, scale_layout="tc")
        B, sB = mxq.hadamard_mx_quantize(b, "col", fmt, scale_layout="tc")
    else:
        A, sA = mxq.mx_quantize(a, "col", fmt, scale_layout="tc")
        B, sB = mxq.mx_quantize(b, "col", fmt, scale_layout="tc")
    return a, b, A, sA, B, sB


@pytest.mark.parametrize("fmt,had", [("e2m1", True), ("e4m3", False), ("e5m2", False)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grouped_equals_single_calls(fmt, had, out_dtype):
    kq = 256
    shapes = [(256, 384, 2 * kq), (640, 256, 4 * kq), (304, 520, 3 * kq), (128, 1024, kq)]
    probs, singles = [], []
    for i, (M, N, K) in enumerate(shapes):
        _, _, A, sA, B, sB = _operands(M, N, K, fmt, 10 * i, had)
        probs.append((A, sA, B, sB, M, N, K))
        singles.append(mxq.mx_gemm(A, sA, B, sB, fmt, M, N, K, out_dtype, scale_layout="tc"))
    outs = mxq.mx_gemm_grouped(probs, fmt, out_dtype)
    mxq.check()
    for (M, N, K), got, ref in zip(shapes, outs, singles):
        assert torch.equal(got, ref), (M, N, K)


def test_grouped_matches_oracle():
    # two MXFP4 Wgrad-like problems (rotated E2M1 along the token axis) and
    # their fp64 oracle products, element by element
    shapes = [(384, 256, 512), (256, 640, 256)]
    probs, refs = [], []
    for i, (M, N, K) in enumerate(shapes):
        a, b, A, sA, B, sB = _operands(M, N, K, "e2m1", 50 + i, True)
        probs.append((A, sA, B, sB, M, N, K))
        oA, osA = O.hadamard_mx_quantize(bf16_to_f32_np(a), "col", "e2m1")
        oB, osB = O.hadamard_mx_quantize(bf16_to_f32_np(b), "col", "e2m1")
        refs.append(O.mx_gemm_f64(oA, osA, oB, osB, "e2m1"))
    outs = mxq.mx_gemm_grouped(probs, "e2m1")
    mxq.check()
    for got, (ref, S) in zip(outs, refs):
        assert np.all(np.abs(to_np(got).astype(np.float64) - ref) <= 2e-4 * S)


def test_grouped_block_wgrad_shapes_match_single_calls():
    # the four Wgrad GEMMs of a Llama-3.1-8B decoder block at 8192 tokens,
    # grouped as the benchmark runs them, against one launch per GEMM
    T = 8192
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    probs, singles = [], []
    for fin, fout in [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]:
        A = torch.randint(0, 256, (fout, T // 2), dtype=torch.uint8, device="cuda", generator=g)
        B = torch.randint(0, 256, (fin, T // 2), dtype=torch.uint8, device="cuda", generator=g)
        sA = torch.randint(118, 136, (mxq.mxq_scales_tc_bytes(fout, T),), dtype=torch.uint8,
                           device="cuda", generator=g)
        sB = torch.randint(118, 136, (mxq.mxq_scales_tc_bytes(fin, T),), dtype=torch.uint8,
                           device="cuda", generator=g)
        probs.append((A, sA, B, sB, fout, fin, T))
        singles.append(mxq.mx_gemm(A, sA, B, sB, "e2m1", fout, fin, T, scale_layout="tc"))
    outs = mxq.mx_gemm_grouped(probs, "e2m1")
    mxq.check()
    for got, ref in zip(outs, singles):
        assert torch.equal(got, ref)


@pytest.mark.parametrize("n_problems", [1, 8])
def test_grouped_limits_match_single_calls(n_problems):
    # the group of one (the single-problem path) and the largest group (8
    # problems of mixed shapes: single tiles, ragged M and N, K from one to
    # five 128-element chunks), MXFP8 with bf16 output
    shapes = [(128, 128, 128), (256, 384, 256), (200, 264, 384), (512, 128, 640),
              (128, 520, 128), (384, 256, 512), (136, 392, 256), (256, 1024, 128)][:n_problems]
    probs, singles = [], []
    for i, (M, N, K) in enumerate(shapes):
        _, _, A, sA, B, sB = _operands(M, N, K, "e4m3", 70 + 3 * i, False)
        probs.append((A, sA, B, sB, M, N, K))
        singles.append(mxq.mx_gemm(A, sA, B, sB, "e4m3", M, N, K, torch.bfloat16,
                                   scale_layout="tc"))
    outs = mxq.mx_gemm_grouped(probs, "e4m3", torch.bfloat16)
    mxq.check()
    assert len(outs) == n_problems
    for (M, N, K), got, ref in zip(shapes, outs, singles):
        assert torch.equal(got, ref), (M, N, K)
