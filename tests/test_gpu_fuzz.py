"""Seeded random shapes through the quantizers and the GEMM, against the
oracle: ragged rows, columns and K tails in every combination the
preconditions allow, each format and layout."""

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


def _quant_cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        axis = ["row", "col"][i % 2]
        fmt = ["e4m3", "e2m1", "e5m2"][(i // 2) % 3]
        had = bool(rng.integers(0, 2))
        if axis == "row":
            rows, cols = int(rng.integers(1, 300)), 32 * int(rng.integers(1, 14))
        else:
            rows, cols = 32 * int(rng.integers(1, 12)), 8 * int(rng.integers(1, 50))
        out.append((axis, fmt, had, rows, cols, int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("case", _quant_cases(), ids=lambda c: f"{c[0]}-{c[1]}-h{int(c[2])}-{c[3]}x{c[4]}")
def test_quantizer_random_shapes(case):
    axis, fmt, had, rows, cols, seed = case
    x = synth.normal_with_outliers((rows, cols), seed).cuda()
    q = mxq.hadamard_mx_quantize if had else mxq.mx_quantize
    codes, scales = q(x, axis, fmt)
    mxq.check()
    ec, es = O.quantize_any(bf16_to_f32_np(x), axis, fmt, had)
    np.testing.assert_array_equal(to_np(scales), es)
    np.testing.assert_array_equal(to_np(codes), ec)


def _gemm_cases(n=18, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        fmt = ["e4m3", "e2m1", "e5m2"][i % 3]
        M = int(rng.integers(1, 700))
        N = 4 * int(rng.integers(1, 180))
        K = 32 * int(rng.integers(1, 48))
        out.append((fmt, M, N, K, int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("case", _gemm_cases(), ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}")
def test_gemm_random_shapes(case):
    fmt, M, N, K, seed = case
    rng = np.random.default_rng(seed)
    xa = torch.from_numpy((rng.standard_t(3, (M, K)) * 0.5).astype(np.float32)).to(torch.bfloat16)
    xb = torch.from_numpy((rng.standard_normal((N, K)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    A, sA = O.mx_quantize(xa.float().numpy(), "row", fmt)
    B, sB = O.mx_quantize(xb.float().numpy(), "row", fmt)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    C = mxq.mx_gemm(t(A), t(sA), t(B), t(sB), fmt, M, N, K)
    mxq.check()
    ref, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
    err = np.abs(to_np(C).astype(np.float64) - ref)
    assert np.all(err <= 2e-4 * S), f"{(err > 2e-4 * S).sum()} outside the bound"


def _dual_cases(n=12, seed=99):
    # the one-pass quantizer takes E4M3 and E2M1 (E5M2 is refused as unsupported)
    rng = np.random.default_rng(seed)
    fmts = ["e4m3", "e2m1"]
    out = []
    for i in range(n):
        rows, cols = 32 * int(rng.integers(1, 12)), 32 * int(rng.integers(1, 12))
        out.append((fmts[i % 2], bool(rng.integers(0, 2)), fmts[(i // 2) % 2],
                    bool(rng.integers(0, 2)), rows, cols, int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("case", _dual_cases(),
                         ids=lambda c: f"{c[0]}h{int(c[1])}-{c[2]}h{int(c[3])}-{c[4]}x{c[5]}")
def test_dual_random_shapes(case):
    fr, hr, fc, hc, rows, cols, seed = case
    x = synth.normal_with_outliers((rows, cols), seed).cuda()
    cr, sr, cc, sc = mxq.mx_quantize_dual(x, fr, hr, fc, hc)
    mxq.check()
    xf = bf16_to_f32_np(x)
    ec, es = O.quantize_any(xf, "row", fr, hr)
    np.testing.assert_array_equal(to_np(sr), es)
    np.testing.assert_array_equal(to_np(cr), ec)
    ec, es = O.quantize_any(xf, "col", fc, hc)
    np.testing.assert_array_equal(to_np(sc), es)
    np.testing.assert_array_equal(to_np(cc), ec)


def _ablation_cases(n=12, seed=5150):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        axis = ["row", "col"][i % 2]
        fmt = ["e4m3", "e2m1", "e5m2"][(i // 2) % 3]
        if axis == "row":
            rows, cols = int(rng.integers(1, 200)), 32 * int(rng.integers(1, 10))
        else:
            rows, cols = 32 * int(rng.integers(1, 8)), 8 * int(rng.integers(1, 40))
        had = bool(rng.integers(0, 2))
        mask = int(rng.integers(0, 1 << 32)) if had else 0   # a sign mask needs the rotation
        out.append((axis, fmt, had, mask, True, rows, cols,
                    int(rng.integers(0, 1 << 63))))
    return out


@pytest.mark.parametrize("case", _ablation_cases(),
                         ids=lambda c: f"{c[0]}-{c[1]}-h{int(c[2])}-{c[5]}x{c[6]}")
def test_ablation_random_shapes(case):
    axis, fmt, had, mask, sr, rows, cols, seed = case
    x = synth.normal_with_outliers((rows, cols), seed & 0xFFFF).cuda()
    codes, scales = mxq.mx_quantize_ablation(x, axis, fmt, had, mask, sr, seed)
    mxq.check()
    ec, es = O.mx_quantize_ablation(bf16_to_f32_np(x), axis, fmt, had, mask, sr, seed)
    np.testing.assert_array_equal(to_np(scales), es)
    np.testing.assert_array_equal(to_np(codes), ec)
