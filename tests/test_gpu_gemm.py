"""Parity of the tcgen05 block-scaled GEMM with the fp64 oracle.

Small shapes: the operands are quantized by the oracle on the CPU and
uploaded, so the GEMM is checked alone, element by element.  Full-size
shapes: the CUDA quantizers feed the CUDA GEMM (the path end to end); the
oracle quantizes only the sampled rows and columns from the same bf16
inputs and computes those outputs in fp64.

Acceptance per element: |C - C_ref| <= 2e-4 * sum_k |a_k b_k| for fp32
output; bf16 output may add its own rounding, 2^-8 |C_ref|.
"""

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq, synth
from tests.libutil import bf16_to_f32_np, ensure_built, to_np

pytestmark = pytest.mark.gpu

REL = 2e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _assert_close(got, ref, S, bf16=False):
    tol = REL * S + (2.0 ** -8 * np.abs(ref) if bf16 else 0.0)
    err = np.abs(got.astype(np.float64) - ref)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{bad.sum()} of {bad.size} outside the bound; first at {tuple(i)}: "
            f"got {got[tuple(i)]!r}, ref {ref[tuple(i)]!r}, S {S[tuple(i)]!r}")


def _oracle_operands(M, N, K, fmt, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_t(3, size=(M, K)) * np.exp(rng.standard_normal(K))[None, :]).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    wb = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    A, sA = O.mx_quantize(xb, "row", fmt)
    B, sB = O.mx_quantize(wb, "row", fmt)
    return A, sA, B, sB


def _run_gpu(A, sA, B, sB, fmt, M, N, K, out_dtype):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    C = mxq.mx_gemm(t(A), t(sA), t(B), t(sB), fmt, M, N, K, out_dtype=out_dtype)
    mxq.check()
    return to_np(C.float())


SHAPES = [
    (128, 256, 128),    # one tile, one K stage
    (128, 256, 1024),
    (256, 512, 512),    # several tiles
    (200, 264, 160),    # ragged M, N and a partial K stage
    (64, 40, 96),       # smaller than one tile
    (384, 776, 2080),   # odd tile counts, many K stages, K tail
    (1, 4, 32),         # degenerate: one row, four columns, one k-block
    (3, 12, 64),        # a few rows and columns, one E2M1 MMA's worth of K
    (257, 260, 4128),   # one row / four columns past a tile, K just past a stage
]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_small_full_compare(fmt, shape):
    M, N, K = shape
    A, sA, B, sB = _oracle_operands(M, N, K, fmt, seed=M + N + K)
    ref, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
    got = _run_gpu(A, sA, B, sB, fmt, M, N, K, torch.float32)
    _assert_close(got, ref, S)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_gemm_bf16_output(fmt):
    M, N, K = 256, 264, 512
    A, sA, B, sB = _oracle_operands(M, N, K, fmt, seed=3)
    ref, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
    got = _run_gpu(A, sA, B, sB, fmt, M, N, K, torch.bfloat16)
    _assert_close(got, ref, S, bf16=True)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
def test_gemm_integer_exact(fmt):
    # small-integer elements with unit scales: fp32 accumulation is exact
    rng = np.random.default_rng(4)
    M, N, K = 128, 256, 256
    table = O.decode_table(fmt)
    ints = [c for c, v in enumerate(table) if np.isfinite(v) and v == int(v) and abs(v) <= 4]
    a = rng.choice(ints, size=(M, K)).astype(np.uint8)
    b = rng.choice(ints, size=(N, K)).astype(np.uint8)
    if fmt == "e2m1":
        a, b = O.pack_e2m1(a), O.pack_e2m1(b)
    sA = np.full((M, K // 32), 127, np.uint8)
    sB = np.full((N, K // 32), 127, np.uint8)
    ref, _ = O.mx_gemm_f64(a, sA, b, sB, fmt)
    got = _run_gpu(a, sA, b, sB, fmt, M, N, K, torch.float32)
    np.testing.assert_array_equal(got, ref.astype(np.float32))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "e5m2"])
def test_gemm_scale_placement(fmt):
    # one distinct scale per (row, k-block) for A and B, unit elements: every
    # output is a sum of distinct powers of two, so a scale read from the
    # wrong row or k-block changes the result
    rng = np.random.default_rng(5)
    M, N, K = 256, 512, 512
    one = {"e4m3": 0x38, "e2m1": 0x2, "e5m2": 0x3C}[fmt]
    a = np.full((M, K), one, np.uint8)
    b = np.full((N, K), one, np.uint8)
    if fmt == "e2m1":
        a, b = O.pack_e2m1(a), O.pack_e2m1(b)
    sA = rng.integers(100, 154, size=(M, K // 32)).astype(np.uint8)
    sB = rng.integers(100, 154, size=(N, K // 32)).astype(np.uint8)
    ref, S = O.mx_gemm_f64(a, sA, b, sB, fmt)
    got = _run_gpu(a, sA, b, sB, fmt, M, N, K, torch.float32)
    _assert_close(got, ref, S)


def test_gemm_deterministic_and_workspace_reuse():
    M, N, K = 384, 512, 1024
    A, sA, B, sB = _oracle_operands(M, N, K, "e4m3", seed=9)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = mxq.gemm_workspace(M, N, K, "e4m3", "cuda")
    c1 = mxq.mx_gemm(t(A), t(sA), t(B), t(sB), "e4m3", M, N, K, workspace=ws)
    c2 = mxq.mx_gemm(t(A), t(sA), t(B), t(sB), "e4m3", M, N, K, workspace=ws)
    mxq.check()
    assert torch.equal(c1, c2)


def test_gemm_argument_errors():
    t = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    s = mxq._stream()
    assert mxq.mxq_gemm(p, p, p, p, 0, 128, 128, 48, p, 0, p, 1024, s) == 1      # K % 32
    assert mxq.mxq_gemm(p, p, p, p, 0, 128, 130, 64, p, 0, p, 1 << 20, s) == 2   # N % 4
    assert mxq.mxq_gemm(p, p, p, p, 0, 128, 128, 64, p, 0, p, 16, s) == 6        # workspace
    assert mxq.mxq_gemm(p, p, p, p, 5, 128, 128, 64, p, 0, p, 1 << 20, s) == 1   # fmt
    # scales padded to 256 rows for A (a pair of m-tiles) and B (one n-tile)
    assert mxq.mxq_gemm_workspace_size(128, 256, 4096, 0) == 256 * 128 + 256 * 128


def _sample_idx(n, rng, k=192):
    pick = rng.choice(n, size=min(k, n), replace=False)
    return np.unique(np.concatenate([pick, np.arange(min(32, n)), np.arange(max(0, n - 32), n)]))


def test_mlp_up_forward_full_size_sampled():
    # X 8192x4096 (row-wise E4M3) times W 4096x14336 given as K x N
    # (column-wise transposed E4M3 -> [14336][4096]), fp32 out
    d = synth.mlp_up_forward()
    x, w = d["x"].cuda(), d["w"].cuda()
    M, K = x.shape
    N = w.shape[1]
    A, sA = mxq.mx_quantize(x, "row", "e4m3")
    B, sB = mxq.mx_quantize(w, "col", "e4m3")
    C = mxq.mx_gemm(A, sA, B, sB, "e4m3", M, N, K)
    mxq.check()
    rng = np.random.default_rng(1234)
    rows, cols = _sample_idx(M, rng), _sample_idx(N, rng)
    xn = bf16_to_f32_np(d["x"])
    wn = bf16_to_f32_np(d["w"])
    oA, osA = O.mx_quantize(xn[rows], "row", "e4m3")
    oB, osB = O.mx_quantize(wn[:, cols], "col", "e4m3")
    ref, S = O.mx_gemm_f64(oA, osA, oB, osB, "e4m3")
    got = to_np(C[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    _assert_close(got, ref, S)
    # one full row and one full column
    r0, c0 = int(rows[len(rows) // 2]), int(cols[len(cols) // 2])
    oBf, osBf = O.mx_quantize(wn, "col", "e4m3")
    ref_r, S_r = O.mx_gemm_f64(oA[[list(rows).index(r0)]], osA[[list(rows).index(r0)]], oBf, osBf, "e4m3")
    _assert_close(to_np(C[r0:r0 + 1]), ref_r, S_r)
    oAf, osAf = O.mx_quantize(xn, "row", "e4m3")
    j = list(cols).index(c0)
    ref_c, S_c = O.mx_gemm_f64(oAf, osAf, oB[[j]], osB[[j]], "e4m3")
    _assert_close(to_np(C[:, c0:c0 + 1]), ref_c, S_c)


def test_mlp_wgrad_hadamard_fp4_full_size_sampled():
    # dW = (H dY)^T (H X): dY 16384x14336, X 16384x4096, both rotated along
    # tokens and quantized column-wise to E2M1; fp32 out 14336x4096
    d = synth.mlp_wgrad()
    dy, x = d["dy"].cuda(), d["x"].cuda()
    T, n_out = dy.shape
    n_in = x.shape[1]
    A, sA = mxq.hadamard_mx_quantize(dy, "col", "e2m1")
    B, sB = mxq.hadamard_mx_quantize(x, "col", "e2m1")
    C = mxq.mx_gemm(A, sA, B, sB, "e2m1", n_out, n_in, T)
    mxq.check()
    rng = np.random.default_rng(1234)
    rows, cols = _sample_idx(n_out, rng), _sample_idx(n_in, rng)
    dyn = bf16_to_f32_np(d["dy"][:, torch.from_numpy(rows)])
    xn = bf16_to_f32_np(d["x"][:, torch.from_numpy(cols)])
    oA, osA = O.hadamard_mx_quantize(dyn, "col", "e2m1")
    oB, osB = O.hadamard_mx_quantize(xn, "col", "e2m1")
    # the sampled operand rows equal the GPU's bit for bit
    np.testing.assert_array_equal(to_np(A[torch.from_numpy(rows).cuda()]), oA)
    ref, S = O.mx_gemm_f64(oA, osA, oB, osB, "e2m1")
    got = to_np(C[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    _assert_close(got, ref, S)
