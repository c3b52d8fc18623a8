"""GPU test of mxq_gemm_noalloc, the GEMM entry point for callers that cannot
allocate device memory when they call (a plug-in that receives only its input
and output buffers from a host application owning the memory pool, or code
under a fixed memory budget).  Its scale scratch is a fixed buffer inside the
library instead of a caller workspace.

The file is named to be collected last.  Through the C ABI it checks, on
calls in a row that share the fixed buffer:
  * the output against the oracle's fp64 product of the same operands, within
    the GEMM bound of the parity tests (2e-4 * sum_k |a_k b_k| per element),
    and against mxq_gemm (the entry point with a caller workspace);
  * that no call depends on what an earlier call left in the buffer: the
    first call poisons it (every scale byte 0xFF, the E8M0 NaN, over a larger
    footprint than the later calls use), so a later call that read a stale
    scale for one of its k-blocks -- the zero padding past K included --
    would produce a non-finite output;
  * the rejection of problems larger than the buffer.
"""

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq
from tests.libutil import ensure_built, to_np

pytestmark = pytest.mark.gpu

REL = 2e-4   # the GEMM tolerance of the parity tests: 2e-4 * sum_k |a_k b_k|
BUF = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _operands(M, N, K, fmt, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_t(3, size=(M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    A, sA = O.mx_quantize(torch.from_numpy(x).to(torch.bfloat16).float().numpy(), "row", fmt)
    B, sB = O.mx_quantize(torch.from_numpy(w).to(torch.bfloat16).float().numpy(), "row", fmt)
    return A, sA, B, sB


def _noalloc(d, fmt, M, N, K):
    f = mxq.E4M3 if fmt == "e4m3" else mxq.E2M1
    stream = mxq._stream()
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = mxq.mxq_gemm_noalloc(d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), d[3].data_ptr(),
                              f, M, N, K, c.data_ptr(), mxq.OUT_F32, stream)
    assert st == 0, mxq.STATUS.get(st, st)
    assert mxq.mxq_check(stream) == 0
    return to_np(c)


def _poison():
    # E4M3 operands whose every scale is 0xFF: the call writes 0xFF over
    # (512 + 768) rows x 132 k-blocks of the buffer (padding included)
    M, N, K = 512, 768, 4224
    A = torch.full((M, K), 0x38, dtype=torch.uint8, device="cuda")
    B = torch.full((N, K), 0x38, dtype=torch.uint8, device="cuda")
    sA = torch.full((M, K // 32), 0xFF, dtype=torch.uint8, device="cuda")
    sB = torch.full((N, K // 32), 0xFF, dtype=torch.uint8, device="cuda")
    return (A, sA, B, sB), M, N, K


def test_noalloc_matches_oracle_on_calls_in_a_row():
    d, M, N, K = _poison()
    assert mxq.mxq_gemm_workspace_size(M, N, K, mxq.E4M3) <= BUF
    poisoned = _noalloc(d, "e4m3", M, N, K)
    # every product carries two 0xFF scales (NaN, or 2^128 if read as a
    # number): no output is finite
    assert not np.isfinite(poisoned).any()
    foot0 = mxq.mxq_gemm_workspace_size(M, N, K, mxq.E4M3)
    # later calls: ragged M, N and K (padding rows and k-blocks), both formats,
    # each footprint inside the poisoned one
    for (M, N, K, fmt, seed) in [(200, 264, 160, "e2m1", 2), (384, 520, 2080, "e4m3", 1),
                                 (257, 300, 4160, "e2m1", 3)]:
        f = mxq.E4M3 if fmt == "e4m3" else mxq.E2M1
        assert mxq.mxq_gemm_workspace_size(M, N, K, f) <= foot0
        A, sA, B, sB = _operands(M, N, K, fmt, seed)
        ref, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
        d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (A, sA, B, sB)]
        got = _noalloc(d, fmt, M, N, K).astype(np.float64)
        assert np.isfinite(got).all(), (M, N, K, fmt)
        assert np.all(np.abs(got - ref) <= REL * S), (M, N, K, fmt)
        # and the same as the entry point with a caller workspace
        c_ws = mxq.mx_gemm(d[0], d[1], d[2], d[3], fmt, M, N, K)
        mxq.check()
        np.testing.assert_array_equal(got, to_np(c_ws).astype(np.float64))


def test_noalloc_rejects_problems_beyond_the_buffer():
    # (65536 + 65536) rows x 256 k-blocks of scales = 32 MiB > 16 MiB
    assert mxq.mxq_gemm_workspace_size(65536, 65536, 8192, mxq.E4M3) > BUF
    p = torch.zeros(16, dtype=torch.uint8, device="cuda").data_ptr()
    st = mxq.mxq_gemm_noalloc(p, p, p, p, mxq.E4M3, 65536, 65536, 8192, p, mxq.OUT_F32,
                              mxq._stream())
    assert st == 6  # MXQ_ERR_WORKSPACE, nothing queued
    assert mxq.mxq_check(mxq._stream()) == 0
