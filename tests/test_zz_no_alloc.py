"""GPU test of mxq_gemm_noalloc, the GEMM entry point for callers that cannot
allocate device memory when they call (a plug-in that receives only its input
and output buffers from a host application owning the memory pool, or code
under a fixed memory budget).  Its scale scratch is a fixed buffer inside the
library instead of a caller workspace.

The file is named to be collected last.  It checks the entry point through
the C ABI against mxq_gemm (the entry point with a caller workspace) on two
calls in a row, and the rejection of problems larger than the fixed buffer.
"""

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq
from tests.libutil import ensure_built, to_np

pytestmark = pytest.mark.gpu

REL = 2e-4   # the GEMM tolerance of the parity tests: 2e-4 * sum_k |a_k b_k|


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


def _both(M, N, K, fmt, seed):
    A, sA, B, sB = _operands(M, N, K, fmt, seed)
    _, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
    d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (A, sA, B, sB)]
    f = mxq.E4M3 if fmt == "e4m3" else mxq.E2M1
    stream = mxq._stream()
    c_new = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = mxq.mxq_gemm_noalloc(d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), d[3].data_ptr(),
                              f, M, N, K, c_new.data_ptr(), mxq.OUT_F32, stream)
    assert st == 0, mxq.STATUS.get(st, st)
    c_ref = mxq.mx_gemm(d[0], d[1], d[2], d[3], fmt, M, N, K)
    assert mxq.mxq_check(stream) == 0
    return to_np(c_new), to_np(c_ref), S


def test_noalloc_matches_workspace_gemm_twice():
    # two calls in a row that share the fixed scratch: the second (smaller K,
    # other format) must not see the first one's leftovers
    for (M, N, K, fmt, seed) in [(384, 520, 2080, "e4m3", 1), (200, 264, 160, "e2m1", 2)]:
        new, ref, S = _both(M, N, K, fmt, seed)
        err = np.abs(new.astype(np.float64) - ref.astype(np.float64))
        assert np.all(err <= REL * S), (M, N, K, fmt)


def test_noalloc_rejects_problems_beyond_the_buffer():
    # (65536 + 65536) rows x 256 k-blocks of scales = 32 MiB > 16 MiB
    assert mxq.mxq_gemm_workspace_size(65536, 65536, 8192, mxq.E4M3) > 16 << 20
    p = torch.zeros(16, dtype=torch.uint8, device="cuda").data_ptr()
    st = mxq.mxq_gemm_noalloc(p, p, p, p, mxq.E4M3, 65536, 65536, 8192, p, mxq.OUT_F32,
                              mxq._stream())
    assert st == 6  # MXQ_ERR_WORKSPACE, nothing queued
    assert mxq.mxq_check(mxq._stream()) == 0
