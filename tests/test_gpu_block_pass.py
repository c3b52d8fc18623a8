"""Parity of the decoder-block pass that bench.py times, at its full size.

The four Llama-3.1-8B linear layers at 8192 tokens run through the same
functions the benchmark uses (dual quantizers writing their scales in the
tensor cores' chunk layout, forward / dgrad MXFP8 GEMMs with bf16 output,
Hadamard-MXFP4 Wgrad with fp32 output, all reading those scales in place).  The oracle
quantizes only sampled rows and columns of the same bf16 inputs and
computes those outputs in fp64; every sampled output must meet the GEMM
bound (2e-4 * sum|ab|, plus 2^-8 |C| for bf16 outputs).
"""

import numpy as np
import pytest
import torch

import bench
from oracle import mx_oracle as O
from tests.libutil import bf16_to_f32_np, ensure_built, to_np

pytestmark = pytest.mark.gpu

REL = 2e-4


@pytest.fixture(scope="module")
def block():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    plan = bench.layer_plan(8192)
    layers = bench.build_device_state(plan, torch.device("cuda", 0))
    bench.run_step(layers)
    torch.cuda.synchronize()
    from precision_mx_quantize_gb300 import mxq
    mxq.check()
    yield layers
    del layers
    torch.cuda.empty_cache()


def _close(got, ref, S, bf16):
    tol = REL * S + (2.0 ** -8 * np.abs(ref) if bf16 else 0.0)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= tol), f"{(err > tol).sum()} of {err.size} outside the bound"


def _pick(n, rng, k=64):
    return np.unique(np.concatenate([rng.choice(n, size=min(k, n), replace=False), [0, n - 1]]))


@pytest.mark.parametrize("layer", [0, 1, 2, 3], ids=["qkv", "o", "gate_up", "down"])
def test_block_pass_layer(block, layer):
    st = block[layer]
    h = st["host"]
    T, fin, fout = st["L"]["T"], st["L"]["fin"], st["L"]["fout"]
    rng = np.random.default_rng(100 + layer)
    x = bf16_to_f32_np(h["x"])
    w = bf16_to_f32_np(h["w"])
    dy = bf16_to_f32_np(h["dy"])
    t_rows, o_rows, i_rows = _pick(T, rng), _pick(fout, rng), _pick(fin, rng)

    # forward Y = X W^T (row-wise E4M3 operands), bf16 out
    A, sA = O.mx_quantize(x[t_rows], "row", "e4m3")
    B, sB = O.mx_quantize(w[o_rows], "row", "e4m3")
    ref, S = O.mx_gemm_f64(A, sA, B, sB, "e4m3")
    got = to_np(st["y"][torch.from_numpy(t_rows).cuda()][:, torch.from_numpy(o_rows).cuda()].float())
    _close(got, ref, S, bf16=True)

    # dgrad dX = dY W: A row-wise E4M3(dY), B column-wise E4M3(W) -> [in][out]
    A, sA = O.mx_quantize(dy[t_rows], "row", "e4m3")
    B, sB = O.mx_quantize(np.ascontiguousarray(w[:, i_rows]), "col", "e4m3")
    ref, S = O.mx_gemm_f64(A, sA, B, sB, "e4m3")
    got = to_np(st["dx"][torch.from_numpy(t_rows).cuda()][:, torch.from_numpy(i_rows).cuda()].float())
    _close(got, ref, S, bf16=True)

    # Wgrad dW = (H dY)^T (H X): column-wise Hadamard E2M1 along tokens, fp32 out
    A, sA = O.hadamard_mx_quantize(np.ascontiguousarray(dy[:, o_rows]), "col", "e2m1")
    B, sB = O.hadamard_mx_quantize(np.ascontiguousarray(x[:, i_rows]), "col", "e2m1")
    ref, S = O.mx_gemm_f64(A, sA, B, sB, "e2m1")
    got = to_np(st["dw"][torch.from_numpy(o_rows).cuda()][:, torch.from_numpy(i_rows).cuda()])
    _close(got, ref, S, bf16=False)

    # the quantizer outputs the GEMMs consumed are the oracle's, bit for bit
    # (scales in the tensor cores' chunk layout: byte (line, block) of chunk
    # (line / 128) * (blocked / 128) + block / 4 at (line % 32) * 16 +
    # ((line % 128) / 32) * 4 + block % 4)
    xr, sxr, xc, sxc = st["xq"]
    ec, es = O.mx_quantize(x[t_rows], "row", "e4m3")
    np.testing.assert_array_equal(to_np(xr[torch.from_numpy(t_rows).cuda()]), ec)
    np.testing.assert_array_equal(_tc_rows(to_np(sxr), t_rows, fin), es)
    ec, es = O.hadamard_mx_quantize(np.ascontiguousarray(x[:, i_rows]), "col", "e2m1")
    np.testing.assert_array_equal(to_np(xc[torch.from_numpy(i_rows).cuda()]), ec)
    np.testing.assert_array_equal(_tc_rows(to_np(sxc), i_rows, T), es)


def _tc_rows(buf, lines, blocked):
    """Row-major scales of the given lines, read out of a chunk-layout buffer."""
    kcs = blocked // 128
    out = np.zeros((len(lines), blocked // 32), np.uint8)
    for i, line in enumerate(lines):
        for b in range(blocked // 32):
            chunk = (line // 128) * kcs + b // 4
            out[i, b] = buf[chunk * 512 + (line % 32) * 16 + ((line % 128) // 32) * 4 + b % 4]
    return out
