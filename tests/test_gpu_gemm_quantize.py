"""Parity of the GEMM whose epilogue writes row-wise MX codes of the product.

Exact products: with integer-valued codes and one scale per row of A and
of B, every partial sum is an integer times a power of two below 2^24, so
the fp32 accumulators hold the exact product in any order.  There the
epilogue's codes and scales must equal the oracle's MX quantization of the
exact product bit for bit (ties to even included).

General products: the GPU accumulates in fp32 in its own order, so its
product differs from the oracle's fp64 product by up to the GEMM bound
(2e-4 * sum|ab|), and a value next to a rounding boundary may legitimately
round either way.  The check therefore takes what is unique and tests the
rest for validity:

* each block's scale must lie between the scales of the smallest and the
  largest block amax the bound allows (and equal it when those agree);
* under that scale, each element's decoded value must lie between the
  oracle's roundings of the two ends of its bound interval (rounding is
  monotone), and equal the oracle's code wherever both ends round alike.

Most elements and blocks are decided uniquely (at least 75%: products of
E2M1 codes over short K often land exactly on a rounding midpoint, which
the bound leaves open); the test asserts that too, so it cannot pass
vacuously.
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


def _scale_bytes(amax, fmt):
    blk = np.zeros(amax.shape + (32,))
    blk[..., 0] = amax
    return O.shared_exponent(blk, fmt)[0].astype(np.int64)


def check_epilogue_codes(codes, scales, ref, S, fmt_out, min_unique=0.75):
    codes, scales = np.asarray(codes), np.asarray(scales).astype(np.int64)
    M, N = ref.shape
    tol = REL * S
    rb, tb = ref.reshape(M, N // 32, 32), tol.reshape(M, N // 32, 32)
    s_lo = _scale_bytes(np.max(np.maximum(np.abs(rb) - tb, 0.0), axis=2), fmt_out)
    s_hi = _scale_bytes(np.max(np.abs(rb) + tb, axis=2), fmt_out)
    assert np.all((scales >= s_lo) & (scales <= s_hi)), "a block scale outside the bound"
    assert np.mean(s_lo == s_hi) >= min_unique
    e = (scales - 127)[..., None]
    lo, hi = np.ldexp(rb - tb, -e), np.ldexp(rb + tb, -e)
    q_lo, q_hi = O.round_to_element(lo, fmt_out), O.round_to_element(hi, fmt_out)
    c = O.unpack_e2m1(codes) if fmt_out == "e2m1" else codes
    c = c.reshape(M, N // 32, 32)
    got = O.decode_table(fmt_out)[c]
    bad = ~((got >= q_lo) & (got <= q_hi))
    assert not bad.any(), f"{bad.sum()} elements outside their rounding interval"
    unique = (q_lo == q_hi) & ((lo > 0) | (hi < 0) | (q_lo != 0))
    assert np.mean(unique) >= min_unique
    np.testing.assert_array_equal(c[unique], O.encode_element(q_lo[unique], fmt_out))


def _operands(M, N, K, fmt, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_t(3, size=(M, K)) * np.exp(rng.standard_normal(K))[None, :]).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    wb = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    A, sA = O.mx_quantize(xb, "row", fmt)
    B, sB = O.mx_quantize(wb, "row", fmt)
    return A, sA, B, sB


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _integer_operands(M, N, K, fmt, seed):
    # integer-valued codes in [-4, 4] and one E8M0 scale per row: exact
    # products (|C| <= 16 K 2^(sa + sb - 254) with 16 K < 2^24)
    rng = np.random.default_rng(seed)
    table = O.decode_table(fmt)
    ints = [c for c, v in enumerate(table) if np.isfinite(v) and v == int(v) and abs(v) <= 4]
    a = rng.choice(ints, size=(M, K)).astype(np.uint8)
    b = rng.choice(ints, size=(N, K)).astype(np.uint8)
    if fmt == "e2m1":
        a, b = O.pack_e2m1(a), O.pack_e2m1(b)
    sA = np.repeat(rng.integers(118, 136, size=(M, 1)), K // 32, axis=1).astype(np.uint8)
    sB = np.repeat(rng.integers(118, 136, size=(N, 1)), K // 32, axis=1).astype(np.uint8)
    return a, sA, b, sB


@pytest.mark.parametrize("fmt_in", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("fmt_out", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("shape", [(128, 256, 256), (200, 288, 1024), (384, 800, 2080)],
                         ids=lambda s: "x".join(map(str, s)))
def test_epilogue_codes_exact_products(fmt_in, fmt_out, shape):
    M, N, K = shape
    a, sA, b, sB = _integer_operands(M, N, K, fmt_in, seed=M + N + K)
    codes, scales = mxq.mx_gemm_quantize(_dev(a), _dev(sA), _dev(b), _dev(sB), fmt_in, M, N, K,
                                         out_fmt=fmt_out)
    mxq.check()
    ref, _ = O.mx_gemm_f64(a, sA, b, sB, fmt_in)
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)   # exact in fp32
    ec, es = O.mx_quantize(ref.astype(np.float32), "row", fmt_out)
    np.testing.assert_array_equal(to_np(scales), es)
    np.testing.assert_array_equal(to_np(codes), ec)


def test_epilogue_codes_exact_products_full_size_sampled():
    # 8192 x 14336 x 4096 (the MLP up-projection forward shape), exact
    # integer products, E4M3 codes; sampled rows checked in full
    M, N, K = 8192, 14336, 4096
    a, sA, b, sB = _integer_operands(M, N, K, "e4m3", seed=99)
    codes, scales = mxq.mx_gemm_quantize(_dev(a), _dev(sA), _dev(b), _dev(sB), "e4m3", M, N, K,
                                         out_fmt="e4m3")
    mxq.check()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.choice(M, 24, replace=False), [0, M - 1]]))
    ref, _ = O.mx_gemm_f64(a[rows], sA[rows], b, sB, "e4m3")
    ec, es = O.mx_quantize(ref.astype(np.float32), "row", "e4m3")
    r_t = torch.from_numpy(rows).cuda()
    np.testing.assert_array_equal(to_np(scales[r_t]), es)
    np.testing.assert_array_equal(to_np(codes[r_t]), ec)


SHAPES = [(128, 256, 128), (200, 288, 160), (64, 96, 96), (384, 800, 2080), (256, 512, 1024)]


@pytest.mark.parametrize("fmt_in", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("fmt_out", ["e4m3", "e2m1", "e5m2"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_epilogue_codes_small(fmt_in, fmt_out, shape):
    M, N, K = shape
    A, sA, B, sB = _operands(M, N, K, fmt_in, seed=M + 3 * N + K)
    codes, scales = mxq.mx_gemm_quantize(_dev(A), _dev(sA), _dev(B), _dev(sB), fmt_in, M, N, K,
                                         out_fmt=fmt_out)
    mxq.check()
    ref, S = O.mx_gemm_f64(A, sA, B, sB, fmt_in)
    check_epilogue_codes(to_np(codes), to_np(scales), ref, S, fmt_out)


def test_epilogue_codes_narrow_stores_and_determinism():
    # codes at a 16- but not 32-byte aligned address take the 128-bit store
    # path; scale rows of N/32 % 4 != 0 take the byte path; repeated calls
    # give identical bits
    M, N, K = 256, 544, 512
    A, sA, B, sB = _operands(M, N, K, "e4m3", seed=17)
    buf = torch.empty(M * N + 16, dtype=torch.uint8, device="cuda")
    codes = buf[16:].view(M, N)
    scales = torch.empty((M, N // 32), dtype=torch.uint8, device="cuda")
    dA, dsA, dB, dsB = _dev(A), _dev(sA), _dev(B), _dev(sB)
    mxq.mx_gemm_quantize(dA, dsA, dB, dsB, "e4m3", M, N, K, out_fmt="e4m3", out=(codes, scales))
    c2, s2 = mxq.mx_gemm_quantize(dA, dsA, dB, dsB, "e4m3", M, N, K, out_fmt="e4m3")
    mxq.check()
    assert torch.equal(codes, c2) and torch.equal(scales, s2)
    ref, S = O.mx_gemm_f64(A, sA, B, sB, "e4m3")
    check_epilogue_codes(to_np(codes), to_np(scales), ref, S, "e4m3")


def test_epilogue_argument_errors():
    t = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    s = mxq._stream()
    Q = mxq.mxq_gemm_quantize
    assert Q(p, p, p, p, 0, 128, 136, 64, 0, p, p, p, 1 << 16, s) == 1          # N % 32
    assert Q(p, p, p, p, 0, 128, 128, 64, 7, p, p, p, 1 << 16, s) == 1          # out_fmt
    assert Q(p, p, p, p, 0, 128, 128, 64, 0, p, None, p, 1 << 16, s) == 1       # scales
    assert Q(p, p, p, p, 0, 128, 128, 64, 0, p + 8, p, p, 1 << 16, s) == 2      # codes alignment
    assert Q(p, p, p, p, 0, 128, 128, 64, 0, p, p, p, 16, s) == 6               # workspace
    mxq.check()


def test_mlp_up_forward_epilogue_codes_full_size_sampled():
    # X 8192x4096 (row-wise E4M3) times W 4096x14336 given as K x N, the
    # epilogue writing E4M3 codes of the 8192x14336 product (the next
    # layer's forward operand); sampled rows x sampled 32-column blocks
    d = synth.mlp_up_forward()
    x, w = d["x"].cuda(), d["w"].cuda()
    M, K = x.shape
    N = w.shape[1]
    A, sA = mxq.mx_quantize(x, "row", "e4m3")
    B, sB = mxq.mx_quantize(w, "col", "e4m3")
    codes, scales = mxq.mx_gemm_quantize(A, sA, B, sB, "e4m3", M, N, K, out_fmt="e4m3")
    mxq.check()
    rng = np.random.default_rng(4321)
    rows = np.unique(np.concatenate([rng.choice(M, 48, replace=False), [0, M - 1]]))
    blks = np.unique(np.concatenate([rng.choice(N // 32, 12, replace=False), [0, N // 32 - 1]]))
    cols = (blks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    oA, osA = O.mx_quantize(bf16_to_f32_np(d["x"])[rows], "row", "e4m3")
    oB, osB = O.mx_quantize(bf16_to_f32_np(d["w"])[:, cols], "col", "e4m3")
    ref, S = O.mx_gemm_f64(oA, osA, oB, osB, "e4m3")
    r_t, c_t = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    b_t = torch.from_numpy(blks).cuda()
    got_c = to_np(codes[r_t][:, c_t])
    got_s = to_np(scales[r_t][:, b_t])
    # with K = 4096 and heavy cancellation the bound is wide next to the
    # E4M3 step, so fewer elements are decided uniquely
    check_epilogue_codes(got_c, got_s, ref, S, "e4m3", min_unique=0.5)


@pytest.mark.parametrize("fmt_in,fmt_out", [("e4m3", "e4m3"), ("e2m1", "e2m1"), ("e4m3", "e2m1")])
def test_epilogue_tc_scale_layouts_and_chaining(fmt_in, fmt_out):
    # tensor-core scale layout on the input side and on the output side:
    # the same codes, the same scales rearranged, and the output feeds the
    # next GEMM in place with results bitwise equal to the row-major path
    from tests.test_gpu_scales_tc import tc_from_rowmajor
    M, N, K = 200, 512, 512
    a, sA, b, sB = _integer_operands(M, N, K, fmt_in, seed=31)
    dA, dB = _dev(a), _dev(b)
    c_rm, s_rm = mxq.mx_gemm_quantize(dA, _dev(sA), dB, _dev(sB), fmt_in, M, N, K, out_fmt=fmt_out)
    tA = _dev(tc_from_rowmajor(sA, M, K))
    tB = _dev(tc_from_rowmajor(sB, N, K))
    c_tc, s_tc = mxq.mx_gemm_quantize(dA, tA, dB, tB, fmt_in, M, N, K, out_fmt=fmt_out,
                                      scale_layout="tc", out_scale_layout="tc")
    mxq.check()
    assert torch.equal(c_rm, c_tc)
    np.testing.assert_array_equal(to_np(s_tc), tc_from_rowmajor(to_np(s_rm), M, N))
    # next layer: Z = Y W2^T with Y the quantized product (K2 = N)
    N2 = 256
    w2 = synth.weight(N2, N, seed=5).cuda()
    w_rm = mxq.mx_quantize(w2, "row", fmt_out)
    w_tc = mxq.mx_quantize(w2, "row", fmt_out, scale_layout="tc")
    z_rm = mxq.mx_gemm(c_rm, s_rm, *w_rm, fmt_out, M, N2, N)
    z_tc = mxq.mx_gemm(c_tc, s_tc, *w_tc, fmt_out, M, N2, N, scale_layout="tc")
    mxq.check()
    assert torch.equal(z_rm, z_tc)


@pytest.mark.parametrize("in_layout,out_layout", [("rowmajor", "tc"), ("tc", "rowmajor")])
def test_epilogue_mixed_scale_layouts(in_layout, out_layout):
    from tests.test_gpu_scales_tc import tc_from_rowmajor
    M, N, K = 136, 256, 512
    a, sA, b, sB = _integer_operands(M, N, K, "e4m3", seed=41)
    if in_layout == "tc":
        sA, sB = tc_from_rowmajor(sA, M, K), tc_from_rowmajor(sB, N, K)
    codes, scales = mxq.mx_gemm_quantize(_dev(a), _dev(sA), _dev(b), _dev(sB), "e4m3", M, N, K,
                                         out_fmt="e4m3", scale_layout=in_layout,
                                         out_scale_layout=out_layout)
    mxq.check()
    a2, sA2, b2, sB2 = _integer_operands(M, N, K, "e4m3", seed=41)
    ref, _ = O.mx_gemm_f64(a2, sA2, b2, sB2, "e4m3")
    ec, es = O.mx_quantize(ref.astype(np.float32), "row", "e4m3")
    np.testing.assert_array_equal(to_np(codes), ec)
    exp_s = tc_from_rowmajor(es, M, N) if out_layout == "tc" else es
    np.testing.assert_array_equal(to_np(scales), exp_s)
