"""Parity cases run against the bounds-checked build of the library.

Run as ``MXQ_BOUNDS_CHECKED=1 python -m tests.bounds_checked_cases`` (the
GPU test in test_gpu_bounds_checked.py does so in a subprocess).  In that
build every kernel checks each global index it computes against the extent
its arguments imply; a violation is recorded as MXQ_ERR_BOUNDS and the access
is skipped.  Every case below must report no error through mxq_check and
still match the CPU oracle: the small, ragged and degenerate shapes of the
parity tests, for the quantizers (single, one-pass, ablation), the
dequantizer and the GEMMs (both scale layouts, the quantizing epilogue).
Prints one JSON line with the number of cases and the errors found.
"""

import json
import sys

import numpy as np
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq, synth
from tests.libutil import ensure_built, to_np

FMTS = ["e4m3", "e2m1", "e5m2"]


def main():
    assert mxq.BOUNDS_CHECKED and mxq.LIB_PATH.endswith("libmxq_debug.so"), mxq.LIB_PATH
    ensure_built()
    errors, n = [], 0

    def checked(tag):
        nonlocal n
        n += 1
        st = mxq.mxq_check(mxq._stream())
        if st != 0:
            errors.append((tag, mxq.STATUS.get(st, st)))
        return st == 0

    # single-layout quantizers, ragged rows / columns / tails
    for (R, C) in [(1, 32), (33, 64), (257, 416)]:
        x = synth.normal_with_outliers((R, C), R).cuda()
        for fmt in FMTS:
            for had in (False, True):
                q = mxq.hadamard_mx_quantize if had else mxq.mx_quantize
                codes, sc = q(x, "row", fmt)
                if checked(f"row {R}x{C} {fmt} {had}"):
                    ec, es = O.quantize_any(x.float().cpu().numpy(), "row", fmt, had)
                    assert np.array_equal(to_np(codes), ec) and np.array_equal(to_np(sc), es)
    for (R, C) in [(32, 8), (96, 136), (288, 392)]:
        x = synth.normal_with_outliers((R, C), C).cuda()
        for fmt in FMTS:
            for had in (False, True):
                q = mxq.hadamard_mx_quantize if had else mxq.mx_quantize
                codes, sc = q(x, "col", fmt)
                if checked(f"col {R}x{C} {fmt} {had}"):
                    ec, es = O.quantize_any(x.float().cpu().numpy(), "col", fmt, had)
                    assert np.array_equal(to_np(codes), ec) and np.array_equal(to_np(sc), es)
    # one-pass quantizer, both scale layouts
    for (R, C) in [(96, 160), (384, 256)]:
        x = synth.activation(R, C, 7).cuda()
        for fr, hr, fc, hc in [("e4m3", False, "e2m1", True), ("e4m3", False, "e4m3", False),
                               ("e5m2", True, "e2m1", True)]:
            cr, sr, cc, scc = mxq.mx_quantize_dual(x, fr, hr, fc, hc)
            if checked(f"dual {R}x{C} {fr}{hr} {fc}{hc}"):
                xn = x.float().cpu().numpy()
                er, esr = O.quantize_any(xn, "row", fr, hr)
                ec, esc = O.quantize_any(xn, "col", fc, hc)
                assert np.array_equal(to_np(cr), er) and np.array_equal(to_np(sr), esr)
                assert np.array_equal(to_np(cc), ec) and np.array_equal(to_np(scc), esc)
    x = synth.activation(256, 512, 3).cuda()
    mxq.mx_quantize_dual(x, "e4m3", False, "e2m1", True, scale_layout="tc")
    checked("dual tc 256x512")
    # ablation (random-sign rotation, stochastic rounding)
    x = synth.activation(96, 160, 5).cuda()
    for axis in ("row", "col"):
        codes, sc = mxq.mx_quantize_ablation(x, axis, "e2m1", True, 0xA5A5F00F, True, 11)
        if checked(f"ablation {axis}"):
            ec, es = O.mx_quantize_ablation(x.float().cpu().numpy(), axis, "e2m1", True,
                                            0xA5A5F00F, True, 11)
            assert np.array_equal(to_np(codes), ec) and np.array_equal(to_np(sc), es)
    # dequantizer, ragged column counts
    for (R, C) in [(64, 37), (96, 130), (160, 258)]:
        g = torch.Generator().manual_seed(R + C)
        for fmt in FMTS:
            cb = R // 2 if fmt == "e2m1" else R
            codes = torch.randint(0, 256, (C, cb), dtype=torch.uint8, generator=g)
            scales = torch.randint(90, 170, (C, R // 32), dtype=torch.uint8, generator=g)
            for od in (torch.float32, torch.bfloat16):
                got = mxq.mx_dequantize(codes.cuda(), scales.cuda(), R, C, "col", fmt, od)
                if checked(f"dequant col {R}x{C} {fmt}"):
                    exp = O.mx_dequantize(codes.numpy(), scales.numpy(), fmt,
                                          "f32" if od == torch.float32 else "bf16").T
                    assert np.array_equal(to_np(got.float()), exp, equal_nan=True)
    x = synth.normal_with_outliers((96, 160), 1).cuda()
    for fmt in FMTS:
        c, s = mxq.mx_quantize(x, "row", fmt)
        got = mxq.mx_dequantize(c, s, 96, 160, "row", fmt)
        if checked(f"dequant row {fmt}"):
            assert np.array_equal(to_np(got), O.mx_dequantize(to_np(c), to_np(s), fmt))
    # GEMMs: ragged M, N, K; row-major scales (re-layout pass) and chunk layout
    for (M, N, K, fmt) in [(200, 264, 160, "e2m1"), (384, 520, 2080, "e4m3"),
                           (257, 300, 4160, "e5m2"), (1, 8, 64, "e2m1")]:
        rng = np.random.default_rng(M + N + K)
        a = rng.standard_t(3, size=(M, K)).astype(np.float32)
        b = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
        A, sA = O.mx_quantize(a, "row", fmt)
        B, sB = O.mx_quantize(b, "row", fmt)
        ref, S = O.mx_gemm_f64(A, sA, B, sB, fmt)
        d = [torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in (A, sA, B, sB)]
        C_ = mxq.mx_gemm(*d, fmt, M, N, K)
        if checked(f"gemm {M}x{N}x{K} {fmt}"):
            assert np.all(np.abs(to_np(C_).astype(np.float64) - ref) <= 2e-4 * S)
    xa = synth.activation(256, 512, 1).cuda()
    xb = synth.weight(384, 512, 2).cuda()
    A, sA = mxq.mx_quantize(xa, "row", "e4m3", scale_layout="tc")
    B, sB = mxq.mx_quantize(xb, "row", "e4m3", scale_layout="tc")
    mxq.mx_gemm(A, sA, B, sB, "e4m3", 256, 384, 512, scale_layout="tc")
    checked("gemm tc")
    # chunk-layout output scales need N % 128 (E4M3) -- N is 384
    mxq.mx_gemm_quantize(A, sA, B, sB, "e4m3", 256, 384, 512, out_fmt="e4m3",
                         scale_layout="tc", out_scale_layout="tc")
    checked("gemm quantize tc")
    print(json.dumps({"cases": n, "errors": errors}))
    return 0 if not errors else 1


if __name__ == "__main__":
    sys.exit(main())
