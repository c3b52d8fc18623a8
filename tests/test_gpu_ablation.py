"""Parity of the ablation quantizer (random-sign Hadamard rotation, stochastic
rounding) with the CPU oracle.

The random bits are Philox4x32-10 of each element's input index on both
sides, so codes and scales must match bit for bit: on ragged shapes in both
layouts, on the degenerate blocks, for seeds with high bits set, and for
element indices at and above 2^34, where the counter's high word is used.
"""

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O
from precision_mx_quantize_gb300 import mxq, synth
from tests.libutil import bf16_to_f32_np, ensure_built, to_np

pytestmark = pytest.mark.gpu

FMTS = ["e4m3", "e2m1", "e5m2"]
# (hadamard, sign mask, stochastic)
MODES = [(True, 0xB5C3A96E, False), (True, 0x0F0F3355, True), (False, 0, True), (True, 0, True)]
SEED = 0x0123456789ABCDEF


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _check(x, axis, fmt, had, mask, sr, seed=SEED):
    codes, scales = mxq.mx_quantize_ablation(x, axis, fmt, had, mask, sr, seed)
    mxq.check()
    ec, es = O.mx_quantize_ablation(bf16_to_f32_np(x), axis, fmt, had, mask, sr, seed)
    np.testing.assert_array_equal(to_np(scales), es)
    np.testing.assert_array_equal(to_np(codes), ec)
    return codes


def _mode_id(m):
    return f"had{int(m[0])}-mask{m[1]:08x}-sr{int(m[2])}"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES, ids=_mode_id)
@pytest.mark.parametrize("shape", [(1, 32), (33, 64), (200, 160), (257, 416)])
def test_rowwise_ablation_parity(fmt, mode, shape):
    x = synth.activation(*shape, seed=shape[0]).cuda()
    _check(x, "row", fmt, *mode)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES, ids=_mode_id)
@pytest.mark.parametrize("shape", [(32, 8), (64, 40), (160, 200), (288, 392)])
def test_colwise_ablation_parity(fmt, mode, shape):
    x = synth.activation(*shape, seed=shape[1]).cuda()
    _check(x, "col", fmt, *mode)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES, ids=_mode_id)
def test_ablation_special_values(fmt, mode):
    # zeros, NaN, +-Inf, huge and subnormal magnitudes, values at the format
    # maxima, blocks of all zeros and of subnormal maxima
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((128, 256)) * np.exp2(rng.integers(-30, 30, (128, 1)))).astype(np.float32)
    flat = x.reshape(-1)
    idx = rng.choice(flat.size, size=flat.size // 50, replace=False)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 3.0e38, -3.3e38, 2.0 ** -133,
                         -(2.0 ** -130), 1e-40, 448.0, 500.0, 6.0, 7.5, -5.0, 57344.0],
                        dtype=np.float32)
    flat[idx] = specials[rng.integers(0, len(specials), size=idx.size)]
    x[:32, :32] = 0.0
    x[64:96, :32] = 2.0 ** -130
    xb = torch.from_numpy(x).to(torch.bfloat16).cuda()
    _check(xb, "row", fmt, *mode)
    _check(xb, "col", fmt, *mode)


def test_reduces_to_the_deterministic_entry_points():
    x = synth.activation(96, 160, seed=3).cuda()
    for axis in ("row", "col"):
        a = mxq.mx_quantize_ablation(x, axis, "e2m1", True, 0, False, 5)
        b = mxq.hadamard_mx_quantize(x, axis, "e2m1")
        c = mxq.mx_quantize_ablation(x, axis, "e4m3", False, 0, False, 5)
        d = mxq.mx_quantize(x, axis, "e4m3")
        mxq.check()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        assert torch.equal(c[0], d[0]) and torch.equal(c[1], d[1])


def test_seed_determinism_and_dependence():
    x = synth.activation(512, 768, seed=5).cuda()
    a = mxq.mx_quantize_ablation(x, "col", "e2m1", True, 0x1234, True, 11)
    b = mxq.mx_quantize_ablation(x, "col", "e2m1", True, 0x1234, True, 11)
    c = mxq.mx_quantize_ablation(x, "col", "e2m1", True, 0x1234, True, 12)
    mxq.check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[1], c[1])              # block exponents are deterministic
    assert not torch.equal(a[0], c[0])          # the rounding is not


def test_full_size_wgrad_operand_sampled():
    # a 16384 x 8192 output gradient, column-wise random-sign Hadamard E2M1
    # with stochastic rounding (the Wgrad operand of the ablation); sampled
    # output rows (= input columns) against the oracle
    g = torch.Generator(device="cuda")
    g.manual_seed(8)
    T, F = 16384, 8192
    x = torch.randn(T, F, device="cuda", generator=g).to(torch.bfloat16)
    codes, scales = mxq.mx_quantize_ablation(x, "col", "e2m1", True, 0xA5A5F00F, True, SEED)
    mxq.check()
    rng = np.random.default_rng(9)
    cols = np.unique(np.concatenate([rng.choice(F, 24, replace=False), [0, F - 1]]))
    xs = bf16_to_f32_np(x[:, torch.from_numpy(cols).cuda()])
    for j, c in enumerate(cols):
        # input column c alone, with the random bits of its elements' indices
        # r * F + c in the full tensor
        ec, es = O.mx_quantize_ablation(xs[:, j:j + 1], "col", "e2m1", True, 0xA5A5F00F, True, SEED,
                                        first_col=int(c), total_cols=F)
        np.testing.assert_array_equal(to_np(scales[int(c):int(c) + 1]), es)
        np.testing.assert_array_equal(to_np(codes[int(c):int(c) + 1]), ec)


def test_counter_high_word_rows_past_2_to_34():
    # (2^17 + 64) x 2^17 bf16 (32 GiB): the last 64 rows hold element indices
    # >= 2^34, whose Philox counters have a non-zero high word
    R, C = (1 << 17) + 64, 1 << 17
    g = torch.Generator(device="cuda")
    g.manual_seed(12)
    x = torch.randn(R, C, device="cuda", dtype=torch.bfloat16, generator=g)
    codes, scales = mxq.mx_quantize_ablation(x, "row", "e4m3", True, 0x600DF00D, True, SEED)
    mxq.check()
    tail = bf16_to_f32_np(x[R - 64:])
    ec, es = O.mx_quantize_ablation(tail, "row", "e4m3", True, 0x600DF00D, True, SEED,
                                    first_row=R - 64, total_cols=C)
    np.testing.assert_array_equal(to_np(scales[R - 64:]), es)
    np.testing.assert_array_equal(to_np(codes[R - 64:]), ec)
    head = bf16_to_f32_np(x[:8])
    ec, es = O.mx_quantize_ablation(head, "row", "e4m3", True, 0x600DF00D, True, SEED,
                                    first_row=0, total_cols=C)
    np.testing.assert_array_equal(to_np(codes[:8]), ec)
    del x, codes, scales
    torch.cuda.empty_cache()
