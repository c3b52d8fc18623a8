"""CPU oracle for the MX quantized-training hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
table or constant with the CUDA library; the two meet only in the seeded
input generators.

It is written to be read against its sources, not to be fast:

* "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題" (hzrcw.cc), §02: MXFP4 splits
  a tensor into small blocks, each with its own dynamic scaling exponent; the
  weight-gradient (Wgrad) path is quantized after a fixed, deterministic
  Hadamard rotation (an orthogonal transform that does not change between
  steps).  §02 also names the three GEMM roles: forward, activation gradient
  (dgrad) and weight gradient (Wgrad).
* "MindSpeed LLM FSDP2量化特性：低比特大模型训练完全指南", "第 1 步：选择量化配方":
  MX granularity with block size 32 and E4M3 elements for inputs, weights
  and gradients (recipe ``dynamic_MX-1-1-32_E4M3_E4M3_E4M3``).
* "Lumen：AMD原生大模型量化训练框架的技术突破与实践", §1 "多精度量化格式支持":
  FP8 E4M3, MXFP8 and FP4 as the formats of quantized training.

The pages fix neither bit layouts nor rounding.  Those come from the public
OCP Microscaling Formats (MX) v1.0 and OCP 8-bit Floating Point
specifications, restated here from their definitions:

* E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
  infinities; S.1111.111 is NaN; largest finite magnitude 1.75 * 2**8 = 448.
* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
  {0, .5, 1, 1.5, 2, 3, 4, 6}; largest 6 = 1.5 * 2**2.
* E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits, IEEE-style
  specials: S.11111.00 is infinity, S.11111.xx (xx != 0) NaN; largest
  finite magnitude 1.75 * 2**15 = 57344.  The other MXFP8 element type
  ("Lumen：AMD原生大模型量化训练框架的技术突破与实践", §1 names FP8 E4M3 and E5M2).
* E8M0 shared scale: an unsigned biased exponent, value 2**(s - 127); 0xFF
  is NaN.
* The shared exponent of a block is floor(log2(amax)) - emax_elem, where
  emax_elem is the exponent of the element format's largest normal (8 for
  E4M3, 2 for E2M1, 15 for E5M2).  Elements are x / 2**e rounded to nearest, ties to
  even, clamped to the largest finite element magnitude.

Readings taken where the sources are silent (each is also listed in the
design notes):

R1  amax == 0 gives scale byte 0x00 (log2 0 = -inf, clamped to -127) and
    every element code +0 or -0.
R2  a block holding NaN or +-Inf gets scale 0xFF and all element codes 0.
R3  the exponent uses floor, so block maxima in (448, 512), (6, 8) or
    (57344, 65536) times 2**e saturate to the largest element (E5M2 elements
    saturate too: they never become infinity).
R4  signs are kept: a negative value that rounds to zero encodes as -0
    (0x80 for E4M3, 0x8 for E2M1).
R5  E2M1 codes are packed two per byte, the even element in the low nibble.
R6  the column-wise layout quantizes 32-blocks that run down the rows and
    stores the result transposed: output row c holds input column c.
R7  the Hadamard rotation is the natural-order (Sylvester) 32-point
    transform, computed as five radix-2 stages h = 1, 2, 4, 8, 16 in fp32
    with every add and subtract rounded to nearest (no fused operations),
    then one multiply by c = RN_fp32(2**-2.5); the quantizer consumes the
    fp32 result without rounding it to bf16.
R8  the GEMM is C[m, n] = sum_k dec(A[m, k]) * dec(B[n, k]) over the exactly
    dequantized operands (both K-major, "TN"), accumulated in fp64.
R9  the ablation's random Hadamard rotation is H_32 * diag(d): one random
    sign vector d (a 32-bit mask drawn by the caller) shared by every block
    of the tensor, applied to the inputs before the fixed butterflies.
R10 stochastic rounding rounds |v| up to the next grid point with
    probability frac(|v| / q) (q the grid step at |v|), decided with 32
    random bits per element: up iff bits < floor(frac * 2**32).  The block
    exponent is the deterministic one (from the block amax).
R11 the random bits of the element at input row r, column c come from
    Philox4x32-10 keyed by the seed, counter (r * cols + c) // 4, word
    (r * cols + c) % 4, for either output layout.

Every function's citation is in its docstring.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32  # MX block size ("MindSpeed LLM FSDP2量化特性", 第 1 步: MX-1-1-32)

# --------------------------------------------------------------------------
# Element formats: parameters of the bit layouts (OCP FP8 / OCP MX v1.0)
# --------------------------------------------------------------------------

E4M3 = "e4m3"
E2M1 = "e2m1"
E5M2 = "e5m2"

_FMT = {
    # ebits, mbits, bias, max finite magnitude, emax_elem, total bits
    E4M3: dict(ebits=4, mbits=3, bias=7, maxval=448.0, emax=8, bits=8),
    E2M1: dict(ebits=2, mbits=1, bias=1, maxval=6.0, emax=2, bits=4),
    E5M2: dict(ebits=5, mbits=2, bias=15, maxval=57344.0, emax=15, bits=8),
}


def fmt_params(fmt: str) -> dict:
    return _FMT[fmt]


def decode_element(code: int, fmt: str) -> float:
    """Value of one element code, straight from the bit formula.

    OCP MX v1.0 element types: normal (E > 0) is (1 + m / 2**mbits) *
    2**(E - bias); subnormal (E == 0) is m / 2**mbits * 2**(1 - bias).
    E4M3 "fn": only S.1111.111 is NaN (no infinities).  E5M2: an all-ones
    exponent is infinity (mantissa 0) or NaN (mantissa != 0).
    """
    p = _FMT[fmt]
    nb, mb = p["bits"], p["mbits"]
    sign = (code >> (nb - 1)) & 1
    E = (code >> mb) & ((1 << p["ebits"]) - 1)
    m = code & ((1 << mb) - 1)
    if fmt == E4M3 and E == 15 and m == 7:
        return float("nan")
    if fmt == E5M2 and E == 31:
        return float("nan") if m else (float("-inf") if sign else float("inf"))
    if E == 0:
        mag = (m / (1 << mb)) * 2.0 ** (1 - p["bias"])
    else:
        mag = (1.0 + m / (1 << mb)) * 2.0 ** (E - p["bias"])
    return -mag if sign else mag


def decode_table(fmt: str) -> np.ndarray:
    """All code values of a format, index = code (256 for E4M3/E5M2, 16 for E2M1)."""
    n = 1 << _FMT[fmt]["bits"]
    return np.array([decode_element(c, fmt) for c in range(n)], dtype=np.float64)


# --------------------------------------------------------------------------
# Rounding a real value onto the element grid (round to nearest, ties to
# even, saturating, sign kept)
# --------------------------------------------------------------------------

def round_to_element(v: np.ndarray, fmt: str) -> np.ndarray:
    """Round exact float64 values onto the element format's grid.

    OCP MX v1.0: conversion to an element is round-to-nearest-even with
    saturation to the largest finite magnitude (readings R3, R4).  On the
    binade [2**k, 2**(k+1)) the grid step is 2**(k - mbits); below the
    smallest normal 2**(1 - bias) the step is that of the subnormals.  A tie
    rounds to the even multiple of the step, i.e. the code whose last
    mantissa bit is 0.
    """
    p = _FMT[fmt]
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    emin = 1 - p["bias"]
    _, ex = np.frexp(a)                      # a = f * 2**ex, f in [0.5, 1)
    k = np.maximum(ex - 1, emin)             # floor(log2 a), at least emin
    k = np.where(a == 0, emin, k)
    step = np.ldexp(1.0, (k - p["mbits"]).astype(np.int64))
    r = np.rint(a / step) * step             # np.rint: halves go to even
    r = np.minimum(r, p["maxval"])           # saturate
    return np.where(np.signbit(v), -r, r)


def encode_element(r: np.ndarray, fmt: str) -> np.ndarray:
    """Code of a value that already lies on the element grid (sign kept)."""
    p = _FMT[fmt]
    r = np.asarray(r, dtype=np.float64)
    a = np.abs(r)
    emin = 1 - p["bias"]
    _, ex = np.frexp(a)
    k = ex - 1
    normal = (a != 0) & (k >= emin)
    E = np.where(normal, k + p["bias"], 0)
    kk = np.where(normal, k, emin)
    m = a / np.ldexp(1.0, (kk - p["mbits"]).astype(np.int64))
    m = np.where(normal, m - (1 << p["mbits"]), m)
    m = np.nan_to_num(m).astype(np.int64)   # NaN blocks are zeroed by the caller
    sign = np.signbit(r).astype(np.int64)
    nb = p["bits"]
    code = (sign << (nb - 1)) | (E.astype(np.int64) << p["mbits"]) | m
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# Shared block exponent (E8M0)
# --------------------------------------------------------------------------

def shared_exponent(blocks: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """Per-block E8M0 scale byte and the unbiased exponent used for scaling.

    "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §02: every block carries its
    own dynamically chosen exponent.  OCP MX v1.0: e = floor(log2 amax) -
    emax_elem, clamped to the E8M0 range [-127, 127]; scale byte e + 127.
    floor(log2) is read off the binary exponent (frexp), never a logarithm.
    blocks: [..., 32] float array (bf16 values widened, or fp32).
    Returns (scale_u8 [...], e_int64 [...]); NaN/Inf blocks give 0xFF (R2),
    all-zero blocks 0x00 (R1).
    """
    p = _FMT[fmt]
    b = np.asarray(blocks, dtype=np.float64)
    bad = ~np.all(np.isfinite(b), axis=-1)
    amax = np.max(np.abs(np.where(np.isfinite(b), b, 0.0)), axis=-1)
    _, ex = np.frexp(amax)
    floor_log2 = ex - 1
    e = np.where(amax == 0, -127, floor_log2 - p["emax"])
    e = np.clip(e, -127, 127).astype(np.int64)
    s = (e + 127).astype(np.int64)
    s = np.where(bad, 255, s)
    return s.astype(np.uint8), e


# --------------------------------------------------------------------------
# Quantize / dequantize
# --------------------------------------------------------------------------

def _quantize_rows(x: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """Row-wise MX quantization: 32-blocks run along the last axis.

    x: [R, C] float32/float64 values (C % 32 == 0).
    Returns codes [R, C] uint8 (one code per element, unpacked) and
    scales [R, C // 32] uint8.
    """
    R, C = x.shape
    assert C % BLOCK == 0
    blocks = np.asarray(x, dtype=np.float64).reshape(R, C // BLOCK, BLOCK)
    s, e = shared_exponent(blocks, fmt)
    v = np.ldexp(blocks, -e[..., None])      # exact: a power-of-two scaling
    codes = encode_element(round_to_element(v, fmt), fmt)
    codes = np.where((s == 255)[..., None], np.uint8(0), codes)
    return codes.reshape(R, C), s


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis, even index in the low nibble (R5)."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def mx_quantize(x: np.ndarray, axis: str, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """MX quantization of a [rows, cols] tensor.

    axis == "row": blocks of 32 along the columns; codes [R, C] (E4M3) or
    [R, C/2] (E2M1, packed), scales [R, C/32].
    axis == "col": blocks of 32 along the rows, stored transposed (R6):
    codes [C, R] or [C, R/2], scales [C, R/32] -- the copy that the Wgrad
    GEMM consumes ("AMD顛覆行業認知！…", §02).
    """
    x = np.asarray(x)
    src = x if axis == "row" else x.T
    codes, s = _quantize_rows(src, fmt)
    if fmt == E2M1:
        codes = pack_e2m1(codes)
    return np.ascontiguousarray(codes), np.ascontiguousarray(s)


def element_values(codes: np.ndarray, fmt: str) -> np.ndarray:
    """float64 value of each (unpacked for E2M1) element code."""
    table = decode_table(fmt)
    c = unpack_e2m1(codes) if fmt == E2M1 else np.asarray(codes, dtype=np.uint8)
    return table[c]


def dequantize_f64(codes: np.ndarray, scales: np.ndarray, fmt: str) -> np.ndarray:
    """Exact value of every element: dec(code) * 2**(s - 127); s == 0xFF is NaN.

    OCP MX v1.0: the value of an MX element is the product of the shared
    scale and the element value.  Layout is that of the codes (row-wise
    or transposed), blocks along the last axis.
    """
    vals = element_values(codes, fmt)
    R, C = vals.shape
    s = np.asarray(scales, dtype=np.int64).reshape(R, C // BLOCK)
    sc = np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))
    return (vals.reshape(R, C // BLOCK, BLOCK) * sc[..., None]).reshape(R, C)


def mx_dequantize(codes, scales, fmt: str, out: str = "f32") -> np.ndarray:
    """Dequantize to fp32 (exact; overflow to inf) or to bf16 (RNE of that fp32).

    Returns a float32 array; for out == "bf16" it holds bf16-representable
    values (rounded to nearest even by torch's CPU cast).
    """
    with np.errstate(over="ignore", invalid="ignore"):
        f32 = dequantize_f64(codes, scales, fmt).astype(np.float32)
    if out == "f32":
        return f32
    import torch  # plain CPU cast: round to nearest even
    return torch.from_numpy(f32).to(torch.bfloat16).to(torch.float32).numpy()


# --------------------------------------------------------------------------
# Fixed 32-point Hadamard rotation
# --------------------------------------------------------------------------

def fwht_scale(dtype=np.float32):
    """c = 2**-2.5 rounded once to the working precision (R7)."""
    return dtype(2.0 ** -2.5)


def fwht32(blocks: np.ndarray, dtype=np.float32) -> np.ndarray:
    """Normalized natural-order 32-point Walsh-Hadamard transform of each block.

    "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §02: one fixed orthogonal
    rotation applied identically everywhere (deterministic, no random signs).
    Steps (R7): radix-2 stages with half-width h = 1, 2, 4, 8, 16; in each,
    for every j with (j & h) == 0, (a[j], a[j+h]) <- (a[j] + a[j+h],
    a[j] - a[j+h]), each result rounded to ``dtype``; then every entry times
    c = RN(2**-2.5) = 1/sqrt(32).  blocks: [..., 32].
    """
    a = np.array(blocks, dtype=dtype, copy=True)
    lead = a.shape[:-1]
    h = 1
    while h < BLOCK:
        a = a.reshape(lead + (BLOCK // (2 * h), 2, h))
        lo = a[..., 0, :]
        hi = a[..., 1, :]
        a = np.stack([lo + hi, lo - hi], axis=-2)  # same dtype: one rounding each
        h *= 2
    a = a.reshape(lead + (BLOCK,))
    return a * fwht_scale(dtype)


def hadamard_matrix(n: int = BLOCK) -> np.ndarray:
    """Sylvester Hadamard matrix H[i, j] = (-1)**popcount(i & j) (integer)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    pc = np.vectorize(lambda t: bin(int(t)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def hadamard_rotate(x: np.ndarray, axis: str, dtype=np.float32) -> np.ndarray:
    """Apply fwht32 to every 32-block along the quantization axis of [R, C] x."""
    x = np.asarray(x)
    if axis == "row":
        R, C = x.shape
        return fwht32(x.reshape(R, C // BLOCK, BLOCK), dtype).reshape(R, C)
    return hadamard_rotate(x.T, "row", dtype).T


def hadamard_mx_quantize(x: np.ndarray, axis: str, fmt: str):
    """Rotate each 32-block with fwht32 (fp32), then MX-quantize the fp32 result.

    "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §02: the deterministic
    Hadamard rotation precedes the MXFP4 quantization of the Wgrad operands.
    """
    src = np.asarray(x, dtype=np.float32)
    src = src if axis == "row" else src.T
    y = hadamard_rotate(src, "row", np.float32)
    codes, s = _quantize_rows(y, fmt)
    if fmt == E2M1:
        codes = pack_e2m1(codes)
    return np.ascontiguousarray(codes), np.ascontiguousarray(s)


def quantize_any(x, axis: str, fmt: str, hadamard: bool):
    return hadamard_mx_quantize(x, axis, fmt) if hadamard else mx_quantize(x, axis, fmt)


# --------------------------------------------------------------------------
# Block-scaled GEMM over the dequantized operands
# --------------------------------------------------------------------------

def mx_gemm_f64(A, sA, B, sB, fmt: str):
    """C = A_deq @ B_deq^T and S = |A_deq| @ |B_deq|^T in fp64 (R8).

    "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §02-§03: forward, dgrad and
    Wgrad GEMMs run on MX codes; their exact value is the product of the
    dequantized operands.  A: [M, K] codes (packed [M, K/2] for E2M1),
    sA [M, K/32]; B likewise with N rows.  Returns (C, S), both [M, N].
    """
    a = dequantize_f64(A, sA, fmt)
    b = dequantize_f64(B, sB, fmt)
    return a @ b.T, np.abs(a) @ np.abs(b).T


def mx_gemm_f64_rows(A, sA, B, sB, fmt: str, rows, cols):
    """The same product restricted to C[rows][:, cols] (rows and cols index arrays)."""
    a = dequantize_f64(np.asarray(A)[rows], np.asarray(sA)[rows], fmt)
    b = dequantize_f64(np.asarray(B)[cols], np.asarray(sB)[cols], fmt)
    return a @ b.T, np.abs(a) @ np.abs(b).T


# --------------------------------------------------------------------------
# Ablation: random-sign Hadamard rotation and stochastic rounding
# --------------------------------------------------------------------------
# "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §01: the approaches the paper
# argues against -- random Hadamard rotations and stochastic rounding, which
# add randomness to the quantization error.  They are built here as an
# ablation of the deterministic path.
#
# Random numbers come from Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
# "Parallel random numbers: as easy as 1, 2, 3", SC 2011), a counter-based
# generator both sides implement from that definition.  The element at
# linear index i of the input tensor (row-major, i = r * cols + c, whatever
# the output layout) uses word i % 4 of Philox(counter = (i // 4 low 32 bits,
# i // 4 high 32 bits, 0, 0), key = (seed low 32 bits, seed high 32 bits)).

_PHILOX_M0, _PHILOX_M1 = 0xD2511F53, 0xCD9E8D57   # round multipliers
_PHILOX_W0, _PHILOX_W1 = 0x9E3779B9, 0xBB67AE85   # key increments (golden ratio, sqrt(3)-1)


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on arrays: ctr [..., 4], key [..., 2] (uint32)."""
    c = [np.asarray(ctr[..., i], dtype=np.uint64) for i in range(4)]
    k0 = np.asarray(key[..., 0], dtype=np.uint64)
    k1 = np.asarray(key[..., 1], dtype=np.uint64)
    mask = np.uint64(0xFFFFFFFF)
    for rnd in range(10):
        p0 = np.uint64(_PHILOX_M0) * c[0]        # exact 64-bit products of 32-bit words
        p1 = np.uint64(_PHILOX_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        if rnd < 9:
            k0 = (k0 + np.uint64(_PHILOX_W0)) & mask
            k1 = (k1 + np.uint64(_PHILOX_W1)) & mask
    return np.stack([x.astype(np.uint32) for x in c], axis=-1)


def element_random_bits(seed: int, index: np.ndarray) -> np.ndarray:
    """32 random bits for each element linear index (see the rule above)."""
    idx = np.asarray(index, dtype=np.uint64)
    block = idx >> np.uint64(2)
    ctr = np.zeros(idx.shape + (4,), dtype=np.uint32)
    ctr[..., 0] = (block & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    ctr[..., 1] = (block >> np.uint64(32)).astype(np.uint32)
    key = np.zeros(idx.shape + (2,), dtype=np.uint32)
    key[..., 0] = np.uint32(seed & 0xFFFFFFFF)
    key[..., 1] = np.uint32((seed >> 32) & 0xFFFFFFFF)
    words = philox4x32_10(ctr, key)
    return np.take_along_axis(words, (idx & np.uint64(3)).astype(np.int64)[..., None], axis=-1)[..., 0]


def stochastic_round_to_element(v: np.ndarray, fmt: str, r: np.ndarray) -> np.ndarray:
    """Round exact float64 values onto the element grid stochastically.

    With lo <= |v| < hi the neighbouring grid points (step q, as in
    round_to_element), F = floor(frac(|v| / q) * 2^32) and r the element's 32
    random bits: the magnitude rounds up to hi when r < F, else down to lo,
    so P(up) = (|v| - lo) / q up to 2^-32.  Values on the grid stay; the
    result saturates at the largest finite magnitude; the sign is kept.
    """
    p = _FMT[fmt]
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    emin = 1 - p["bias"]
    _, ex = np.frexp(a)
    k = np.maximum(ex - 1, emin)
    k = np.where(a == 0, emin, k)
    step = np.ldexp(1.0, (k - p["mbits"]).astype(np.int64))
    t = a / step                                   # exact power-of-two scaling
    lo = np.floor(t)
    F = np.floor((t - lo) * 2.0 ** 32)             # exact: the fraction has few bits
    up = np.asarray(r, dtype=np.float64) < F
    mag = np.where(up, lo + 1.0, lo) * step
    mag = np.minimum(mag, p["maxval"])
    return np.where(np.signbit(v), -mag, mag)


def apply_sign_mask(blocks: np.ndarray, sign_mask: int) -> np.ndarray:
    """Negate element i of every 32-block where bit i of sign_mask is set (exact)."""
    b = np.asarray(blocks)
    d = np.array([-1.0 if (sign_mask >> i) & 1 else 1.0 for i in range(BLOCK)], dtype=b.dtype)
    return b * d


def mx_quantize_ablation(x, axis: str, fmt: str, hadamard: bool, sign_mask: int,
                         stochastic: bool, seed: int, first_row: int = 0, first_col: int = 0,
                         total_cols=None):
    """MX quantization with the ablation's randomness.

    hadamard: rotate each block by H_32 * diag(d), d_i = -1 where bit i of
    sign_mask is set (a random diagonal drawn by the caller); sign_mask = 0 is
    the deterministic rotation.  stochastic: element codes by
    stochastic_round_to_element with Philox bits of each element's input
    index; else round to nearest even.  The block exponent is chosen exactly
    as in mx_quantize (from the rotated block's amax).

    first_row, first_col, total_cols: x may be the window of a larger
    row-major tensor (total_cols columns) whose top-left element is
    (first_row, first_col); the random bits then follow each element's index
    in that tensor.
    """
    xf = np.asarray(x, dtype=np.float32)
    R, C = xf.shape
    ncol = C if total_cols is None else int(total_cols)
    idx = ((np.uint64(first_row) + np.arange(R, dtype=np.uint64))[:, None] * np.uint64(ncol)
           + np.uint64(first_col) + np.arange(C, dtype=np.uint64)[None, :])
    src, sidx = (xf, idx) if axis == "row" else (xf.T, idx.T)
    rows, cols = src.shape
    blocks = src.reshape(rows, cols // BLOCK, BLOCK)
    if hadamard:
        blocks = fwht32(apply_sign_mask(blocks, sign_mask), np.float32)
    s, e = shared_exponent(blocks, fmt)
    v = np.ldexp(np.asarray(blocks, dtype=np.float64), -e[..., None])
    if stochastic:
        r = element_random_bits(seed, np.ascontiguousarray(sidx).reshape(rows, cols // BLOCK, BLOCK))
        q = stochastic_round_to_element(v, fmt, r)
    else:
        q = round_to_element(v, fmt)
    codes = encode_element(q, fmt)
    codes = np.where((s == 255)[..., None], np.uint8(0), codes).reshape(rows, cols)
    if fmt == E2M1:
        codes = pack_e2m1(codes)
    return np.ascontiguousarray(codes), np.ascontiguousarray(s)
