// MX quantizer kernel (row-wise, column-wise transposed, dual) with the
// optional fixed or random-sign 32-point Hadamard rotation and optional
// stochastic rounding, plus its host-side launcher.  Included by the
// translation units that instantiate it; each gets its own error word.
//
// Operation: "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §02 -- blocks with
// their own dynamic exponent (microscaling) and a deterministic Hadamard
// rotation before the MXFP4 quantization of the Wgrad operands;
// "MindSpeed LLM FSDP2量化特性：低比特大模型训练完全指南", 第 1 步 -- block size
// 32, E4M3 elements.  Bit-level rules: OCP MX v1.0 / OCP FP8.
//
// Design (HBM-bound): a persistent grid of 2 CTAs per SM.  Thread 0 of each
// CTA streams 128x128 bf16 tiles into a 2-stage shared-memory ring with TMA
// (128-byte swizzle, two 64-column boxes per tile); all 8 warps read the tile
// from shared memory:
//   row path: a thread owns the same 32-column block of rows r and r+64;
//   col path: a thread owns the same 32-row block of two adjacent columns.
// Unrotated blocks (and the ablation variants) travel through the packed
// fp32x2 ALU side by side, one block per lane of each pair; rotated blocks
// go one after the other with adjacent elements paired, the first
// butterfly stage taken straight from the bf16 inputs.
// Each block is (optionally) rotated in registers, its amax reduced, its
// E8M0 exponent taken from the amax bits, and its elements converted with
// the hardware's round-to-nearest-even saturating E4M3/E2M1 conversions.
// Codes go to a swizzled shared-memory staging tile that one TMA store per
// layout writes out (the transposed column-wise tile included), so global
// writes are whole-tile bulk copies; scales leave as one 4-byte word per
// row or column of the tile, either row-major or straight into the GEMM's
// tensor-core chunk layout (a tile is exactly one 512-byte chunk).  The
// grid is launched with programmatic stream serialization and waits for the
// previous grid (griddepcontrol) before touching global memory.
//
// Ablation variants (template flag ABL): the same AMD FP4 page, §01, sets
// its deterministic rotation against random Hadamard rotations and
// stochastic rounding.  ABL_SIGN flips the sign of the inputs selected by a
// 32-bit mask before the butterflies (H_32 * diag(d)); ABL_SR replaces the
// round-to-nearest by stochastic rounding driven by Philox4x32-10 bits of
// each element's input index.
#pragma once

#include <string.h>

#include "mxq_common.cuh"
#include "mxq_host.h"

namespace mxq {
namespace {

__device__ uint32_t g_err_quant;

constexpr int Q_THREADS = 256;
constexpr int Q_ROWS = 128;             // tile rows
constexpr int Q_COLS = 128;             // tile cols (two 64-column swizzled halves)
constexpr int Q_HALF = Q_ROWS * 128;    // bytes of one half: 128 rows of 128 B
constexpr int Q_TILE = 2 * Q_HALF;      // 32 KB of bf16
constexpr int Q_STAGES = 2;
constexpr int Q_STAGE_OUT = 16384;      // staging of one layout's codes (<= 128 x 128 B)
constexpr int Q_OFF_OUT_R = Q_STAGES * Q_TILE;
constexpr int Q_OFF_OUT_C = Q_OFF_OUT_R + Q_STAGE_OUT;
constexpr int Q_OFF_SC_R = Q_OFF_OUT_C + Q_STAGE_OUT;   // 128 rows x 4 scale bytes
constexpr int Q_OFF_SC_C = Q_OFF_SC_R + 512;            // 128 cols x 4 scale bytes
constexpr int Q_OFF_BAR = Q_OFF_SC_C + 512;
constexpr int Q_SMEM = Q_OFF_BAR + 64 + 1024;

enum : int { ABL_SIGN = 1, ABL_SR = 2 };

struct QArgs {
  int64_t R, C;
  int32_t n_ct, n_tiles;
  uint8_t* scales_r;
  uint8_t* scales_c;
  uint64_t timeout_ns;
  uint32_t sign_mask;         // ABL_SIGN: bit i negates element i of every block
  uint32_t seed_lo, seed_hi;  // ABL_SR: Philox key
  int32_t sc_tc;              // scales in the GEMM's tensor-core chunk layout
  int64_t kcs_r, kcs_c;       // chunks per 128-line tile of each output (tc layout)
};

template <int FMT>
struct Elem;
// emax: exponent of the largest normal; mbits / emin / maxv: mantissa bits,
// smallest normal exponent and largest finite magnitude (the element grid).
template <>
struct Elem<MXQ_E4M3> {
  static constexpr uint32_t emax = 8;  // 448 = 1.75 * 2^8
  static constexpr int words = 8;      // 32 one-byte codes
  static constexpr int mbits = 3, emin = -6;
  static constexpr float maxv = 448.0f;
};
template <>
struct Elem<MXQ_E5M2> {
  static constexpr uint32_t emax = 15;  // 57344 = 1.75 * 2^15
  static constexpr int words = 8;       // 32 one-byte codes
  static constexpr int mbits = 2, emin = -14;
  static constexpr float maxv = 57344.0f;
};
template <>
struct Elem<MXQ_E2M1> {
  static constexpr uint32_t emax = 2;  // 6 = 1.5 * 2^2
  static constexpr int words = 4;      // 32 four-bit codes
  static constexpr int mbits = 1, emin = 0;
  static constexpr float maxv = 6.0f;
};

// RN_fp32(2^-2.5) = RN_fp32(sqrt(2)) / 8: the normalization of H_32.
MXQ_DEV float hadamard_c() { return __uint_as_float(0x3E3504F3u); }

// Packed fp32x2 arithmetic, each lane rounded to nearest (one instruction
// per pair, no fused multiply-add).
MXQ_DEV float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
MXQ_DEV float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "sub.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
MXQ_DEV float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Natural-order radix-2 Walsh-Hadamard butterflies on two independent
// 32-blocks at once (lane .x and lane .y): stages h = 1, 2, 4, 8, 16, every
// add/subtract rounded to nearest, no fused multiply-add.  The final
// multiply by c is left to the caller.
MXQ_DEV void fwht32_pair(float2 (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if ((j & h) == 0) {
        const float2 a = v[j], b = v[j + h];
        v[j] = add2(a, b);
        v[j + h] = sub2(a, b);
      }
    }
  }
}

// One 32-block in v[16] with v[i] = (x[2i], x[2i+1]) and stage h = 1 already
// applied: stages h = 2, 4, 8, 16 on packed pairs of adjacent elements (for
// h >= 2 elements 2i and 2i + 1 have the same partner offset).
MXQ_DEV void fwht32_single_from2(float2 (&v)[16]) {
#pragma unroll
  for (int hh = 1; hh < 16; hh <<= 1) {  // hh = h / 2, in pairs
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & hh) == 0) {
        const float2 a = v[i], b = v[i + hh];
        v[i] = add2(a, b);
        v[i + hh] = sub2(a, b);
      }
    }
  }
}

// First butterfly stage straight from bf16 inputs with the mixed-precision
// add: for a the bf16 in the low (bfly_lo) or high (bfly_hi) half of w and
// c an fp32, s = RN(a + c) and d = RN(a - c) -- the same values as widening
// a first (widening is exact), one integer op fewer per pair.
MXQ_DEV void bfly_lo(uint32_t w, float c, float& s, float& d) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, l, %3;\n\t}"
      : "=f"(s), "=f"(d)
      : "r"(w), "f"(c));
}
MXQ_DEV void bfly_hi(uint32_t w, float c, float& s, float& d) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, h, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
      : "=f"(s), "=f"(d)
      : "r"(w), "f"(c));
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds, each two 32x32 -> 64-bit products
// whose halves are xored with the other two words and the round key, the key
// stepping by the Weyl constants between rounds.  Counter (c0, c1, 0, 0).
MXQ_DEV uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
  uint32_t x0 = c0, x1 = c1, x2 = 0u, x3 = 0u;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    // one 32x32 -> 64-bit multiply each gives both halves
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * x0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * x2;
    const uint32_t lo0 = static_cast<uint32_t>(p0), hi0 = static_cast<uint32_t>(p0 >> 32);
    const uint32_t lo1 = static_cast<uint32_t>(p1), hi1 = static_cast<uint32_t>(p1 >> 32);
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(x0, x1, x2, x3);
}

// The four random words of the element group g = index / 4 (element index
// = input row * cols + input column); word index % 4 belongs to the element.
MXQ_DEV uint4 group_bits(uint64_t g, const QArgs& a) {
  return philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(g >> 32), a.seed_lo,
                       a.seed_hi);
}

// Stochastic rounding of one scaled element v onto the element grid.  With
// k = max(floor(log2|v|), emin) the grid step at |v| is q = 2^(k - mbits);
// t = |v| / q, F = floor(frac(t) * 2^32), and the magnitude becomes
// (floor(t) + [r < F]) * q, saturated at the largest finite element.  The
// sign is kept; the result lies on the grid, so the round-to-nearest
// conversion that follows encodes it unchanged.
//  - General form (sr_round_fp): every step is an exact fp32 operation on
//    power-of-two scalings (multiply, floor, subtraction of the floor).
//  - E4M3 / E5M2 fast path: for |v| >= 2^emin, q is one unit in bit
//    23 - mbits of |v|'s fp32 pattern, so floor(t) * q is the pattern with
//    the lower bits cleared, frac(t) * 2^32 is those lower bits shifted to
//    the top of a word, and adding the unit rounds up (a carry into the
//    exponent is the next binade's first grid point): integer work only.
//    Values under 2^emin (rare for these formats) take the general form.
//    E2M1 keeps the general form for all values: its subnormal range [0, 1)
//    holds many scaled elements, and a divergent branch would cost more.
template <int FMT>
MXQ_DEV float sr_round_fp(float v, uint32_t r) {
  const uint32_t b = __float_as_uint(v);
  const uint32_t sign = b & 0x80000000u;
  const float av = __uint_as_float(b ^ sign);
  const int k = max(static_cast<int>((b >> 23) & 0xFFu) - 127, Elem<FMT>::emin);
  const float t = av * __uint_as_float(static_cast<uint32_t>(127 + Elem<FMT>::mbits - k) << 23);
  const float lo = floorf(t);
  const uint32_t F = __float2uint_rz((t - lo) * 4294967296.0f);
  const float m = (lo + (r < F ? 1.0f : 0.0f)) *
                  __uint_as_float(static_cast<uint32_t>(127 - Elem<FMT>::mbits + k) << 23);
  return __uint_as_float(__float_as_uint(fminf(m, Elem<FMT>::maxv)) | sign);
}

template <int FMT>
MXQ_DEV float sr_round(float v, uint32_t r) {
  if constexpr (FMT == MXQ_E2M1) {
    return sr_round_fp<FMT>(v, r);
  } else {
    constexpr int MB = Elem<FMT>::mbits;
    const uint32_t b = __float_as_uint(v);
    const uint32_t sign = b & 0x80000000u;
    const uint32_t a = b ^ sign;
    if (static_cast<int>(a >> 23) - 127 < Elem<FMT>::emin) return sr_round_fp<FMT>(v, r);
    const uint32_t unit = 1u << (23 - MB);
    const uint32_t F = a << (9 + MB);
    const uint32_t m = (a & ~(unit - 1u)) + (r < F ? unit : 0u);
    return __uint_as_float(__float_as_uint(fminf(__uint_as_float(m), Elem<FMT>::maxv)) | sign);
  }
}

// Quantize two 32-blocks held lane-wise in v.  For the unrotated path the
// caller passes the amax bits (fp32 layout) of each block.
//
// Rotated path: the rotated value is y = RN(a * c) with a the butterfly
// output.  Its block amax is RN(max|a| * c) (rounding is monotone), and
// RN(a * c) * 2^(127-s) equals RN(a * (c * 2^(127-s))) whenever the result
// is a normal fp32; below that both are far under half the smallest element
// step and encode as a zero of the same sign.  So one multiply by the
// constant c * 2^(127-s) replaces two.  That constant is exact: a finite
// butterfly output is below 2^128, so the rotated amax is below 2^125.5 and
// s <= 252 - emax <= 250 for every element format, which keeps
// c * 2^(127-s) >= 2^-125.5 a normal fp32 (a NaN or infinite amax gives
// s = 255, whose codes are discarded).
//
// With ABL_SR the scaled elements are rounded stochastically before the
// conversion; rnd(g, ra, rb) supplies the random words of elements 4g..4g+3
// of block A (ra) and block B (rb).  Below the smallest normal fp32 the
// folded multiply may differ from the two-step product, but such values are
// below 2^-110 of a grid step, where the round-up threshold F is 0 either way.
template <int FMT, bool HAD, int ABL, class Rnd>
MXQ_DEV void quant_pair(float2 (&v)[32], uint32_t abA, uint32_t abB,
                        uint32_t (&oA)[Elem<FMT>::words], uint32_t (&oB)[Elem<FMT>::words],
                        uint32_t& sA, uint32_t& sB, const Rnd& rnd) {
  if constexpr (HAD) {
    fwht32_pair(v);
    float mA = fabsf(v[0].x), mB = fabsf(v[0].y);
#pragma unroll
    for (int j = 1; j < 31; j += 2) {
      mA = max3_abs_nan(mA, v[j].x, v[j + 1].x);
      mB = max3_abs_nan(mB, v[j].y, v[j + 1].y);
    }
    mA = max3_abs_nan(mA, v[31].x, v[31].x);
    mB = max3_abs_nan(mB, v[31].y, v[31].y);
    const float c = hadamard_c();
    abA = __float_as_uint(__fmul_rn(mA, c)) & 0x7FFFFFFFu;
    abB = __float_as_uint(__fmul_rn(mB, c)) & 0x7FFFFFFFu;
    sA = scale_of(abA, Elem<FMT>::emax);
    sB = scale_of(abB, Elem<FMT>::emax);
    const float2 m2 = make_float2(__fmul_rn(c, inv_scale(sA)), __fmul_rn(c, inv_scale(sB)));
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = mul2(v[j], m2);
  } else {
    sA = scale_of(abA, Elem<FMT>::emax);
    sB = scale_of(abB, Elem<FMT>::emax);
    const float2 m2 = make_float2(inv_scale(sA), inv_scale(sB));
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = mul2(v[j], m2);  // exact power-of-two scaling
  }
  if constexpr ((ABL & ABL_SR) != 0) {
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      uint4 ra, rb;
      rnd(g, ra, rb);
      const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[4 * g + i].x = sr_round<FMT>(v[4 * g + i].x, wa[i]);
        v[4 * g + i].y = sr_round<FMT>(v[4 * g + i].y, wb[i]);
      }
    }
  }
  if constexpr (FMT == MXQ_E4M3) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      oA[k] = cvt_e4m3x4(v[4 * k].x, v[4 * k + 1].x, v[4 * k + 2].x, v[4 * k + 3].x);
      oB[k] = cvt_e4m3x4(v[4 * k].y, v[4 * k + 1].y, v[4 * k + 2].y, v[4 * k + 3].y);
    }
  } else if constexpr (FMT == MXQ_E5M2) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      oA[k] = cvt_e5m2x4(v[4 * k].x, v[4 * k + 1].x, v[4 * k + 2].x, v[4 * k + 3].x);
      oB[k] = cvt_e5m2x4(v[4 * k].y, v[4 * k + 1].y, v[4 * k + 2].y, v[4 * k + 3].y);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      oA[k] = cvt_e2m1x8(v[8 * k].x, v[8 * k + 1].x, v[8 * k + 2].x, v[8 * k + 3].x,
                         v[8 * k + 4].x, v[8 * k + 5].x, v[8 * k + 6].x, v[8 * k + 7].x);
      oB[k] = cvt_e2m1x8(v[8 * k].y, v[8 * k + 1].y, v[8 * k + 2].y, v[8 * k + 3].y,
                         v[8 * k + 4].y, v[8 * k + 5].y, v[8 * k + 6].y, v[8 * k + 7].y);
    }
  }
  if (sA == 255u) {
#pragma unroll
    for (int k = 0; k < Elem<FMT>::words; ++k) oA[k] = 0u;
  }
  if (sB == 255u) {
#pragma unroll
    for (int k = 0; k < Elem<FMT>::words; ++k) oB[k] = 0u;
  }
}

// Rotate (stage 1 already applied), scale and encode one 32-block held as
// v[16] = (x[2i], x[2i+1]) pairs: the same arithmetic as quant_pair's
// rotated path for one block.  Processing the two blocks of a thread one
// after the other, rather than packed lane-wise, leaves the scheduler two
// independent instruction streams and saves the widening of stage-1 inputs
// (measured: dual Hadamard E2M1 16384 x 8192 from 0.62 to 0.66 of the copy
// rate, bit-identical outputs).
template <int FMT>
MXQ_DEV void quant_single_had(float2 (&v)[16], uint32_t (&o)[Elem<FMT>::words], uint32_t& sc) {
  fwht32_single_from2(v);
  float t[6];
#pragma unroll
  for (int i = 0; i < 5; ++i)
    t[i] = max3_abs_nan(max3_abs_nan(v[3 * i].x, v[3 * i].y, v[3 * i + 1].x), v[3 * i + 1].y,
                        max3_abs_nan(v[3 * i + 2].x, v[3 * i + 2].y, v[3 * i + 2].y));
  t[5] = max3_abs_nan(v[15].x, v[15].y, v[15].y);
  const float m =
      max3_abs_nan(max3_abs_nan(t[0], t[1], t[2]), max3_abs_nan(t[3], t[4], t[5]), t[5]);
  const float c = hadamard_c();
  sc = scale_of(__float_as_uint(__fmul_rn(m, c)) & 0x7FFFFFFFu, Elem<FMT>::emax);
  const float k = __fmul_rn(c, inv_scale(sc));  // exact: s <= 250 (see quant_pair)
  const float2 m2 = make_float2(k, k);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = mul2(v[i], m2);
  if constexpr (FMT == MXQ_E4M3) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      o[k] = cvt_e4m3x4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  } else if constexpr (FMT == MXQ_E5M2) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      o[k] = cvt_e5m2x4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = cvt_e2m1x8(v[4 * k].x, v[4 * k].y, v[4 * k + 1].x, v[4 * k + 1].y, v[4 * k + 2].x,
                        v[4 * k + 2].y, v[4 * k + 3].x, v[4 * k + 3].y);
  }
  if (sc == 255u) {
#pragma unroll
    for (int k = 0; k < Elem<FMT>::words; ++k) o[k] = 0u;
  }
}

// Byte offset of (row r, byte b of its 128-byte row) in a 128B-swizzled tile.
MXQ_DEV int swz128(int r, int b) { return r * 128 + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15)); }
// Byte offset of (row r, byte b of its 64-byte row) in a 64B-swizzled tile.
MXQ_DEV int swz64(int r, int b) { return r * 64 + (((((b >> 4) ^ (r >> 1)) & 3) << 4) | (b & 15)); }

// Write one block's codes into a staging tile whose rows are 128 B (one-byte
// codes, 128B swizzle) or 64 B (E2M1, 64B swizzle).
template <int FMT>
MXQ_DEV void stage_block(uint8_t* tile, int row, int block, const uint32_t (&o)[Elem<FMT>::words]) {
  if constexpr (FMT != MXQ_E2M1) {
    *reinterpret_cast<uint4*>(tile + swz128(row, 32 * block)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(tile + swz128(row, 32 * block + 16)) = make_uint4(o[4], o[5], o[6], o[7]);
  } else {
    *reinterpret_cast<uint4*>(tile + swz64(row, 16 * block)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int FMT, bool HAD, int ABL>
MXQ_DEV void row_path(const uint8_t* st, uint8_t* out_tile, uint8_t* sc_tile, int64_t R0,
                      int64_t C0, const QArgs& a, int tid) {
  const int r = tid & 63, q = tid >> 6;
  if (C0 + 32 * q >= a.C) return;
  const uint8_t* half = st + (q >> 1) * Q_HALF;
  const int cb = (q & 1) * 4;
  uint32_t wa[16], wb[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int off = ((cb + i) ^ (r & 7)) << 4;
    const uint4 A = *reinterpret_cast<const uint4*>(half + r * 128 + off);
    const uint4 B = *reinterpret_cast<const uint4*>(half + (r + 64) * 128 + off);
    wa[4 * i] = A.x; wa[4 * i + 1] = A.y; wa[4 * i + 2] = A.z; wa[4 * i + 3] = A.w;
    wb[4 * i] = B.x; wb[4 * i + 1] = B.y; wb[4 * i + 2] = B.z; wb[4 * i + 3] = B.w;
  }
  if constexpr (HAD && ABL == 0) {
    // stage 1 pairs elements 2k (low half) and 2k + 1 (high half) of word k
    uint32_t oA[Elem<FMT>::words], oB[Elem<FMT>::words], sA, sB;
    {
      float2 v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) bfly_lo(wa[k], bf16hi(wa[k]), v[k].x, v[k].y);
      quant_single_had<FMT>(v, oA, sA);
    }
    {
      float2 v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) bfly_lo(wb[k], bf16hi(wb[k]), v[k].x, v[k].y);
      quant_single_had<FMT>(v, oB, sB);
    }
    stage_block<FMT>(out_tile, r, q, oA);
    stage_block<FMT>(out_tile, r + 64, q, oB);
    sc_tile[r * 4 + q] = static_cast<uint8_t>(sA);
    sc_tile[(r + 64) * 4 + q] = static_cast<uint8_t>(sB);
    return;
  }
  if constexpr ((ABL & ABL_SIGN) != 0) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {  // word k holds elements 2k (low half) and 2k + 1
      const uint32_t m = (((a.sign_mask >> (2 * k)) & 1u) << 15) |
                         (((a.sign_mask >> (2 * k + 1)) & 1u) << 31);
      wa[k] ^= m;
      wb[k] ^= m;
    }
  }
  uint32_t abA = 0, abB = 0;
  if constexpr (!HAD) {
    uint32_t ma = wa[0], mb = wb[0];
#pragma unroll
    for (int k = 1; k < 16; ++k) {
      ma = max_abs_bf16x2(ma, wa[k]);
      mb = max_abs_bf16x2(mb, wb[k]);
    }
    abA = max(ma & 0x7FFFu, (ma >> 16) & 0x7FFFu) << 16;
    abB = max(mb & 0x7FFFu, (mb >> 16) & 0x7FFFu) << 16;
  }
  float2 v[32];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    v[2 * k] = make_float2(bf16lo(wa[k]), bf16lo(wb[k]));
    v[2 * k + 1] = make_float2(bf16hi(wa[k]), bf16hi(wb[k]));
  }
  // element indices of the first elements of the two blocks (C % 32 == 0,
  // so each is a multiple of 4 and element 4g + i takes word i of group g)
  const uint64_t gA = static_cast<uint64_t>((R0 + r) * a.C + C0 + 32 * q) >> 2;
  const uint64_t gB = gA + ((static_cast<uint64_t>(a.C) * 64) >> 2);
  auto rnd = [&](int g, uint4& ra, uint4& rb) {
    ra = group_bits(gA + g, a);
    rb = group_bits(gB + g, a);
  };
  uint32_t oA[Elem<FMT>::words], oB[Elem<FMT>::words], sA, sB;
  quant_pair<FMT, HAD, ABL>(v, abA, abB, oA, oB, sA, sB, rnd);
  stage_block<FMT>(out_tile, r, q, oA);
  stage_block<FMT>(out_tile, r + 64, q, oB);
  sc_tile[r * 4 + q] = static_cast<uint8_t>(sA);
  sc_tile[(r + 64) * 4 + q] = static_cast<uint8_t>(sB);
}

template <int FMT, bool HAD, int ABL>
MXQ_DEV void col_path(const uint8_t* st, uint8_t* out_tile, uint8_t* sc_tile, int64_t R0,
                      int64_t C0, const QArgs& a, int tid) {
  const int cp = tid & 63, b = tid >> 6;
  // b is warp-uniform.  With stochastic rounding the lanes of a warp trade
  // random words, so lanes past the last column stay and compute on the
  // zero-filled tile; their staging rows and scales fall outside the output
  // and are never stored.
  if (R0 + 32 * b >= a.R) return;
  if constexpr ((ABL & ABL_SR) == 0) {
    if (C0 + 2 * cp >= a.C) return;
  }
  const uint8_t* half = st + (cp >> 5) * Q_HALF;
  const int pb = (cp & 31) * 4;  // byte of the column pair inside its 128-byte row
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) w[j] = *reinterpret_cast<const uint32_t*>(half + swz128(32 * b + j, pb));
  if constexpr (HAD && ABL == 0) {
    // stage 1 pairs rows j and j + 1 of each column (column A in the low
    // halves, column B in the high halves)
    uint32_t oA[Elem<FMT>::words], oB[Elem<FMT>::words], sA, sB;
    {
      float2 v[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) bfly_lo(w[j], bf16lo(w[j + 1]), v[j / 2].x, v[j / 2].y);
      quant_single_had<FMT>(v, oA, sA);
    }
    {
      float2 v[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) bfly_hi(w[j], bf16hi(w[j + 1]), v[j / 2].x, v[j / 2].y);
      quant_single_had<FMT>(v, oB, sB);
    }
    stage_block<FMT>(out_tile, 2 * cp, b, oA);
    stage_block<FMT>(out_tile, 2 * cp + 1, b, oB);
    sc_tile[(2 * cp) * 4 + b] = static_cast<uint8_t>(sA);
    sc_tile[(2 * cp + 1) * 4 + b] = static_cast<uint8_t>(sB);
    return;
  }
  if constexpr ((ABL & ABL_SIGN) != 0) {
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] ^= ((a.sign_mask >> j) & 1u) * 0x80008000u;
  }
  uint32_t abA = 0, abB = 0;
  if constexpr (!HAD) {
    uint32_t m = w[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) m = max_abs_bf16x2(m, w[j]);
    abA = (m & 0x7FFFu) << 16;
    abB = ((m >> 16) & 0x7FFFu) << 16;
  }
  float2 v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = make_float2(bf16lo(w[j]), bf16hi(w[j]));
  // Element j of the column pair sits at index (R0 + 32b + j) * C + c, c
  // even, C % 8 == 0: the group of 4 words of row j covers columns
  // c - c%4 .. c - c%4 + 3, words (x, y) for an even pair index cp and (z, w)
  // for an odd one.  Lanes cp and cp ^ 1 (adjacent lanes) therefore need the
  // same groups: for each row pair (j, j + 1) the even lane draws row j, the
  // odd lane row j + 1, and each hands the other the two words it needs.
  const int64_t i0 = (R0 + 32 * b) * a.C + C0 + 2 * cp;
  const bool odd = (cp & 1) != 0;
  auto rnd = [&](int g, uint4& ra, uint4& rb) {
    uint32_t xa[4], xb[4];
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
      const int j = 4 * g + i + (odd ? 1 : 0);
      const uint4 w4 = group_bits(static_cast<uint64_t>(i0 + j * a.C) >> 2, a);
      const uint32_t keep0 = odd ? w4.z : w4.x, keep1 = odd ? w4.w : w4.y;
      const uint32_t give0 = odd ? w4.x : w4.z, give1 = odd ? w4.y : w4.w;
      const uint32_t got0 = __shfl_xor_sync(0xFFFFFFFFu, give0, 1);
      const uint32_t got1 = __shfl_xor_sync(0xFFFFFFFFu, give1, 1);
      xa[i] = odd ? got0 : keep0;
      xb[i] = odd ? got1 : keep1;
      xa[i + 1] = odd ? keep0 : got0;
      xb[i + 1] = odd ? keep1 : got1;
    }
    ra = make_uint4(xa[0], xa[1], xa[2], xa[3]);
    rb = make_uint4(xb[0], xb[1], xb[2], xb[3]);
  };
  uint32_t oA[Elem<FMT>::words], oB[Elem<FMT>::words], sA, sB;
  quant_pair<FMT, HAD, ABL>(v, abA, abB, oA, oB, sA, sB, rnd);
  stage_block<FMT>(out_tile, 2 * cp, b, oA);
  stage_block<FMT>(out_tile, 2 * cp + 1, b, oB);
  sc_tile[(2 * cp) * 4 + b] = static_cast<uint8_t>(sA);
  sc_tile[(2 * cp + 1) * 4 + b] = static_cast<uint8_t>(sB);
}

// Scale bytes of one tile: 4 per tile row (row-wise) or tile column
// (column-wise), written as one word when the destination is aligned.
MXQ_DEV void store_scales(const uint8_t* sc_tile, uint8_t* dst, int64_t n_lines, int64_t line0,
                          int64_t nsb, int64_t blk0, int64_t nblk_valid, int i) {
  const int64_t line = line0 + i;
  if (line >= n_lines) return;
  if (!MXQ_IN_BOUNDS(blk0 >= 0 && blk0 + (nblk_valid < 4 ? nblk_valid : int64_t(4)) <= nsb, &g_err_quant,
                     SITE_B_QUANT_SCALE))
    return;
  uint8_t* d = dst + line * nsb + blk0;
  const uint32_t w = *reinterpret_cast<const uint32_t*>(sc_tile + 4 * i);
  if (nblk_valid >= 4 && (reinterpret_cast<uintptr_t>(d) & 3u) == 0) {
    *reinterpret_cast<uint32_t*>(d) = w;
  } else {
    for (int k = 0; k < 4 && k < nblk_valid; ++k) d[k] = static_cast<uint8_t>(w >> (8 * k));
  }
}

// Scale bytes of one tile in the tensor-core chunk layout the GEMM's
// tcgen05.cp reads: a 128-line x 128-element tile has exactly one 512-byte
// chunk (128 lines x 4 blocks), chunk (line0 / 128) * kcs + kc, with the 4
// bytes of line i at (i % 32) * 16 + (i / 32) * 4.  Lines past the tensor
// get zero scales, so the chunk never holds a stale or NaN byte.
MXQ_DEV void store_scales_tc(const uint8_t* sc_tile, uint8_t* dst, int64_t n_lines, int64_t line0,
                             int64_t kcs, int64_t kc, int i) {
  if (!MXQ_IN_BOUNDS(line0 >= 0 && line0 < n_lines && kc >= 0 && kc < kcs && i >= 0 && i < 128,
                     &g_err_quant, SITE_B_QUANT_SCALE_TC))
    return;
  uint8_t* chunk = dst + ((line0 >> 7) * kcs + kc) * 512;
  const uint32_t w = line0 + i < n_lines ? *reinterpret_cast<const uint32_t*>(sc_tile + 4 * i) : 0u;
  *reinterpret_cast<uint32_t*>(chunk + (i & 31) * 16 + (i >> 5) * 4) = w;
}

MXQ_DEV void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
MXQ_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
MXQ_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
MXQ_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
MXQ_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Tile t -> (tile row, tile column).  Row-major order, or, for kernels
// whose column-wise output has one-byte codes (GROUPED), groups of
// Q_GROUP tile columns with the tile rows of a group and its columns
// fastest: the CTAs resident at one time then cover about 2 * SMs /
// Q_GROUP tile rows of Q_GROUP columns, so each column-wise output line
// receives a longer run of consecutive 128-byte pieces.  Measured
// (fraction of the copy rate): column-wise E4M3 16384 x 8192 0.93 -> 0.95;
// dual E4M3 / E4M3 16384 x 8192 0.82 -> 0.86-0.88, 28672 x 4096 0.81 ->
// 0.85-0.87, 4096 x 14336 0.82 -> 0.85, 6144 x 4096 0.78 -> 0.74.  The dual
// gains appear only with the arithmetic exactly as below (tile rows derived
// by a division on every call, 64-bit products and quotients): the same
// order with precomputed tile rows or in 32-bit arithmetic ran at 0.82.
// The cause is not known.  Column-wise E2M1 tiles fill half lines and ran
// 12-15% slower grouped, so they keep row-major order.
constexpr int Q_GROUP = 8;

template <bool GROUPED>
MXQ_DEV void tile_rc(int t, const QArgs& a, int& rt, int& ct) {
  if constexpr (!GROUPED) {
    rt = t / a.n_ct;
    ct = t - rt * a.n_ct;
  } else {
    const int64_t n_rt = a.n_tiles / a.n_ct;
    const int64_t per = int64_t(Q_GROUP) * n_rt;      // tiles of one full group
    const int64_t g = t / per, r = t - g * per;
    const int64_t w = min(int64_t(Q_GROUP), int64_t(a.n_ct) - g * Q_GROUP);  // group width
    rt = static_cast<int>(r / w);
    ct = static_cast<int>(g * Q_GROUP + (r - int64_t(rt) * w));
  }
}

template <bool ROW, bool COL, int FR, bool HR, int FC, bool HC, int ABL>
__global__ void __launch_bounds__(Q_THREADS, 2)
    mx_quant_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tm_r,
                    const __grid_constant__ CUtensorMap tm_c, const QArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Q_OFF_BAR);
  uint8_t* out_r = smem + Q_OFF_OUT_R;
  uint8_t* out_c = smem + Q_OFF_OUT_C;
  uint8_t* sc_r = smem + Q_OFF_SC_R;
  uint8_t* sc_c = smem + Q_OFF_SC_C;
  const int tid = threadIdx.x;
  constexpr bool GROUPED = COL && FC != MXQ_E2M1;
  if (tid == 0) {
    prefetch_tmap(&tmap);
    if constexpr (ROW) prefetch_tmap(&tm_r);
    if constexpr (COL) prefetch_tmap(&tm_c);
#pragma unroll
    for (int s = 0; s < Q_STAGES; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();               // the previous kernel's writes are visible
  griddep_launch_dependents();

  auto issue = [&](int t, int s) {
    int rt, ct;
    tile_rc<GROUPED>(t, a, rt, ct);
    const uint32_t bar = smem_u32(&bars[s]);
    const uint32_t dst = smem_u32(smem + s * Q_TILE);
    // x of a TMA copy must be a multiple of 16 bytes (8 bf16 elements)
    if (!MXQ_IN_BOUNDS(((ct * Q_COLS) & 7) == 0, &g_err_quant, SITE_B_QUANT_TMA)) return;
    mbar_arrive_expect_tx(bar, Q_TILE);
    tma_load_2d(dst, &tmap, bar, ct * Q_COLS, rt * Q_ROWS);
    tma_load_2d(dst + Q_HALF, &tmap, bar, ct * Q_COLS + 64, rt * Q_ROWS);
  };
  if (tid == 0) {
    for (int s = 0; s < Q_STAGES; ++s) {
      const int t = blockIdx.x + s * gridDim.x;
      if (t < a.n_tiles) issue(t, s);
    }
  }

  const int64_t nsb_r = a.C >> 5, nsb_c = a.R >> 5;
  int it = 0;
  bool failed = false;
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++it) {
    const int s = it % Q_STAGES;
    const uint32_t parity = (it / Q_STAGES) & 1;
    const bool ok = mbar_wait(smem_u32(&bars[s]), parity, a.timeout_ns);
    if (tid == 0) bulk_wait_read0();  // the previous tile's stores have read the staging
    if (!__syncthreads_and(ok)) {
      failed = true;
      break;
    }
    int rt, ct;
    tile_rc<GROUPED>(t, a, rt, ct);
    const int64_t R0 = int64_t(rt) * Q_ROWS, C0 = int64_t(ct) * Q_COLS;
    // the same value in every thread: a tile outside the tensor is skipped whole
    const bool inb = MXQ_IN_BOUNDS(rt >= 0 && ct >= 0 && R0 < a.R && C0 < a.C, &g_err_quant,
                                   SITE_B_QUANT_TILE);
    const uint8_t* st = smem + s * Q_TILE;
    if constexpr (ROW) if (inb) row_path<FR, HR, ABL>(st, out_r, sc_r, R0, C0, a, tid);
    if constexpr (COL) if (inb) col_path<FC, HC, ABL>(st, out_c, sc_c, R0, C0, a, tid);
    fence_async_smem();
    __syncthreads();  // staging complete; stage s fully read
    if (tid == 0) {
      // x of a TMA store must be a multiple of 16 bytes
      const int64_t xr = FR != MXQ_E2M1 ? C0 : C0 / 2, xc = FC != MXQ_E2M1 ? R0 : R0 / 2;
      if constexpr (ROW)
        if (inb && MXQ_IN_BOUNDS((xr & 15) == 0, &g_err_quant, SITE_B_QUANT_TMA))
          tma_store_2d(&tm_r, smem_u32(out_r), static_cast<int32_t>(xr), static_cast<int32_t>(R0));
      if constexpr (COL)
        if (inb && MXQ_IN_BOUNDS((xc & 15) == 0, &g_err_quant, SITE_B_QUANT_TMA))
          tma_store_2d(&tm_c, smem_u32(out_c), static_cast<int32_t>(xc), static_cast<int32_t>(C0));
      bulk_commit();
      const int tn = t + Q_STAGES * gridDim.x;
      if (tn < a.n_tiles) issue(tn, s);
    }
    if constexpr (ROW) {
      if (inb && tid < Q_ROWS) {
        if (a.sc_tc) store_scales_tc(sc_r, a.scales_r, a.R, R0, a.kcs_r, C0 >> 7, tid);
        else store_scales(sc_r, a.scales_r, a.R, R0, nsb_r, C0 >> 5, (a.C - C0 + 31) >> 5, tid);
      }
    }
    if constexpr (COL) {
      if (inb && tid >= Q_THREADS - Q_COLS) {
        const int i = tid - (Q_THREADS - Q_COLS);
        if (a.sc_tc) store_scales_tc(sc_c, a.scales_c, a.C, C0, a.kcs_c, R0 >> 7, i);
        else store_scales(sc_c, a.scales_c, a.C, C0, nsb_c, R0 >> 5, (a.R - R0 + 31) >> 5, i);
      }
    }
  }
  if (tid == 0) bulk_wait0();
  if (failed && tid == 0) {
    record_error(&g_err_quant, MXQ_ERR_TIMEOUT, SITE_QUANT_FULL);
    // Give copies still in flight into this CTA's shared memory a bounded
    // chance to land before the CTA exits.
    for (int k = it; k < it + Q_STAGES; ++k) {
      const int t = blockIdx.x + k * gridDim.x;
      if (t >= a.n_tiles) break;
      if (!mbar_wait(smem_u32(&bars[k % Q_STAGES]), (k / Q_STAGES) & 1, a.timeout_ns))
        record_error(&g_err_quant, MXQ_ERR_TIMEOUT, SITE_QUANT_DRAIN);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

using QuantKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const QArgs);

bool valid_fmt(int f) { return f == MXQ_E4M3 || f == MXQ_E2M1 || f == MXQ_E5M2; }

// Validates the arguments, encodes the tensor maps of x and of the code
// outputs, and launches kernel k (chosen by the caller for these formats)
// as a persistent grid of up to 2 CTAs per SM.
mxq_status quant_launch_k(QuantKernel k, const void* x, int64_t R, int64_t C, bool row, bool col,
                          int fr, void* codes_r, uint8_t* scales_r, int fc, void* codes_c,
                          uint8_t* scales_c, uint32_t sign_mask, uint64_t seed, void* stream,
                          int scale_layout = MXQ_SCALES_ROWMAJOR) {
  if (R < 0 || C < 0) return MXQ_ERR_ARG;
  if (R == 0 || C == 0) return MXQ_OK;
  if (R >= (int64_t(1) << 31) || C >= (int64_t(1) << 31)) return MXQ_ERR_ARG;
  if (!x) return MXQ_ERR_ARG;
  if (row && (!valid_fmt(fr) || !codes_r || !scales_r)) return MXQ_ERR_ARG;
  if (col && (!valid_fmt(fc) || !codes_c || !scales_c)) return MXQ_ERR_ARG;
  if (row && C % 32 != 0) return MXQ_ERR_ARG;
  if (col && (R % 32 != 0 || C % 8 != 0)) return MXQ_ERR_ARG;
  if (!aligned16(x) || (row && !aligned16(codes_r)) || (col && !aligned16(codes_c)))
    return MXQ_ERR_ALIGN;
  if (scale_layout != MXQ_SCALES_ROWMAJOR && scale_layout != MXQ_SCALES_TC) return MXQ_ERR_ARG;
  const bool tc = scale_layout == MXQ_SCALES_TC;
  if (tc) {
    // whole chunks only: the blocked dimension covers whole 128-element
    // chunks, and whole chunk pairs (one E2M1 GEMM stage) for E2M1
    if (row && C % (fr == MXQ_E2M1 ? 256 : 128) != 0) return MXQ_ERR_ARG;
    if (col && R % (fc == MXQ_E2M1 ? 256 : 128) != 0) return MXQ_ERR_ARG;
    if ((row && !aligned16(scales_r)) || (col && !aligned16(scales_c))) return MXQ_ERR_ALIGN;
  }

  CUtensorMap map;
  CUresult cr = tensor_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(C),
                              static_cast<uint64_t>(R), static_cast<uint64_t>(C) * 2, 64, Q_ROWS,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (cr != CUDA_SUCCESS) return MXQ_ERR_CUDA;

  // Code outputs: 2-D byte tensors written by TMA stores of 128-row tiles.
  // Rows of 128 B (one-byte codes) use the 128-byte swizzle, rows of 64 B
  // (E2M1) the 64-byte swizzle, matching the staging layout in the kernel.
  auto code_map = [&](CUtensorMap* m, void* base, int64_t lines, int64_t line_elems,
                      int fmt) -> CUresult {
    const int64_t lb = fmt != MXQ_E2M1 ? line_elems : line_elems / 2;
    return tensor_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, static_cast<uint64_t>(lb),
                         static_cast<uint64_t>(lines), static_cast<uint64_t>(lb),
                         fmt != MXQ_E2M1 ? 128u : 64u, static_cast<uint32_t>(Q_ROWS),
                         fmt != MXQ_E2M1 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE);
  };
  CUtensorMap map_r, map_c;
  memset(&map_r, 0, sizeof(map_r));
  memset(&map_c, 0, sizeof(map_c));
  if (row && code_map(&map_r, codes_r, R, C, fr) != CUDA_SUCCESS) return MXQ_ERR_CUDA;
  if (col && code_map(&map_c, codes_c, C, R, fc) != CUDA_SUCCESS) return MXQ_ERR_CUDA;

  QArgs a;
  memset(&a, 0, sizeof(a));
  a.R = R;
  a.C = C;
  a.n_ct = static_cast<int32_t>((C + Q_COLS - 1) / Q_COLS);
  const int64_t n_rt = (R + Q_ROWS - 1) / Q_ROWS;
  if (n_rt * a.n_ct >= (int64_t(1) << 31)) return MXQ_ERR_ARG;
  a.n_tiles = static_cast<int32_t>(n_rt * a.n_ct);
  a.scales_r = scales_r;
  a.scales_c = scales_c;
  a.timeout_ns = wait_timeout_ns();
  a.sign_mask = sign_mask;
  a.seed_lo = static_cast<uint32_t>(seed);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  a.sc_tc = tc ? 1 : 0;
  a.kcs_r = C / 128;
  a.kcs_c = R / 128;

  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(k), Q_SMEM)) return MXQ_ERR_CUDA;
  // persistent grid (every CTA resident), launched so that it may start
  // while the previous kernel on the stream drains
  const int grid = static_cast<int>(std::min<int64_t>(a.n_tiles, int64_t(2) * sm_count()));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Q_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Q_SMEM;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k, map, map_r, map_c, a) != cudaSuccess) return MXQ_ERR_CUDA;
  return launch_status();
}

// Reads and clears this translation unit's device error word.
uint32_t take_error_word() {
  uint32_t h = 0;
  if (cudaMemcpyFromSymbol(&h, g_err_quant, sizeof(h)) != cudaSuccess) return MXQ_ERR_CUDA;
  if (h) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_err_quant, &z, sizeof(z));
  }
  return h;
}

}  // namespace
}  // namespace mxq
