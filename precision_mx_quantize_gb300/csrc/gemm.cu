// Block-scaled MX GEMM on the 5th-generation tensor cores (tcgen05).
//
// Operation: "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §02-§03 -- the
// forward, activation-gradient and weight-gradient GEMMs run natively on MX
// (FP8 / FP4) codes, each 32-element block scaled by its E8M0 exponent:
//   C[m][n] = sum_k dec(A[m][k]) 2^(sA[m][k/32]-127) dec(B[n][k]) 2^(sB[n][k/32]-127)
// accumulated in fp32.  E4M3 operands use kind::mxf8f6f4 (one scale per 32
// along K per MMA of K=32); E2M1 operands use kind::mxf4 on packed nibbles
// (two scales per MMA of K=64).
//
// Kernel structure: clusters of two CTAs on the two SMs of a TPC run the
// pair MMA (cta_group::2) on 256x256 output tiles, persistent over tiles.
// Each CTA holds 128 rows of A and 128 of the tile's 256 B rows; the pair
// MMA reads both halves, so an SM streams 32 KB of operands per K stage
// instead of the 48 KB a single-SM 128x256 tile needs, which keeps the
// shared-memory traffic (TMA writes + tensor-core reads) within bandwidth.
//   warp 0     (both CTAs) TMA producer: own A rows and own B half, 128 B of
//              K per stage with 128-byte swizzle, plus the stage's scale
//              chunks (own 128 A rows, all 256 B rows) into a 6-stage ring;
//   warp 1     (both CTAs) allocates the pair's tensor memory.  In the
//              leader CTA one lane issues the four pair MMAs of each stage
//              into the fp32 accumulators (each CTA: 128 lanes x 256
//              columns), then releases the stage in both CTAs;
//   warps 10-11 (leader) one lane each copies part of each stage's scales
//              into both CTAs' tensor memory (tcgen05.cp) ahead of the MMA
//              lane;
//   warps 2-9  (both CTAs) epilogue: each drains 32 accumulator lanes x 128
//              columns into registers, tells the leader the accumulator is
//              free (a relaxed arrive: it must not wait for earlier stores),
//              and stores its rows -- fp32, bf16, or row-wise MX codes of the
//              product -- paced over the next tile's main loop, with 256-bit
//              stores when aligned.
// Scales: tcgen05.cp reads them in a chunk layout (for every 128-row x
// 4-block chunk, byte (r % 32) * 16 + (r / 32) * 4 + (kb % 4)).  Scales the
// quantizers wrote in that layout are loaded in place; row-major scales are
// first rewritten into it by a small pre-pass kernel in the caller's
// workspace.  The kernel is launched with programmatic stream serialization
// and waits for the previous grid (griddepcontrol) before any global access.
#include <string.h>

#include <mutex>

#include "mxq_common.cuh"
#include "mxq_host.h"

namespace mxq {

__device__ uint32_t g_err_gemm;

namespace {

constexpr int G_CLUSTER = 2;                 // CTA pair of one 2-SM MMA
constexpr int G_BM = 128;                    // rows of A per CTA (pair tile: 256)
constexpr int G_BN = 256;                    // columns of the tile (rows of B)
constexpr int G_BN_CTA = G_BN / G_CLUSTER;   // rows of B each CTA holds
constexpr int G_BKB = 128;                   // bytes of K per stage (one 128 B swizzle row)
constexpr int G_STAGES = 6;
constexpr int G_THREADS = 384;               // 12 warps
constexpr int G_A_BYTES = G_BM * G_BKB;      // 16 KB
constexpr int G_B_BYTES = G_BN_CTA * G_BKB;  // 16 KB
constexpr int G_SFA_BYTES = 1024;            // own 128 rows: up to 2 chunks of 512 B
constexpr int G_SFB_BYTES = 2048;            // all 256 rows: up to 4 chunks of 512 B
constexpr int G_STAGE_BYTES = G_A_BYTES + G_B_BYTES + G_SFA_BYTES + G_SFB_BYTES;
constexpr int G_BAR_BYTES = 512;
constexpr uint32_t kNotYet = 0xFFFFFFFFu;   // peer's stage count not yet reported
constexpr int G_SMEM = G_STAGES * G_STAGE_BYTES + G_BAR_BYTES + 1024;
constexpr uint32_t G_TMEM_COLS = 512;
constexpr uint32_t G_SFA_COL0 = 256;                 // 8 columns per stage
constexpr uint32_t G_SFB_COL0 = 256 + 8 * G_STAGES;  // 16 columns per stage
static_assert(G_SFB_COL0 + 16 * G_STAGES <= G_TMEM_COLS, "tensor memory budget");
static_assert(G_STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");

// One GEMM problem of a launch.  Fields up to q_scale_tc may differ between
// the problems of a grouped launch; the element format, the epilogue kind and
// the wait limit are those of problem 0 for all.
struct GArgs {
  int32_t M, N;
  int32_t tile0;                // first work item of this problem in the launch
  int32_t n_mp, n_nt, n_tiles;  // 256-row pair tiles along M, 256-col tiles along N
  int32_t group;                // tiles per raster group along the grouped dimension
  int32_t group_n;              // 1: groups run along N, 0: along M
  int32_t nk;                   // K stages
  int32_t kc_per_row;           // 512-byte scale chunks per 128-row tile (KBp / 4)
  const uint8_t* sfa;           // chunked scales of A in the workspace
  const uint8_t* sfb;           // chunked scales of B
  void* C;
  int32_t out_bf16;
  int32_t fp4;
  int32_t elem_code;            // A/B element type field of the instruction descriptor
  int32_t wide_stores;          // rows of C are 32-byte aligned: 256-bit stores
  int32_t out_q;                // 1: C receives row-wise MX codes of the product
  int32_t q_fmt;                // their element format
  uint8_t* q_scales;            // their E8M0 scales [M][N/32]
  int32_t q_scale_words;        // scale rows are 4-byte aligned: one word per 4 blocks
  int32_t q_scale_tc;           // output scales in the tensor cores' chunk layout
  uint32_t pace_ns;             // epilogue: pause after each 16/32-byte store (see below)
  uint64_t timeout_ns;
};

// A launch: up to G_MAX_GROUP problems of one element format and their
// tensor maps, the work items of problem i numbered from p[i].tile0.  One
// problem is the plain GEMM; several are independent GEMMs that run as one
// persistent grid (e.g. the weight gradients of several layers, which no
// layer waits for), so their tiles fill the waves together.
constexpr int G_MAX_GROUP = 8;
struct GGroup {
  CUtensorMap ta[G_MAX_GROUP], tb[G_MAX_GROUP], tsa[G_MAX_GROUP], tsb[G_MAX_GROUP];
  GArgs p[G_MAX_GROUP];
  int32_t count;
  int32_t n_tiles;              // work items of all problems
};

// ---- tcgen05 / cluster wrappers --------------------------------------------
MXQ_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

MXQ_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

MXQ_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MXQ_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive (once the pair's earlier tcgen05 operations complete) on the
// barrier at `bar`'s offset in every CTA of cta_mask.
MXQ_DEV void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Shared-memory matrix descriptor: start, leading / stride byte offsets,
// descriptor version 1, layout (0 = no swizzle, 2 = 128-byte swizzle).
MXQ_DEV uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Copy one 512-byte scale chunk (32 rows x 16 B) of each CTA's shared memory
// into 4 columns of the same CTA's tensor memory, replicated to all four
// 32-lane quadrants.
MXQ_DEV void tc_cp_sf_pair(uint32_t taddr, uint32_t smem_addr) {
  const uint64_t d = smem_desc(smem_addr, 0, 128, 0);
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

MXQ_DEV void mma_mxf8_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                           uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
      : "memory");
}

MXQ_DEV void mma_mxf4_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                           uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
      : "memory");
}

// Instruction descriptor of a block-scaled pair MMA: K-major A and B,
// M = 256 (128 per CTA), N = 256, E8M0 scales, scale-factor byte ids.
MXQ_DEV uint32_t idesc_block_scaled(uint32_t fmt_code, uint32_t a_sf, uint32_t b_sf) {
  uint32_t d = 0;
  d |= (b_sf & 3u) << 4;
  d |= (fmt_code & 7u) << 7;    // A format
  d |= (fmt_code & 7u) << 10;   // B format
  d |= static_cast<uint32_t>(G_BN >> 3) << 17;
  d |= 1u << 23;                // scale type: UE8M0
  d |= static_cast<uint32_t>((G_CLUSTER * G_BM) >> 4) << 24;
  d |= (a_sf & 3u) << 29;
  return d;
}

#define MXQ_TMEM_LD32(taddr, r)                                                                  \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "    \
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "    \
      "%28, %29, %30, %31}, [%32];"                                                              \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])            \
      : "r"(taddr))

// 256-bit global store of eight 32-bit words (32-byte aligned address).
MXQ_DEV void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                          uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

MXQ_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

MXQ_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

MXQ_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
MXQ_DEV uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive, without release semantics, on a barrier that may live in another
// CTA of the cluster.  The epilogue uses it to hand the accumulator back: its tensor-memory loads have already completed
// (tcgen05.wait::ld), which is all the next tile's MMAs need, while a
// release arrive would also wait for the thread's earlier global stores
// (the previous tile's output) to complete -- about 1700 cycles per tile
// in which the tensor pipe sat idle.
MXQ_DEV void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Store a word into shared memory of a CTA of the cluster (`addr` from mapa).
MXQ_DEV void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cluster.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

MXQ_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// A bounded wait (cluster-scope acquire) that also gives up once another
// role of this CTA has aborted.
MXQ_DEV bool gwait(uint32_t bar, uint32_t parity, uint64_t limit, volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit) return false;
  }
  return true;
}

MXQ_DEV void gabort(volatile int* abort_flag, uint32_t site) {
  *abort_flag = 1;
  record_error(&g_err_gemm, MXQ_ERR_TIMEOUT, site);
}

// TMA load whose completion is signalled on a barrier that may live in the
// peer CTA of the pair (`bar` is a cluster shared-memory address).
MXQ_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                              int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Store pacing.  A tile's epilogue stores leave the SM in one burst
// (64-256 KB per CTA) right when the next tile's main loop needs the same
// SM-to-L2 path for its TMA loads; the burst lengthens the loads' latency,
// and the latency-bound operand ring stalls the tensor pipe.  Spreading each
// thread's stores over part of the next tile's main loop avoids that (+3-12%
// measured, most on MXFP4 with fp32 output).  The last tile of a CTA is
// stored at full speed, since nothing runs behind it.
MXQ_DEV void pace(uint32_t ns) {
  if (ns) __nanosleep(ns);
}

// Row-wise MX quantization of the 128 fp32 accumulators a thread holds for
// one output row (four 32-column blocks, nblk of them inside N): per block
// the amax of the fp32 values, its E8M0 exponent, the exact power-of-two
// scaling and the round-to-nearest-even saturating conversion -- the rules
// of the quantizer, applied to the fp32 product without a bf16 rounding.
template <int QF>
MXQ_DEV void store_row_codes(const uint32_t (&v)[128], const GArgs& a, int64_t row, int64_t col0,
                             int nblk, uint32_t pace_ns) {
  constexpr uint32_t emax = QF == MXQ_E4M3 ? 8u : (QF == MXQ_E5M2 ? 15u : 2u);
  constexpr int cb = QF == MXQ_E2M1 ? 16 : 32;   // code bytes per block
  const int64_t row_bytes = QF == MXQ_E2M1 ? int64_t(a.N) / 2 : int64_t(a.N);
  uint8_t* crow = static_cast<uint8_t*>(a.C) + row * row_bytes + (col0 / 32) * cb;
  uint32_t sw = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    if (b < nblk) {
      const uint32_t* x = v + 32 * b;
      float m = fabsf(__uint_as_float(x[0]));
#pragma unroll
      for (int j = 1; j < 31; j += 2)
        m = max3_abs_nan(m, __uint_as_float(x[j]), __uint_as_float(x[j + 1]));
      m = max3_abs_nan(m, __uint_as_float(x[31]), __uint_as_float(x[31]));
      const uint32_t sc = scale_of(__float_as_uint(m) & 0x7FFFFFFFu, emax);
      const float k = inv_scale(sc);
      auto f = [&](int j) { return __fmul_rn(__uint_as_float(x[j]), k); };
      uint32_t w[8];
      if constexpr (QF == MXQ_E2M1) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = cvt_e2m1x8(f(8 * q), f(8 * q + 1), f(8 * q + 2), f(8 * q + 3), f(8 * q + 4),
                            f(8 * q + 5), f(8 * q + 6), f(8 * q + 7));
      } else if constexpr (QF == MXQ_E5M2) {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = cvt_e5m2x4(f(4 * q), f(4 * q + 1), f(4 * q + 2), f(4 * q + 3));
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = cvt_e4m3x4(f(4 * q), f(4 * q + 1), f(4 * q + 2), f(4 * q + 3));
      }
      if (sc == 255u) {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = 0u;
      }
      uint8_t* dst = crow + b * cb;
      if constexpr (QF == MXQ_E2M1) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      } else if (a.wide_stores) {
        st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      pace(pace_ns);
      sw |= sc << (8 * b);
    }
  }
  if (!MXQ_IN_BOUNDS(row < a.M && col0 + 32 * nblk <= a.N && (!a.q_scale_tc || nblk == 4),
                     &g_err_gemm, SITE_B_GEMM_QSCALE))
    return;
  if (a.q_scale_tc) {
    // one word of chunk (row / 128, col0 / 128): N % 128 == 0, so nblk == 4
    uint8_t* chunk = a.q_scales + ((row >> 7) * (int64_t(a.N) >> 7) + (col0 >> 7)) * 512;
    *reinterpret_cast<uint32_t*>(chunk + (row & 31) * 16 + ((row & 127) >> 5) * 4) = sw;
    return;
  }
  uint8_t* srow = a.q_scales + row * (int64_t(a.N) / 32) + col0 / 32;
  if (a.q_scale_words && nblk == 4) {
    *reinterpret_cast<uint32_t*>(srow) = sw;
  } else {
    for (int b = 0; b < nblk; ++b) srow[b] = static_cast<uint8_t>(sw >> (8 * b));
  }
}

// Work item t -> (mp, nt).  Tiles are visited in groups of `group` rows (or
// columns, when group_n): inside a group the grouped index runs fastest, so
// the clusters working at one time cover `group` panels of one operand and a
// few of the other, and the grouped operand's panels stay in L2 while the
// group sweeps the other dimension.
MXQ_DEV void tile_coords(int t, const GArgs& a, int& mp, int& nt) {
  const int n_g = a.group_n ? a.n_nt : a.n_mp;   // grouped dimension
  const int n_o = a.group_n ? a.n_mp : a.n_nt;   // swept dimension
  const int per_group = a.group * n_o;
  const int g = t / per_group;
  const int first = g * a.group;
  const int size = min(a.group, n_g - first);
  const int local = t - g * per_group;
  const int gi = first + local % size, oi = local / size;
  mp = a.group_n ? oi : gi;
  nt = a.group_n ? gi : oi;
}

// Problem of work item t: p advances monotonically as a role walks its
// items in increasing order.
MXQ_DEV int problem_of(const GGroup& g, int t, int p) {
  while (p + 1 < g.count && t >= g.p[p + 1].tile0) ++p;
  return p;
}

__global__ void __launch_bounds__(G_THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ GGroup g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G_STAGES * G_STAGE_BYTES);
  uint64_t* empty = full + G_STAGES;
  uint64_t* sf_ready = empty + G_STAGES;
  uint64_t* tmem_full = sf_ready + G_STAGES;
  uint64_t* tmem_empty = tmem_full + 1;      // leader: both CTAs drained the accumulator
  uint64_t* drain = tmem_empty + 1;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);
  // leader: the number of K stages the peer CTA's producer issued, written
  // by the peer when its producer stops (kNotYet until then)
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(abort_flag + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const GArgs& a0 = g.p[0];   // format, epilogue kind and wait limit of the launch
  if (threadIdx.x == 0) {
    for (int i = 0; i < g.count; ++i) {
      prefetch_tmap(&g.ta[i]);
      prefetch_tmap(&g.tb[i]);
      prefetch_tmap(&g.tsa[i]);
      prefetch_tmap(&g.tsb[i]);
    }
    for (int s = 0; s < G_STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);    // leader: one arrival, bytes of both CTAs
      mbar_init(smem_u32(&empty[s]), 1);
      mbar_init(smem_u32(&sf_ready[s]), 2);  // two scale-copy warps
    }
    mbar_init(smem_u32(tmem_full), 1);
    mbar_init(smem_u32(tmem_empty), 8 * G_CLUSTER);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *peer_issued = kNotYet;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_base_slot), G_TMEM_COLS);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs exist before anyone signals the peer
  tc_fence_after();
  griddep_wait();  // the previous kernel's writes (codes, scales) are visible
  griddep_launch_dependents();
  const int cid = blockIdx.x / G_CLUSTER, ncl = gridDim.x / G_CLUSTER;
  const uint32_t tmem = *tmem_base_slot;
  const int n_tiles = g.n_tiles;
  const uint64_t tmo = a0.timeout_ns;

  const int n_sfa = a0.fp4 ? 2 : 1;           // 512-byte chunks of own-A scales per stage
  const uint32_t sf_bytes_a = 512u * n_sfa;   // per 128 rows
  // bytes one CTA brings into a stage; the leader's barrier counts both CTAs
  const uint32_t cta_tx = G_A_BYTES + G_B_BYTES + 3 * sf_bytes_a;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      // every load of both CTAs completes on the leader's stage barrier
      const uint32_t full0 = map_to_rank(smem_u32(&full[0]), 0);
      uint32_t s = 0, phase = 0, issued = 0;
      bool ok = true;
      int pi = 0;
      for (int t = cid; t < n_tiles && ok; t += ncl) {
        pi = problem_of(g, t, pi);
        const GArgs& a = g.p[pi];
        const int nk = a.nk;
        int mp, nt;
        tile_coords(t - a.tile0, a, mp, nt);
        if (!MXQ_IN_BOUNDS(mp >= 0 && mp < a.n_mp && nt >= 0 && nt < a.n_nt, &g_err_gemm,
                           SITE_B_GEMM_TILE)) {
          ok = false;   // the MMA lane then waits out its bounded wait
          break;
        }
        const int mt = G_CLUSTER * mp + static_cast<int>(rank);   // this CTA's 128-row tile
        const int srow_a = mt * a.kc_per_row;                     // first scale chunk rows
        const int srow_b0 = (2 * nt) * a.kc_per_row, srow_b1 = (2 * nt + 1) * a.kc_per_row;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_try_wait_cluster(smem_u32(&empty[s]), phase ^ 1) &&
              !gwait(smem_u32(&empty[s]), phase ^ 1, tmo, abort_flag)) {
            if (!*abort_flag) gabort(abort_flag, SITE_GEMM_EMPTY);
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(smem + s * G_STAGE_BYTES);
          const uint32_t bar = full0 + s * 8;
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[s]), G_CLUSTER * cta_tx);
          tma_load_2d_pair(st, &g.ta[pi], bar, ks * G_BKB, mt * G_BM);
          tma_load_2d_pair(st + G_A_BYTES, &g.tb[pi], bar, ks * G_BKB,
                           nt * G_BN + static_cast<int>(rank) * G_BN_CTA);
          const int kc = ks * n_sfa;
          tma_load_2d_pair(st + G_A_BYTES + G_B_BYTES, &g.tsa[pi], bar, 0, srow_a + kc);
          tma_load_2d_pair(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES, &g.tsb[pi], bar, 0,
                           srow_b0 + kc);
          tma_load_2d_pair(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES + sf_bytes_a, &g.tsb[pi], bar,
                           0, srow_b1 + kc);
          ++issued;
          if (++s == G_STAGES) { s = 0; phase ^= 1; }
        }
      }
      if (!leader) {
        // tell the leader how many stages this CTA's copies were issued for
        st_cluster_u32(map_to_rank(smem_u32(const_cast<uint32_t*>(peer_issued)), 0), issued);
      } else if (!ok) {
        // Every copy of both CTAs signals the leader's stage barriers, and
        // the peer's land in the peer's shared memory, which stays in use
        // until the final cluster barrier.  So before that barrier the leader
        // waits (bounded) for the copies of the last stages either CTA
        // issued; stages only the peer issued get their expected bytes here.
        const uint64_t t0 = global_ns();
        while (*peer_issued == kNotYet && global_ns() - t0 <= 2 * tmo + 1000000) {
        }
        uint32_t last = issued;
        if (*peer_issued != kNotYet && *peer_issued > last) last = *peer_issued;
        for (uint32_t k = last > G_STAGES ? last - G_STAGES : 0; k < last; ++k) {
          if (k >= issued) mbar_arrive_expect_tx(smem_u32(&full[k % G_STAGES]), cta_tx);
          if (!mbar_wait(smem_u32(&full[k % G_STAGES]), (k / G_STAGES) & 1, tmo)) {
            // a stage one CTA never issued: later stages were not issued either
            record_error(&g_err_gemm, MXQ_ERR_TIMEOUT, SITE_GEMM_FULL);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- pair-MMA issuer (leader CTA) ----------------
      // Everything that does not change per stage is computed once: each
      // tcgen05 instruction costs the issuing thread ~100 cycles, so the
      // loop keeps nothing else on its path.
      const uint32_t fmt_code = static_cast<uint32_t>(a0.elem_code);
      uint32_t idesc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sf_id = a0.fp4 ? ((2 * j) & 3) : j;
        idesc[j] = idesc_block_scaled(fmt_code, sf_id, sf_id);
      }
      const uint32_t st0 = smem_u32(smem);
      const uint64_t adesc_s0 = smem_desc(st0, 0, 1024, 2);
      const uint64_t bdesc_s0 = smem_desc(st0 + G_A_BYTES, 0, 1024, 2);
      constexpr uint32_t kStageDesc = G_STAGE_BYTES >> 4;   // stage stride in descriptor units
      const bool fp4 = a0.fp4 != 0;
      uint32_t s = 0, phase = 0, tile_i = 0;
      bool ok = true;
      int pi = 0;
      for (int t = cid; t < n_tiles && ok; t += ncl, ++tile_i) {
        pi = problem_of(g, t, pi);
        const int nk = g.p[pi].nk;
        if (!mbar_try_wait_cluster(smem_u32(tmem_empty), (tile_i & 1) ^ 1) &&
            !gwait(smem_u32(tmem_empty), (tile_i & 1) ^ 1, tmo, abort_flag)) {
          if (!*abort_flag) gabort(abort_flag, SITE_GEMM_TMEM_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_try_wait_cluster(smem_u32(&sf_ready[s]), phase) &&
              !gwait(smem_u32(&sf_ready[s]), phase, tmo, abort_flag)) {
            if (!*abort_flag) gabort(abort_flag, SITE_GEMM_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + G_SFA_COL0 + 8 * s;
          const uint32_t sfb_t = tmem + G_SFB_COL0 + 16 * s;
          const uint64_t ad = adesc_s0 + s * kStageDesc;
          const uint64_t bd = bdesc_s0 + s * kStageDesc;
          // scales of this stage are already in tensor memory (sf_ready)
          if (fp4) {
            // each MMA consumes 32 bytes of K (K=64 packed E2M1), k-blocks 2j, 2j+1
            mma_mxf4_pair(tmem, ad, bd, idesc[0], sfa_t, sfb_t, ks > 0 ? 1u : 0u);
            mma_mxf4_pair(tmem, ad + 2, bd + 2, idesc[1], sfa_t, sfb_t, 1u);
            mma_mxf4_pair(tmem, ad + 4, bd + 4, idesc[2], sfa_t + 4, sfb_t + 8, 1u);
            mma_mxf4_pair(tmem, ad + 6, bd + 6, idesc[3], sfa_t + 4, sfb_t + 8, 1u);
          } else {
            // each MMA consumes 32 bytes of K (K=32 E4M3), k-block j
            mma_mxf8_pair(tmem, ad, bd, idesc[0], sfa_t, sfb_t, ks > 0 ? 1u : 0u);
            mma_mxf8_pair(tmem, ad + 2, bd + 2, idesc[1], sfa_t, sfb_t, 1u);
            mma_mxf8_pair(tmem, ad + 4, bd + 4, idesc[2], sfa_t, sfb_t, 1u);
            mma_mxf8_pair(tmem, ad + 6, bd + 6, idesc[3], sfa_t, sfb_t, 1u);
          }
          tc_commit_pair_mc(smem_u32(&empty[s]), 0x3);   // stage free in both CTAs
          if (++s == G_STAGES) { s = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_mc(smem_u32(tmem_full), 0x3);     // accumulators ready in both CTAs
      }
      // all pair MMAs issued by this thread are complete before teardown
      tc_commit_pair_mc(smem_u32(drain), 0x1);
      if (!mbar_wait(smem_u32(drain), 0, tmo))
        record_error(&g_err_gemm, MXQ_ERR_TIMEOUT, SITE_GEMM_DRAIN);
    }
  } else if (warp >= 10) {
    if (lane == 0 && leader) {
      // ---------------- scale copiers (leader CTA, warps 10 and 11) -------
      // Copy each stage's scales into both CTAs' tensor memory ahead of the
      // MMA lane and signal it through sf_ready (two arrivals per stage).
      // Separate threads get the scales into tensor memory as soon as a
      // stage lands, while the MMA lane is still busy with earlier stages;
      // copies issued by the MMA lane itself, just before each stage's MMAs,
      // measured 10-30% slower.  E4M3: warp 10 copies the A scales and those
      // of B rows 0-127, warp 11 those of B rows 128-255.  E2M1 (twice the
      // chunks): warp 10 the two A chunks and the first B chunk, warp 11 the
      // other three.
      const bool first = warp == 10;
      const uint32_t st0 = smem_u32(smem);
      const bool fp4 = a0.fp4 != 0;
      uint32_t s = 0, phase = 0;
      uint32_t total = 0;   // K stages of this cluster's work items
      {
        int pi = 0;
        for (int t = cid; t < n_tiles; t += ncl) {
          pi = problem_of(g, t, pi);
          total += static_cast<uint32_t>(g.p[pi].nk);
        }
      }
      for (uint32_t it = 0; it < total; ++it) {
        if (!mbar_try_wait_cluster(smem_u32(&full[s]), phase) &&
            !gwait(smem_u32(&full[s]), phase, tmo, abort_flag)) {
          if (!*abort_flag) gabort(abort_flag, SITE_GEMM_FULL);
          break;
        }
        tc_fence_after();
        const uint32_t sfa_smem = st0 + s * G_STAGE_BYTES + G_A_BYTES + G_B_BYTES;
        const uint32_t sfb_smem = sfa_smem + G_SFA_BYTES;
        const uint32_t sfa_t = tmem + G_SFA_COL0 + 8 * s;
        const uint32_t sfb_t = tmem + G_SFB_COL0 + 16 * s;
        // A: chunk c -> columns +4c.  B: k-chunk c of rows 0-127 -> +8c,
        // rows 128-255 -> +8c+4 (rows 128-255 start sf_bytes_a into the slot).
        // E4M3: 3 chunks per stage (2 + 1); E2M1: 6 chunks (3 + 3).
        if (fp4) {
          if (first) {
            tc_cp_sf_pair(sfa_t, sfa_smem);
            tc_cp_sf_pair(sfa_t + 4, sfa_smem + 512);
            tc_cp_sf_pair(sfb_t, sfb_smem);
          } else {
            tc_cp_sf_pair(sfb_t + 8, sfb_smem + 512);
            tc_cp_sf_pair(sfb_t + 4, sfb_smem + sf_bytes_a);
            tc_cp_sf_pair(sfb_t + 12, sfb_smem + sf_bytes_a + 512);
          }
        } else if (first) {
          tc_cp_sf_pair(sfa_t, sfa_smem);
          tc_cp_sf_pair(sfb_t, sfb_smem);
        } else {
          tc_cp_sf_pair(sfb_t + 4, sfb_smem + sf_bytes_a);
        }
        tc_commit_pair_mc(smem_u32(&sf_ready[s]), 0x1);
        if (++s == G_STAGES) { s = 0; phase ^= 1; }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9, both CTAs) ----------------
    const int quad = warp & 3;                   // tensor-memory lane quadrant
    const int colh = (warp - 2) >> 2;            // 0: columns 0-127, 1: 128-255
    const uint32_t empty_leader = map_to_rank(smem_u32(tmem_empty), 0);
    uint32_t tile_i = 0;
    int pi = 0;
    for (int t = cid; t < n_tiles; t += ncl, ++tile_i) {
      pi = problem_of(g, t, pi);
      const GArgs& a = g.p[pi];
      if (!gwait(smem_u32(tmem_full), tile_i & 1, tmo, abort_flag)) {
        if (lane == 0 && !*abort_flag) gabort(abort_flag, SITE_GEMM_TMEM_FULL);
        break;
      }
      tc_fence_after();
      uint32_t v[128];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + colh * 128;
      MXQ_TMEM_LD32(taddr + 0, (v + 0));
      MXQ_TMEM_LD32(taddr + 32, (v + 32));
      MXQ_TMEM_LD32(taddr + 64, (v + 64));
      MXQ_TMEM_LD32(taddr + 96, (v + 96));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(empty_leader);

      int mp, nt;
      tile_coords(t - a.tile0, a, mp, nt);
      const uint32_t pn = t + ncl < n_tiles ? a.pace_ns : 0u;   // last tile: no pacing
      const int64_t row = (int64_t(mp) * G_CLUSTER + rank) * G_BM + quad * 32 + lane;
      const int64_t col0 = int64_t(nt) * G_BN + colh * 128;
      if (a.q_scale_tc && row >= a.M && row < ((int64_t(a.M) + 127) & ~int64_t(127)) &&
          col0 < a.N) {
        // lines past M inside the last 128-line tile: zero scales, as in
        // every chunk-layout buffer
        uint8_t* chunk = a.q_scales + ((row >> 7) * (int64_t(a.N) >> 7) + (col0 >> 7)) * 512;
        *reinterpret_cast<uint32_t*>(chunk + (row & 31) * 16 + ((row & 127) >> 5) * 4) = 0u;
      }
      if (row < a.M && col0 < a.N &&
          MXQ_IN_BOUNDS(mp >= 0 && mp < a.n_mp && nt >= 0 && nt < a.n_nt && row >= 0 &&
                            col0 >= 0 && (col0 & 31) == 0,
                        &g_err_gemm, SITE_B_GEMM_STORE)) {
        const int64_t ncols = (a.N - col0) < 128 ? (a.N - col0) : 128;
        if (a.out_q) {
          const int nblk = static_cast<int>(ncols >> 5);   // N % 32 == 0
          if (a.q_fmt == MXQ_E2M1) store_row_codes<MXQ_E2M1>(v, a, row, col0, nblk, pn);
          else if (a.q_fmt == MXQ_E5M2) store_row_codes<MXQ_E5M2>(v, a, row, col0, nblk, pn);
          else store_row_codes<MXQ_E4M3>(v, a, row, col0, nblk, pn);
        } else if (a.out_bf16) {
          __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(a.C) + row * a.N + col0;
          uint32_t p[64];
#pragma unroll
          for (int u = 0; u < 64; ++u) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(v[2 * u]),
                                                           __uint_as_float(v[2 * u + 1]));
            p[u] = *reinterpret_cast<const uint32_t*>(&b);
          }
          if (a.wide_stores) {
#pragma unroll
            for (int c = 0; c < 128; c += 16)
              if (c < ncols) {
                st_global_v8(crow + c, p[c / 2], p[c / 2 + 1], p[c / 2 + 2], p[c / 2 + 3],
                             p[c / 2 + 4], p[c / 2 + 5], p[c / 2 + 6], p[c / 2 + 7]);
                pace(pn);
              }
          } else {
#pragma unroll
            for (int c = 0; c < 128; c += 8)
              if (c < ncols) {
                *reinterpret_cast<uint4*>(crow + c) =
                    make_uint4(p[c / 2], p[c / 2 + 1], p[c / 2 + 2], p[c / 2 + 3]);
                pace(pn >> 1);
              }
          }
        } else {
          float* crow = static_cast<float*>(a.C) + row * a.N + col0;
          if (a.wide_stores) {
#pragma unroll
            for (int c = 0; c < 128; c += 8)
              if (c < ncols) {
                st_global_v8(crow + c, v[c], v[c + 1], v[c + 2], v[c + 3], v[c + 4], v[c + 5],
                             v[c + 6], v[c + 7]);
                pace(pn);
              }
          } else {
#pragma unroll
            for (int c = 0; c < 128; c += 4)
              if (c < ncols) {
                *reinterpret_cast<uint4*>(crow + c) = make_uint4(v[c], v[c + 1], v[c + 2], v[c + 3]);
                pace(pn >> 1);
              }
          }
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, G_TMEM_COLS);
}

// Row-major E8M0 scales [rows][kb] of A and of B -> chunked tensor-core
// layout, zero padded to rows_p rows and kbp blocks, both operands in one
// launch.  One thread writes the four blocks of one row in one chunk.
struct SfSide {
  const uint8_t* s;
  int64_t rows, rows_p;
  uint8_t* out;
};

__global__ void __launch_bounds__(256)
    sf_to_chunks(SfSide sa, SfSide sb, int64_t kb, int64_t kbp) {
  const int64_t kcs = kbp / 4;
  const int64_t total_a = sa.rows_p * kcs, total = total_a + sb.rows_p * kcs;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const bool is_a = i < total_a;
    const SfSide& d = is_a ? sa : sb;
    const int64_t j = is_a ? i : i - total_a;
    const int64_t r = j % d.rows_p, kc = j / d.rows_p;
    uint32_t w = 0;
    if (r < d.rows) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = kc * 4 + u;
        if (k < kb) w |= static_cast<uint32_t>(d.s[r * kb + k]) << (8 * u);
      }
    }
    const int64_t rt = r / 128, rr = r % 128;
    if (!MXQ_IN_BOUNDS(r < d.rows_p && kc < kcs && kc * 4 + 3 < kbp, &g_err_gemm,
                       SITE_B_SF_CHUNKS))
      continue;
    uint8_t* chunk = d.out + (rt * kcs + kc) * 512;
    *reinterpret_cast<uint32_t*>(chunk + (rr % 32) * 16 + (rr / 32) * 4) = w;
  }
}

struct Plan {
  int64_t kbytes, kb, kbp, mp, np, ws_a, ws_b;
  int skb;
};

bool make_plan(int64_t M, int64_t N, int64_t K, int fmt, Plan& p) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0) return false;
  if (fmt != MXQ_E4M3 && fmt != MXQ_E2M1 && fmt != MXQ_E5M2) return false;
  p.kbytes = fmt != MXQ_E2M1 ? K : K / 2;
  p.kb = K / 32;
  p.skb = fmt != MXQ_E2M1 ? 4 : 8;  // k-blocks per 128-byte stage
  p.kbp = (p.kb + p.skb - 1) / p.skb * p.skb;
  p.mp = (M + G_CLUSTER * G_BM - 1) / (G_CLUSTER * G_BM) * (G_CLUSTER * G_BM);
  p.np = (N + G_BN - 1) / G_BN * G_BN;
  p.ws_a = p.mp * p.kbp;
  p.ws_b = p.np * p.kbp;
  return true;
}

// Clusters of G_CLUSTER GEMM CTAs that fit on the device at once (cached per
// device).
int max_gemm_clusters(cudaLaunchConfig_t cfg) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(G_CLUSTER * sm_count()), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count() / G_CLUSTER;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

uint32_t take_gemm_error() {
  uint32_t h = 0;
  if (cudaMemcpyFromSymbol(&h, g_err_gemm, sizeof(h)) != cudaSuccess) return MXQ_ERR_CUDA;
  if (h) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_err_gemm, &z, sizeof(z));
  }
  return h;
}

}  // namespace mxq

using namespace mxq;

extern "C" size_t mxq_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int fmt) {
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return 0;
  return static_cast<size_t>(p.ws_a + p.ws_b);
}

namespace {

// What the epilogue writes: C as fp32 or bf16, or row-wise MX codes of C
// (q_fmt) with their scales.
struct OutSpec {
  void* C;
  int kind;            // 0: fp32, 1: bf16, 2: MX codes
  int q_fmt;
  uint8_t* q_scales;
  int q_scale_layout;  // mxq_scale_layout of q_scales
};

// The argument checks of one problem: sizes, formats, pointers, alignment,
// workspace.  No CUDA call.
mxq_status gemm_validate(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                         int fmt, int64_t M, int64_t N, int64_t K, const void* C,
                         const void* workspace, size_t workspace_bytes, int scale_layout) {
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return MXQ_ERR_ARG;
  if (scale_layout != MXQ_SCALES_ROWMAJOR && scale_layout != MXQ_SCALES_TC) return MXQ_ERR_ARG;
  const bool tc = scale_layout == MXQ_SCALES_TC;
  if (!A || !sA || !B || !sB || !C || (!tc && !workspace)) return MXQ_ERR_ARG;
  if (tc && K % (fmt == MXQ_E2M1 ? 256 : 128) != 0) return MXQ_ERR_ARG;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return MXQ_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MXQ_ERR_ALIGN;
  if (tc && (!aligned16(sA) || !aligned16(sB))) return MXQ_ERR_ALIGN;
  if (!tc && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MXQ_ERR_ALIGN;
  if (!tc && workspace_bytes < static_cast<size_t>(p.ws_a + p.ws_b)) return MXQ_ERR_WORKSPACE;
  return MXQ_OK;
}

// Validates one problem, runs its scale re-layout pass (row-major scales),
// and fills its launch arguments and tensor maps (tile0 left at 0).
mxq_status gemm_prepare(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                        int fmt, int64_t M, int64_t N, int64_t K, const OutSpec& out,
                        void* workspace, size_t workspace_bytes, void* stream, int scale_layout,
                        GArgs& a, CUtensorMap& ta, CUtensorMap& tb, CUtensorMap& tsa,
                        CUtensorMap& tsb) {
  void* C = out.C;
  const mxq_status vs = gemm_validate(A, sA, B, sB, fmt, M, N, K, C, workspace, workspace_bytes,
                                      scale_layout);
  if (vs != MXQ_OK) return vs;
  Plan p;
  make_plan(M, N, K, fmt, p);
  // scales already in the tensor-core chunk layout: no re-layout pass and
  // no workspace; the chunks are read in place
  const bool tc = scale_layout == MXQ_SCALES_TC;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (!tc) {
    const int64_t total = (p.mp + p.np) * (p.kbp / 4);
    const int grid = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4 * sm_count()));
    const SfSide sa{sA, M, p.mp, ws}, sb{sB, N, p.np, ws + p.ws_a};
    sf_to_chunks<<<grid, 256, 0, st>>>(sa, sb, p.kb, p.kbp);
  }

  if (tensor_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, static_cast<uint64_t>(p.kbytes),
                    static_cast<uint64_t>(M), static_cast<uint64_t>(p.kbytes), G_BKB, G_BM,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
    return MXQ_ERR_CUDA;
  if (tensor_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, static_cast<uint64_t>(p.kbytes),
                    static_cast<uint64_t>(N), static_cast<uint64_t>(p.kbytes), G_BKB, G_BN_CTA,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
    return MXQ_ERR_CUDA;

  // Scale chunks as 2-D tensors of 512-byte rows (128 x uint32), one row per
  // (128-row tile, k-chunk): a stage loads n_sfa consecutive rows.  The
  // workspace holds chunks for the padded 256-row tiles; caller-provided
  // chunks cover only the existing 128-row tiles, and loads of the missing
  // ones read the zero fill.
  {
    const int n_sfa = fmt == MXQ_E2M1 ? 2 : 1;
    const int64_t kcs = p.kbp / 4;
    for (int which = 0; which < 2; ++which) {
      const int64_t lines = which == 0 ? (tc ? M : p.mp) : (tc ? N : p.np);
      const int64_t rows = (lines + G_BM - 1) / G_BM * kcs;
      const void* base = tc ? static_cast<const void*>(which == 0 ? sA : sB)
                            : static_cast<const void*>(ws + (which == 0 ? 0 : p.ws_a));
      if (tensor_map_2d(which == 0 ? &tsa : &tsb, CU_TENSOR_MAP_DATA_TYPE_UINT32, base, 128,
                        static_cast<uint64_t>(rows), 512, 128, static_cast<uint32_t>(n_sfa),
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) !=
          CUDA_SUCCESS)
        return MXQ_ERR_CUDA;
    }
  }

  a = GArgs{};
  a.M = static_cast<int32_t>(M);
  a.N = static_cast<int32_t>(N);
  a.n_mp = static_cast<int32_t>(p.mp / (G_CLUSTER * G_BM));
  a.n_nt = static_cast<int32_t>(p.np / G_BN);
  // one work item = one 256x256 pair tile (one cluster)
  if (int64_t(a.n_mp) * a.n_nt >= (int64_t(1) << 31)) return MXQ_ERR_ARG;
  a.n_tiles = a.n_mp * a.n_nt;
  {
    // Raster: tiles run in groups of `group` panels of one operand (the
    // grouped one) while the group sweeps all panels of the other.  The
    // grouped panels are touched by every wave of the group and stay in L2
    // (budget 64 MB); the swept operand streams from DRAM once per group.
    // Modeled DRAM bytes: grouped_total + swept_total * n_groups; the
    // orientation and group size with the fewest bytes win.
    const double l2_budget = 64.0 * (1 << 20);
    const double panel = double(2 * G_BM) * double(p.kbytes);
    const int g_fit = static_cast<int>(std::max(1.0, std::floor(l2_budget / panel)));
    const double a_bytes = double(p.mp) * p.kbytes, b_bytes = double(p.np) * p.kbytes;
    double best = -1.0;
    for (int orient = 0; orient < 2; ++orient) {
      const int n_g = orient ? a.n_nt : a.n_mp;
      const double grouped = orient ? b_bytes : a_bytes, swept = orient ? a_bytes : b_bytes;
      for (int g = 1; g <= std::min(g_fit, n_g); ++g) {
        const double bytes = grouped + swept * std::ceil(double(n_g) / g);
        if (best < 0.0 || bytes < best - 1.0) {
          best = bytes;
          a.group_n = orient;
          a.group = g;
        }
      }
    }
  }
  a.nk = static_cast<int32_t>((p.kbytes + G_BKB - 1) / G_BKB);
  a.kc_per_row = static_cast<int32_t>(p.kbp / 4);
  a.sfa = tc ? sA : ws;
  a.sfb = tc ? sB : ws + p.ws_a;
  a.C = C;
  a.out_bf16 = out.kind == 1;
  a.out_q = out.kind == 2;
  a.q_fmt = out.q_fmt;
  a.q_scales = out.q_scales;
  a.q_scale_words = (reinterpret_cast<uintptr_t>(out.q_scales) & 3u) == 0 && (N / 32) % 4 == 0;
  a.q_scale_tc = out.kind == 2 && out.q_scale_layout == MXQ_SCALES_TC;
  a.fp4 = fmt == MXQ_E2M1;
  // kind::mxf8f6f4 element types: E4M3 = 0, E5M2 = 1; kind::mxf4: E2M1 = 1
  a.elem_code = fmt == MXQ_E4M3 ? 0 : 1;
  // 256-bit stores need 32-byte aligned rows: fp32 rows of N % 8 == 0,
  // bf16 rows of N % 16 == 0, one-byte code rows of N % 32 == 0
  const int wide_mult = out.kind == 0 ? 8 : (out.kind == 1 ? 16 : 32);
  a.wide_stores = (reinterpret_cast<uintptr_t>(C) & 31u) == 0 && N % wide_mult == 0;
  // Store pacing: a thread's stores of one tile are spread over roughly a
  // third to a half of the next tile's main loop, modeled as nk stages of
  // 64 ns (E4M3/E5M2) or 128 ns (E2M1; its stages are longer and its ring
  // more sensitive to load latency), capped at 1 us per store.  Calibrated
  // by timing 64-512 ns pauses on the block-pass shapes.
  {
    const int stores = out.kind == 0 ? 16 : (out.kind == 1 ? 8 : 4);   // 32-byte stores per row
    const int64_t per_stage_ns = fmt == MXQ_E2M1 ? 128 : 64;
    a.pace_ns = static_cast<uint32_t>(std::min<int64_t>(1000, a.nk * per_stage_ns / stores));
  }
  a.timeout_ns = wait_timeout_ns();
  // every field the kernel dereferences or divides by is set
  if (!a.C || !a.sfa || !a.sfb || a.nk <= 0 || a.kc_per_row <= 0 || a.group <= 0 ||
      a.n_tiles <= 0 || a.n_nt <= 0 || a.n_mp <= 0 || (a.out_q && !a.q_scales))
    return MXQ_ERR_ARG;

  return MXQ_OK;
}

// Launches the prepared problems g.p[0..count) as one persistent grid.
mxq_status gemm_run(GGroup& g, void* stream) {
  int32_t tiles = 0;
  for (int i = 0; i < g.count; ++i) {
    if (int64_t(tiles) + g.p[i].n_tiles >= (int64_t(1) << 31)) return MXQ_ERR_ARG;
    g.p[i].tile0 = tiles;
    tiles += g.p[i].n_tiles;
  }
  g.n_tiles = tiles;
  if (g.count < 1 || g.count > G_MAX_GROUP || tiles <= 0) return MXQ_ERR_ARG;
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(mx_gemm_kernel), G_SMEM))
    return MXQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = G_CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(G_THREADS, 1, 1);
  cfg.dynamicSmemBytes = G_SMEM;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = max_gemm_clusters(cfg);
  // persistent grid (every cluster resident): it may start while the
  // previous kernel on the stream drains, and waits for it in the kernel
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  if (max_clusters <= 0) return MXQ_ERR_CUDA;
  cfg.gridDim = dim3(static_cast<unsigned>(G_CLUSTER * std::min(tiles, max_clusters)), 1, 1);
  if (cudaLaunchKernelEx(&cfg, mx_gemm_kernel, g) != cudaSuccess) return MXQ_ERR_CUDA;
  return launch_status();
}

mxq_status gemm_launch(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, int fmt,
                       int64_t M, int64_t N, int64_t K, const OutSpec& out, void* workspace,
                       size_t workspace_bytes, void* stream, int scale_layout) {
  GGroup g;
  memset(&g, 0, sizeof(g));
  const mxq_status st = gemm_prepare(A, sA, B, sB, fmt, M, N, K, out, workspace, workspace_bytes,
                                     stream, scale_layout, g.p[0], g.ta[0], g.tb[0], g.tsa[0],
                                     g.tsb[0]);
  if (st != MXQ_OK) return st;
  g.count = 1;
  return gemm_run(g, stream);
}

}  // namespace

extern "C" mxq_status mxq_gemm(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                               int fmt, int64_t M, int64_t N, int64_t K, void* C, int out_dtype,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (out_dtype != MXQ_OUT_F32 && out_dtype != MXQ_OUT_BF16) return MXQ_ERR_ARG;
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return MXQ_ERR_ARG;
  if (N % (out_dtype == MXQ_OUT_F32 ? 4 : 8) != 0) return MXQ_ERR_ALIGN;
  const OutSpec out{C, out_dtype == MXQ_OUT_BF16 ? 1 : 0, 0, nullptr, MXQ_SCALES_ROWMAJOR};
  return gemm_launch(A, sA, B, sB, fmt, M, N, K, out, workspace, workspace_bytes, stream,
                     MXQ_SCALES_ROWMAJOR);
}

extern "C" mxq_status mxq_gemm_ex(const void* A, const uint8_t* sA, const void* B,
                                  const uint8_t* sB, int fmt, int64_t M, int64_t N, int64_t K,
                                  void* C, int out_dtype, int scale_layout, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (out_dtype != MXQ_OUT_F32 && out_dtype != MXQ_OUT_BF16) return MXQ_ERR_ARG;
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return MXQ_ERR_ARG;
  if (N % (out_dtype == MXQ_OUT_F32 ? 4 : 8) != 0) return MXQ_ERR_ALIGN;
  const OutSpec out{C, out_dtype == MXQ_OUT_BF16 ? 1 : 0, 0, nullptr, MXQ_SCALES_ROWMAJOR};
  return gemm_launch(A, sA, B, sB, fmt, M, N, K, out, workspace, workspace_bytes, stream,
                     scale_layout);
}

extern "C" mxq_status mxq_gemm_quantize(const void* A, const uint8_t* sA, const void* B,
                                        const uint8_t* sB, int fmt, int64_t M, int64_t N,
                                        int64_t K, int out_fmt, void* out_codes,
                                        uint8_t* out_scales, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (out_fmt != MXQ_E4M3 && out_fmt != MXQ_E5M2 && out_fmt != MXQ_E2M1) return MXQ_ERR_ARG;
  if (!out_scales) return MXQ_ERR_ARG;
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return MXQ_ERR_ARG;
  if (N % 32 != 0) return MXQ_ERR_ARG;
  const OutSpec out{out_codes, 2, out_fmt, out_scales, MXQ_SCALES_ROWMAJOR};
  return gemm_launch(A, sA, B, sB, fmt, M, N, K, out, workspace, workspace_bytes, stream,
                     MXQ_SCALES_ROWMAJOR);
}

extern "C" mxq_status mxq_gemm_quantize_ex(const void* A, const uint8_t* sA, const void* B,
                                           const uint8_t* sB, int fmt, int64_t M, int64_t N,
                                           int64_t K, int scale_layout, int out_fmt,
                                           void* out_codes, uint8_t* out_scales,
                                           int out_scale_layout, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (out_fmt != MXQ_E4M3 && out_fmt != MXQ_E5M2 && out_fmt != MXQ_E2M1) return MXQ_ERR_ARG;
  if (out_scale_layout != MXQ_SCALES_ROWMAJOR && out_scale_layout != MXQ_SCALES_TC)
    return MXQ_ERR_ARG;
  if (!out_scales) return MXQ_ERR_ARG;
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return MXQ_ERR_ARG;
  if (N % 32 != 0) return MXQ_ERR_ARG;
  if (out_scale_layout == MXQ_SCALES_TC) {
    if (N % (out_fmt == MXQ_E2M1 ? 256 : 128) != 0) return MXQ_ERR_ARG;
    if (!aligned16(out_scales)) return MXQ_ERR_ALIGN;
  }
  const OutSpec out{out_codes, 2, out_fmt, out_scales, out_scale_layout};
  return gemm_launch(A, sA, B, sB, fmt, M, N, K, out, workspace, workspace_bytes, stream,
                     scale_layout);
}

extern "C" mxq_status mxq_gemm_grouped(const mxq_gemm_problem* problems, int count, int fmt,
                                       void* stream) {
  if (!problems || count < 1 || count > G_MAX_GROUP) return MXQ_ERR_ARG;
  // every problem is checked before any of them is prepared
  for (int i = 0; i < count; ++i) {
    const mxq_gemm_problem& q = problems[i];
    if (q.out_dtype != MXQ_OUT_F32 && q.out_dtype != MXQ_OUT_BF16) return MXQ_ERR_ARG;
    Plan p;
    if (!make_plan(q.M, q.N, q.K, fmt, p)) return MXQ_ERR_ARG;
    if (q.N % (q.out_dtype == MXQ_OUT_F32 ? 4 : 8) != 0) return MXQ_ERR_ALIGN;
    const mxq_status vs = gemm_validate(q.A, q.sA, q.B, q.sB, fmt, q.M, q.N, q.K, q.C, nullptr, 0,
                                        MXQ_SCALES_TC);
    if (vs != MXQ_OK) return vs;
  }
  GGroup g;
  memset(&g, 0, sizeof(g));
  for (int i = 0; i < count; ++i) {
    const mxq_gemm_problem& q = problems[i];
    const OutSpec out{q.C, q.out_dtype == MXQ_OUT_BF16 ? 1 : 0, 0, nullptr, MXQ_SCALES_ROWMAJOR};
    const mxq_status st = gemm_prepare(q.A, q.sA, q.B, q.sB, fmt, q.M, q.N, q.K, out, nullptr, 0,
                                       stream, MXQ_SCALES_TC, g.p[i], g.ta[i], g.tb[i], g.tsa[i],
                                       g.tsb[i]);
    if (st != MXQ_OK) return st;
  }
  g.count = count;
  return gemm_run(g, stream);
}

// ---------------------------------------------------------------------------
// GEMM without caller-provided scratch
// ---------------------------------------------------------------------------
// Some callers cannot allocate device memory at call time: code embedded in a
// host application that owns the whole device memory pool and hands a plug-in
// only its input and output buffers, or code that runs under a fixed memory
// budget where allocating per call is forbidden.  For them the scale
// re-layout scratch lives in one fixed buffer inside this library.
//
// The buffer is a file-scope device array of kNoAllocScratchBytes (16 MiB).
// Every GPU that loads the library holds it until the process exits.  All
// calls share it and it keeps the previous call's contents; each call
// rewrites every byte it reads, so nothing needs clearing, but calls that
// overlap on the GPU (two streams at once, or two host threads) race on it.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch for each device, taken once per device
// with that device current (in host code the array's name is only a
// host-side stand-in, not a device address).
void* noalloc_scratch_ptr(mxq_status* st) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = MXQ_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      *st = MXQ_ERR_CUDA;
      return nullptr;
    }
    cache[dev] = p;
  }
  *st = MXQ_OK;
  return cache[dev];
}

}  // namespace

extern "C" mxq_status mxq_gemm_noalloc(const void* A, const uint8_t* sA, const void* B,
                                       const uint8_t* sB, int fmt, int64_t M, int64_t N,
                                       int64_t K, void* C, int out_dtype, void* stream) {
  const size_t need = mxq_gemm_workspace_size(M, N, K, fmt);
  if (need == 0) return MXQ_ERR_ARG;
  if (need > kNoAllocScratchBytes) return MXQ_ERR_WORKSPACE;
  mxq_status st;
  void* scratch = noalloc_scratch_ptr(&st);
  if (!scratch) return st;
  return mxq_gemm(A, sA, B, sB, fmt, M, N, K, C, out_dtype, scratch, kNoAllocScratchBytes,
                  stream);
}
