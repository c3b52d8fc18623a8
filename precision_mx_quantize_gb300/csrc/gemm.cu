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
// Kernel structure (one CTA per SM, persistent over 128x256 output tiles):
//   warp 0     TMA producer: A tile 128 rows x 128 B and B tile 256 rows x
//              128 B (128-byte swizzle) plus the stage's scale chunks (bulk
//              copies) into a 4-stage shared-memory ring;
//   warp 1     allocates the tensor memory; one lane copies the stage's
//              scales shared->tensor memory (tcgen05.cp) and issues the four
//              block-scaled MMAs of the stage into the fp32 accumulator
//              (128 lanes x 256 columns), then commits the stage back to the
//              producer;
//   warps 2-9  epilogue: each drains 32 accumulator lanes x 128 columns into
//              registers, frees the accumulator for the next tile, and
//              stores its rows while the next tile's main loop runs.
// The row-major scales are first rewritten (a small pre-pass kernel) into
// the tensor-core chunk layout in the caller's workspace: for every 128-row
// x 4-block chunk, byte (r % 32) * 16 + (r / 32) * 4 + (kb % 4).
#include <mutex>

#include "mxq_common.cuh"
#include "mxq_host.h"

namespace mxq {

__device__ uint32_t g_err_gemm;

namespace {

constexpr int G_BM = 128;                    // accumulator lanes (rows of A)
constexpr int G_BN = 256;                    // accumulator columns (rows of B)
constexpr int G_BKB = 128;                   // bytes of K per stage (one 128 B swizzle row)
constexpr int G_STAGES = 4;
constexpr int G_THREADS = 320;               // 10 warps
constexpr int G_A_BYTES = G_BM * G_BKB;      // 16 KB
constexpr int G_B_BYTES = G_BN * G_BKB;      // 32 KB
constexpr int G_SFA_BYTES = 1024;            // up to 2 chunks of 512 B
constexpr int G_SFB_BYTES = 2048;            // up to 4 chunks of 512 B
constexpr int G_STAGE_BYTES = G_A_BYTES + G_B_BYTES + G_SFA_BYTES + G_SFB_BYTES;
constexpr int G_SMEM = G_STAGES * G_STAGE_BYTES + 1024 + 256;
constexpr uint32_t G_TMEM_COLS = 512;
constexpr uint32_t G_SFA_COL0 = 256;         // 8 columns per stage
constexpr uint32_t G_SFB_COL0 = 256 + 8 * G_STAGES;  // 16 columns per stage

struct GArgs {
  int32_t M, N;
  int32_t n_mt, n_nt, n_tiles;
  int32_t nk;                 // K stages
  int32_t kc_per_row;         // 512-byte scale chunks per 128-row tile (KBp / 4)
  const uint8_t* sfa;         // chunked scales of A in the workspace
  const uint8_t* sfb;         // chunked scales of B
  void* C;
  int32_t out_bf16;
  int32_t fp4;
  uint64_t timeout_ns;
};

// ---- tcgen05 wrappers ------------------------------------------------------
MXQ_DEV void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MXQ_DEV void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

MXQ_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MXQ_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

MXQ_DEV void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

// Copy one 512-byte scale chunk (32 rows x 16 B) into 4 tensor-memory
// columns, replicated to all four 32-lane quadrants.
MXQ_DEV void tc_cp_sf(uint32_t taddr, uint32_t smem_addr) {
  const uint64_t d = smem_desc(smem_addr, 0, 128, 0);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

MXQ_DEV void mma_mxf8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                      uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
      : "memory");
}

MXQ_DEV void mma_mxf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                      uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
      : "memory");
}

// Instruction descriptor of a block-scaled MMA: K-major A and B, M = 128,
// N = 256, E8M0 scales, scale-factor byte ids a_sf / b_sf.
MXQ_DEV uint32_t idesc_block_scaled(uint32_t fmt_code, uint32_t a_sf, uint32_t b_sf) {
  uint32_t d = 0;
  d |= (b_sf & 3u) << 4;
  d |= (fmt_code & 7u) << 7;    // A format
  d |= (fmt_code & 7u) << 10;   // B format
  d |= static_cast<uint32_t>(G_BN >> 3) << 17;
  d |= 1u << 23;                // scale type: UE8M0
  d |= static_cast<uint32_t>(G_BM >> 4) << 24;
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

MXQ_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// A bounded wait that also gives up once another role has aborted.
MXQ_DEV bool gwait(uint32_t bar, uint32_t parity, uint64_t limit, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit) return false;
  }
  return true;
}

MXQ_DEV void gabort(volatile int* abort_flag, uint32_t site) {
  *abort_flag = 1;
  record_error(&g_err_gemm, MXQ_ERR_TIMEOUT, site);
}

__global__ void __launch_bounds__(G_THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G_STAGES * G_STAGE_BYTES);
  uint64_t* empty = full + G_STAGES;
  uint64_t* tmem_full = empty + G_STAGES;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* drain = tmem_empty + 1;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < G_STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(tmem_full), 1);
    mbar_init(smem_u32(tmem_empty), 8);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_base_slot), G_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;

  const int n_sfa = a.fp4 ? 2 : 1;            // 512-byte chunks of A scales per stage
  const uint32_t sf_bytes_a = 512u * n_sfa;   // per 128 rows
  const uint32_t stage_tx = G_A_BYTES + G_B_BYTES + 3 * sf_bytes_a;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x) {
        const int mt = t / a.n_nt, nt = t - mt * a.n_nt;
        for (int ks = 0; ks < a.nk; ++ks, ++it) {
          const uint32_t s = it % G_STAGES;
          if (!gwait(smem_u32(&empty[s]), ((it / G_STAGES) & 1) ^ 1, a.timeout_ns, abort_flag)) {
            if (!*abort_flag) gabort(abort_flag, SITE_GEMM_EMPTY);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * G_STAGE_BYTES;
          const uint32_t bar = smem_u32(&full[s]);
          mbar_arrive_expect_tx(bar, stage_tx);
          tma_load_2d(smem_u32(st), &tmA, bar, ks * G_BKB, mt * G_BM);
          tma_load_2d(smem_u32(st + G_A_BYTES), &tmB, bar, ks * G_BKB, nt * G_BN);
          const int kc = ks * n_sfa;  // first 512-byte chunk column of this stage
          const uint8_t* srcA = a.sfa + (int64_t(mt) * a.kc_per_row + kc) * 512;
          bulk_load(smem_u32(st + G_A_BYTES + G_B_BYTES), srcA, sf_bytes_a, bar);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint8_t* srcB = a.sfb + (int64_t(2 * nt + h) * a.kc_per_row + kc) * 512;
            bulk_load(smem_u32(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES + h * sf_bytes_a), srcB,
                      sf_bytes_a, bar);
          }
        }
      }
      if (!ok) {
        // bounded wait for the copies of the stages issued last
        for (int s = 0; s < G_STAGES; ++s) {
          if (it >= uint32_t(s + 1)) {
            const uint32_t k = it - 1 - s;
            gwait(smem_u32(&full[k % G_STAGES]), (k / G_STAGES) & 1, a.timeout_ns, abort_flag);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t fmt_code = a.fp4 ? 1u : 0u;  // kind::mxf4 E2M1 = 1, kind::mxf8f6f4 E4M3 = 0
      uint32_t it = 0, tile_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x, ++tile_i) {
        if (!gwait(smem_u32(tmem_empty), (tile_i & 1) ^ 1, a.timeout_ns, abort_flag)) {
          if (!*abort_flag) gabort(abort_flag, SITE_GEMM_TMEM_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < a.nk; ++ks, ++it) {
          const uint32_t s = it % G_STAGES;
          if (!gwait(smem_u32(&full[s]), (it / G_STAGES) & 1, a.timeout_ns, abort_flag)) {
            if (!*abort_flag) gabort(abort_flag, SITE_GEMM_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * G_STAGE_BYTES);
          const uint32_t sfa_smem = st + G_A_BYTES + G_B_BYTES;
          const uint32_t sfb_smem = sfa_smem + G_SFA_BYTES;
          const uint32_t sfa_col = G_SFA_COL0 + 8 * s;
          const uint32_t sfb_col = G_SFB_COL0 + 16 * s;
          // scales -> tensor memory.  A: chunk c -> columns sfa_col + 4c.
          // B: k-chunk c of rows 0-127 -> sfb_col + 8c, rows 128-255 -> +4.
          for (int c = 0; c < n_sfa; ++c) {
            tc_cp_sf(tmem + sfa_col + 4 * c, sfa_smem + 512 * c);
            tc_cp_sf(tmem + sfb_col + 8 * c, sfb_smem + 512 * c);
            tc_cp_sf(tmem + sfb_col + 8 * c + 4, sfb_smem + sf_bytes_a + 512 * c);
          }
          const uint64_t adesc0 = smem_desc(st, 0, 1024, 2);
          const uint64_t bdesc0 = smem_desc(st + G_A_BYTES, 0, 1024, 2);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // each MMA consumes 32 bytes of K: K=32 E4M3 or K=64 packed E2M1
            const uint64_t ad = adesc0 + static_cast<uint64_t>((32 * j) >> 4);
            const uint64_t bd = bdesc0 + static_cast<uint64_t>((32 * j) >> 4);
            const uint32_t accum = (ks > 0 || j > 0) ? 1u : 0u;
            if (a.fp4) {
              const uint32_t sf_id = (2 * j) & 3;           // k-blocks 2j, 2j+1
              const uint32_t chunk = (2 * j) >> 2;
              mma_mxf4(tmem, ad, bd, idesc_block_scaled(fmt_code, sf_id, sf_id),
                       tmem + sfa_col + 4 * chunk, tmem + sfb_col + 8 * chunk, accum);
            } else {
              mma_mxf8(tmem, ad, bd, idesc_block_scaled(fmt_code, j, j), tmem + sfa_col,
                       tmem + sfb_col, accum);
            }
          }
          tc_commit(smem_u32(&empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(tmem_full));
      }
      // all MMAs issued by this thread are complete before teardown
      tc_commit(smem_u32(drain));
      if (!mbar_wait(smem_u32(drain), 0, a.timeout_ns))
        record_error(&g_err_gemm, MXQ_ERR_TIMEOUT, SITE_GEMM_DRAIN);
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int quad = warp & 3;                   // tensor-memory lane quadrant
    const int colh = (warp - 2) >> 2;            // 0: columns 0-127, 1: 128-255
    uint32_t tile_i = 0;
    for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++tile_i) {
      if (!gwait(smem_u32(tmem_full), tile_i & 1, a.timeout_ns, abort_flag)) {
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
      if (lane == 0) mbar_arrive(smem_u32(tmem_empty));

      const int mt = t / a.n_nt, nt = t - mt * a.n_nt;
      const int64_t row = int64_t(mt) * G_BM + quad * 32 + lane;
      const int64_t col0 = int64_t(nt) * G_BN + colh * 128;
      if (row < a.M && col0 < a.N) {
        const int64_t ncols = (a.N - col0) < 128 ? (a.N - col0) : 128;
        if (a.out_bf16) {
          __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(a.C) + row * a.N + col0;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            if (c < ncols) {
              uint32_t p[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(v[c + 2 * u]),
                                                               __uint_as_float(v[c + 2 * u + 1]));
                p[u] = *reinterpret_cast<const uint32_t*>(&b);
              }
              *reinterpret_cast<uint4*>(crow + c) = make_uint4(p[0], p[1], p[2], p[3]);
            }
          }
        } else {
          float* crow = static_cast<float*>(a.C) + row * a.N + col0;
#pragma unroll
          for (int c = 0; c < 128; c += 4) {
            if (c < ncols)
              *reinterpret_cast<uint4*>(crow + c) = make_uint4(v[c], v[c + 1], v[c + 2], v[c + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, G_TMEM_COLS);
}

// Row-major E8M0 scales [rows][kb] -> chunked tensor-core layout, zero padded
// to rows_p rows and kbp blocks.  One thread writes the four blocks of one
// row in one chunk.
__global__ void __launch_bounds__(256)
    sf_to_chunks(const uint8_t* __restrict__ s, int64_t rows, int64_t kb, int64_t rows_p,
                 int64_t kbp, uint8_t* __restrict__ out) {
  const int64_t kcs = kbp / 4;
  const int64_t total = rows_p * kcs;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i % rows_p, kc = i / rows_p;
    uint32_t w = 0;
    if (r < rows) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = kc * 4 + u;
        if (k < kb) w |= static_cast<uint32_t>(s[r * kb + k]) << (8 * u);
      }
    }
    const int64_t rt = r / 128, rr = r % 128;
    uint8_t* chunk = out + (rt * kcs + kc) * 512;
    *reinterpret_cast<uint32_t*>(chunk + (rr % 32) * 16 + (rr / 32) * 4) = w;
  }
}

struct Plan {
  int64_t kbytes, kb, kbp, mp, np, ws_a, ws_b;
  int skb;
};

bool make_plan(int64_t M, int64_t N, int64_t K, int fmt, Plan& p) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0) return false;
  if (fmt != MXQ_E4M3 && fmt != MXQ_E2M1) return false;
  p.kbytes = fmt == MXQ_E4M3 ? K : K / 2;
  p.kb = K / 32;
  p.skb = fmt == MXQ_E4M3 ? 4 : 8;  // k-blocks per 128-byte stage
  p.kbp = (p.kb + p.skb - 1) / p.skb * p.skb;
  p.mp = (M + G_BM - 1) / G_BM * G_BM;
  p.np = (N + G_BN - 1) / G_BN * G_BN;
  p.ws_a = p.mp * p.kbp;
  p.ws_b = p.np * p.kbp;
  return true;
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

extern "C" mxq_status mxq_gemm(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                               int fmt, int64_t M, int64_t N, int64_t K, void* C, int out_dtype,
                               void* workspace, size_t workspace_bytes, void* stream) {
  Plan p;
  if (!make_plan(M, N, K, fmt, p)) return MXQ_ERR_ARG;
  if (!A || !sA || !B || !sB || !C || !workspace) return MXQ_ERR_ARG;
  if (out_dtype != MXQ_OUT_F32 && out_dtype != MXQ_OUT_BF16) return MXQ_ERR_ARG;
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return MXQ_ERR_ARG;
  if (N % (out_dtype == MXQ_OUT_F32 ? 4 : 8) != 0) return MXQ_ERR_ALIGN;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MXQ_ERR_ALIGN;
  if (workspace_bytes < static_cast<size_t>(p.ws_a + p.ws_b)) return MXQ_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  {
    const int64_t ta = p.mp * (p.kbp / 4), tb = p.np * (p.kbp / 4);
    const int ga = static_cast<int>(std::min<int64_t>((ta + 255) / 256, 4 * sm_count()));
    const int gb = static_cast<int>(std::min<int64_t>((tb + 255) / 256, 4 * sm_count()));
    sf_to_chunks<<<ga, 256, 0, st>>>(sA, M, p.kb, p.mp, p.kbp, ws);
    sf_to_chunks<<<gb, 256, 0, st>>>(sB, N, p.kb, p.np, p.kbp, ws + p.ws_a);
  }

  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_tiled();
  if (!encode) return MXQ_ERR_CUDA;
  CUtensorMap ta, tb;
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.kbytes), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.kbytes)};
    const cuuint32_t box[2] = {G_BKB, G_BM};
    if (encode(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(A), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MXQ_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.kbytes), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.kbytes)};
    const cuuint32_t box[2] = {G_BKB, G_BN};
    if (encode(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(B), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MXQ_ERR_CUDA;
  }

  GArgs a;
  a.M = static_cast<int32_t>(M);
  a.N = static_cast<int32_t>(N);
  a.n_mt = static_cast<int32_t>(p.mp / G_BM);
  a.n_nt = static_cast<int32_t>(p.np / G_BN);
  if (int64_t(a.n_mt) * a.n_nt >= (int64_t(1) << 31)) return MXQ_ERR_ARG;
  a.n_tiles = a.n_mt * a.n_nt;
  a.nk = static_cast<int32_t>((p.kbytes + G_BKB - 1) / G_BKB);
  a.kc_per_row = static_cast<int32_t>(p.kbp / 4);
  a.sfa = ws;
  a.sfb = ws + p.ws_a;
  a.C = C;
  a.out_bf16 = out_dtype == MXQ_OUT_BF16;
  a.fp4 = fmt == MXQ_E2M1;
  a.timeout_ns = wait_timeout_ns();

  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(mx_gemm_kernel),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM) != cudaSuccess)
    return MXQ_ERR_CUDA;
  const int grid = std::min<int>(a.n_tiles, sm_count());
  mx_gemm_kernel<<<grid, G_THREADS, G_SMEM, st>>>(ta, tb, a);
  return launch_status();
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
