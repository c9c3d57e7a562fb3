// Routed-expert FFN with E4M3 activations (the FP8-activation variant of the
// tensor-core grouped GEMM): both GEMM operands are E4M3 in shared memory and
// tcgen05.mma kind::f8f6f4 multiplies them, so the weight codes feed the
// tensor core without a decode step.
//
// Activations are quantised per row and group of 128 input features, the
// grouping of the weights' 128 x 128 scale blocks: for a group with largest
// magnitude a, codes = E4M3_rn_satfinite(v * fp32(448 / a)), scale
// s = fp32(a / 448) (a == 0: codes and scale 0).  x is quantised when it is
// gathered into expert order; hid (the SwiGLU output, in fp32) by the gate/up
// epilogue, whose 128 gate rows are exactly one group of hid features.
//
// The product of two block-scaled operands needs the scales of both at every
// 128-wide K block:  D[r, t] = sum_b Sw[r, b] Sx[t, b] P_b[r, t],  P_b the
// raw E4M3 x E4M3 sum over block b.  The tensor core accumulates P_b in tensor
// memory (fresh for each block); promoter warps read it, scale it in fp32 and
// add it to the running sum R, also in tensor memory:
//   TMEM columns   0..255  P (two weight blocks x 128 token columns)
//                256..511  R (the same two blocks)
// Each weight block has its own partial sums and barriers, so the tensor
// core computes one block's while the other's are promoted.
// Warp roles (one CTA per SM, tiles as in the fp16-operand GEMM):
//   warp 0      TMA: the step's two E4M3 code blocks (64-byte swizzled);
//   warp 1      TMA: the step's E4M3 token rows (64-byte swizzled), and per
//               tile the promotion factors Sw Sx into shared memory (a
//               weight block's scale is one number per K block, so the
//               factor depends on the token column only);
//   warp 2      one elected thread issues tcgen05.mma kind::f8f6f4
//               (M = 128, N, K = 32), both operands from shared memory;
//   warps 3-10  promote each K block's partial sums: R += Sw Sx P;
//   warps 11-18 epilogue: gate/up SwiGLU + E4M3 quantisation of hid; down
//               y as fp16 with one exponent per 32 columns.
// Every wait is bounded and gives up together with the other roles, as in
// the fp16-operand GEMM (MOE_DEV_WAIT_TIMEOUT).
#include <cuda.h>

#include <cstdlib>
#include <cstring>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {
constexpr int BT = 128;  // token rows per tile (MMA N, at most)
constexpr int BW = 128;  // weight rows per block (MMA M)
constexpr int BK = 64;   // K per step: 64 E4M3 (two MMAs of K = 32)
constexpr int NT = 6, NCD = 5;
constexpr int T_BYTES = BT * BK;      // 8 KB
constexpr int C_BYTES = 2 * BW * BK;  // 16 KB: two code blocks of 8 KB
constexpr int kMaxKb = 16;  // K <= 2048: 128-wide K blocks per row
// a tile's promotion factors Sw[blk, kb] Sx[token, kb], [blk][kb][token]
constexpr int SX_BYTES = 2 * kMaxKb * BT * 4;
constexpr int STG_WARP_BYTES = 4096;
constexpr int OFF_T = 0;
constexpr int OFF_C = OFF_T + NT * T_BYTES;
constexpr int OFF_SX = OFF_C + NCD * C_BYTES;
constexpr int OFF_STG = OFF_SX + 2 * SX_BYTES;
constexpr int kProWarps = 8, kEpiWarps = 8;
constexpr int SMEM_F8 = OFF_STG + kEpiWarps * STG_WARP_BYTES + 1024;
constexpr int W_CODES = 0, W_TOK = 1, W_MMA = 2, W_PRO0 = 3, W_EPI0 = W_PRO0 + kProWarps;
constexpr int kWarps = W_EPI0 + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_P = 0, COL_R = 2 * BT;
static_assert(SMEM_F8 <= 227 * 1024, "shared memory");

struct F8Args {
  const int32_t* expert_off;
  const int32_t* tile_off;  // token-tile prefix per expert, [E + 1]
  int E;
  int K;                // H for gate/up, I for down
  int rows_per_expert;  // I for gate/up, H for down
  const float* s0;      // gate (or down) weight scales
  const float* s1;      // up weight scales (gate/up only)
  const float* xs;      // activation scales [P][xs_ld] (token-major)
  int xs_ld;
  int n_wblocks;  // weight tiles per token tile
  int all_wait;   // 1: the previous kernel wrote the tile offsets (every warp waits)
  int32_t* slot_done;  // gate/up -> down completion counters per token tile
  int slot_need;
  int32_t* status;
  // gate/up: hid codes [P][I] and scales [P][hs_ld] (token-major)
  uint8_t* hid8;
  float* hs;
  int hs_ld;
  // down: y [P][H] fp16 with exponents [H / 32][yexp_rows] (y = y'' 2^s)
  uint16_t* y;
  int16_t* yexp;
  int yexp_rows;
  uint64_t wait_ns;
};

struct F8Shared {
  uint64_t c_full[NCD], c_empty[NCD];
  uint64_t t_full[NT], t_empty[NT];
  uint64_t sx_full[2], sx_empty[2];
  uint64_t p_full[2], p_empty[2];  // per weight block
  uint64_t acc_full, acc_empty;
  // gate/up epilogue's exchange of per-token maxima among the four warps of a
  // half, per chunk pair: written (amx_full) and read (amx_free)
  uint64_t amx_full[2][2], amx_free[2][2];
  uint32_t tmem_base;
  int abort_flag;
  uint64_t wait_ns;
  int tile_off[kMaxExperts + 1];
  int expert_off[kMaxExperts + 1];
  // gate/up epilogue: each warp's per-token largest |hid| over its 32
  // features, [half][chunk pair][lane quarter][token]
  uint32_t amax[2][2][4][32];
};

// Warp-uniform bounded wait on an mbarrier phase (see the fp16-operand GEMM):
// the warp gives up together once the budget is spent or another role gave
// up; the first to give up records MOE_DEV_WAIT_TIMEOUT and where.
__device__ __forceinline__ bool f8_wait(F8Shared& sh, uint64_t* bar, uint32_t parity,
                                        int32_t* status, int bar_id, int step) {
  constexpr unsigned kAll = 0xffffffffu;
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(kAll, done)) return true;
  const WaitBudget b = wait_budget(sh.wait_ns);
  for (uint32_t n = 1;; ++n) {
    if (__any_sync(kAll, done)) {
      for (int r = 0; !done && r < (1 << 16); ++r) done = mbar_try_wait(bar, parity);
      if (__all_sync(kAll, done)) return true;
      break;
    }
    if ((n & 31) == 0) {
      const bool give_up = *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0 || budget_spent(b);
      if (__any_sync(kAll, give_up)) break;
    }
    done = mbar_try_wait(bar, parity);
  }
  if ((threadIdx.x & 31) == 0 && !sh.abort_flag) {
    sh.abort_flag = 1;
    raise_status(status, MOE_DEV_WAIT_TIMEOUT);
    if (status && atomicCAS(status + 1, 0, 1 + (int)(threadIdx.x >> 5)) == 0) {
      status[2] = bar_id;
      status[3] = step;
      status[4] = (int)parity;
      status[5] = (int)blockIdx.x;
    }
  }
  __syncwarp();
  return false;
}

struct F8Tile {
  int e, r0, m0, rows, n, n0, slot;
};

__device__ __forceinline__ F8Tile f8_tile(const F8Shared& sh, const F8Args& a, int t, bool gateup) {
  F8Tile ti;
  const int slot = t / a.n_wblocks, wb = t % a.n_wblocks;
  int lo = 0, hi = a.E;  // largest e with tile_off[e] <= slot
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh.tile_off[mid] <= slot) lo = mid; else hi = mid;
  }
  ti.e = lo;
  ti.slot = slot;
  ti.r0 = sh.expert_off[lo];
  ti.m0 = (slot - sh.tile_off[lo]) * BT;
  ti.rows = min(BT, sh.expert_off[lo + 1] - ti.r0 - ti.m0);
  ti.n = (ti.rows + 15) & ~15;
  ti.n0 = wb * (gateup ? BW : 2 * BW);
  return ti;
}

// K-major operand tile of 64-byte rows, 64-byte swizzled (as TMA writes it):
// 8-row groups 512 bytes apart.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;            // leading byte offset (16 B), ignored here
  d |= (uint64_t)(512 >> 4) << 32;   // stride byte offset: 8 rows x 64 B
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)4 << 61;            // 64-byte swizzle
  return d;
}

// D (+)= A B^T, A [128 x 32] and B [N x 32] E4M3 from shared memory, fp32 D.
__device__ __forceinline__ void mma_f8_ss(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One float -> E4M3 code, round to nearest even, saturated to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}

}  // namespace

template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
k_expert_gemm_f8(const __grid_constant__ CUtensorMap cm0, const __grid_constant__ CUtensorMap cm1,
                 const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_y,
                 const F8Args args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ F8Shared sh;
  // As in the fp16-operand GEMM, only the warps that read the previous
  // kernel's output (the token rows and their scales) wait for it.
  if (args.all_wait) griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const F8Args& a = args;
  const int n_tiles = a.tile_off[a.E] * a.n_wblocks;
  const int tstride = (int)gridDim.x;
  if ((int)blockIdx.x >= n_tiles) return;  // uniform per CTA, before any barrier
  const int nK = a.K / BK;
  const int nKb = a.K / kScaleBlock;  // K blocks (two steps each)
  const int nRb = cdiv(a.rows_per_expert, kScaleBlock);

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t smem_base = smem_u32(smem);
  float* sx_buf = reinterpret_cast<float*>(smem + OFF_SX);  // [2][2][kMaxKb][BT]

  if (tid == 0) {
    for (int s = 0; s < NCD; ++s) {
      mbar_init(&sh.c_full[s], 1);
      mbar_init(&sh.c_empty[s], 1);
    }
    for (int s = 0; s < NT; ++s) {
      mbar_init(&sh.t_full[s], 1);
      mbar_init(&sh.t_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.sx_full[s], 1);
      mbar_init(&sh.sx_empty[s], kProWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.p_full[b], 1);
      mbar_init(&sh.p_empty[b], kProWarps / 2);
    }
    mbar_init(&sh.acc_full, kProWarps);
    mbar_init(&sh.acc_empty, kEpiWarps);
    for (int h = 0; h < 2; ++h)
      for (int i = 0; i < 2; ++i) {
        mbar_init(&sh.amx_full[h][i], 4);
        mbar_init(&sh.amx_free[h][i], 4);
      }
    sh.abort_flag = 0;
    sh.wait_ns = a.wait_ns;
    fence_mbar_init();
  }
  for (int i = tid; i <= a.E; i += kThreads) {
    sh.tile_off[i] = a.tile_off[i];
    sh.expert_off[i] = a.expert_off[i];
  }
  if (warp == 0) {
    tc::tmem_alloc(&sh.tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == W_CODES) {
    // ------------------------------------------------ E4M3 weight codes (TMA)
    int j = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += tstride) {
      const F8Tile ti = f8_tile(sh, a, t, GATEUP);
      const int row = ti.e * a.rows_per_expert + ti.n0;
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sc = j % NCD;
        if (j >= NCD && !f8_wait(sh, &sh.c_empty[sc], (uint32_t)(((j / NCD) - 1) & 1), a.status, 1, j)) {
          ok = false;
          break;
        }
        if (tc::elect_one()) {
          uint8_t* dst = smem + OFF_C + sc * C_BYTES;
          mbar_arrive_expect_tx(&sh.c_full[sc], C_BYTES);
          if (GATEUP) {
            tc::tma_load_2d(dst, &cm0, ks * BK, row, &sh.c_full[sc]);
            tc::tma_load_2d(dst + BW * BK, &cm1, ks * BK, row, &sh.c_full[sc]);
          } else {
            tc::tma_load_2d(dst, &cm0, ks * BK, row, &sh.c_full[sc]);
            tc::tma_load_2d(dst + BW * BK, &cm0, ks * BK, row + BW, &sh.c_full[sc]);
          }
        }
        __syncwarp();
      }
    }
    if (lane == 0)
      for (int i = max(0, j - NCD); i < j; ++i) mbar_wait(&sh.c_full[i % NCD], (uint32_t)((i / NCD) & 1));
    __syncwarp();
  } else if (warp == W_TOK) {
    // ------------------------------------------------ E4M3 token rows (TMA) + their scales
    if (GATEUP && !a.all_wait) griddep_wait();  // x codes and scales: the previous kernel's
    int j = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += tstride, ++tl) {
      const F8Tile ti = f8_tile(sh, a, t, GATEUP);
      if (!GATEUP) {
        // this token tile's hid codes and scales are stored by every gate/up
        // weight-block tile of the slot (bounded warp-uniform poll)
        const WaitBudget b = wait_budget(sh.wait_ns);
        bool done = false;
        for (uint32_t n = 0; !done; ++n) {
          done = __all_sync(0xffffffffu, tc::ld_acquire_gpu(a.slot_done + ti.slot) >= a.slot_need);
          if (!done && (n & 31) == 31) {
            const bool give_up =
                *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0 || budget_spent(b);
            if (__any_sync(0xffffffffu, give_up)) break;
          }
        }
        if (!done) {
          if (lane == 0 && !sh.abort_flag) {
            sh.abort_flag = 1;
            raise_status(a.status, MOE_DEV_WAIT_TIMEOUT);
            if (a.status && atomicCAS(a.status + 1, 0, 1 + W_TOK) == 0) {
              a.status[2] = 9;
              a.status[3] = ti.slot;
              a.status[4] = tc::ld_acquire_gpu(a.slot_done + ti.slot);
              a.status[5] = (int)blockIdx.x;
            }
          }
          __syncwarp();
          break;
        }
        tc::fence_proxy_async_global();
      }
      // the tile's promotion factors Sw[blk, kb] Sx[token, kb], laid out
      // [blk][kb][token] (0 past the tile's rows), once the promoters have
      // released the buffer; lane kb holds the two weight blocks' scales
      const int sb = tl & 1;
      if (tl >= 2 && !f8_wait(sh, &sh.sx_empty[sb], (uint32_t)(((tl >> 1) - 1) & 1), a.status, 12, tl))
        break;
      float* fs = sx_buf + sb * (2 * kMaxKb * BT);
      float sw[2];
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const float* sp = (GATEUP && blk) ? a.s1 : a.s0;
        const size_t srow = (size_t)ti.e * nRb + ti.n0 / kScaleBlock + (GATEUP ? 0 : blk);
        sw[blk] = lane < nKb ? __ldg(sp + srow * nKb + lane) : 0.f;
      }
      for (int r = lane; r < BT; r += 32) {
        const bool real = r < ti.rows;
        const float* src = a.xs + (size_t)(ti.r0 + ti.m0 + r) * a.xs_ld;
        for (int b = 0; b < nKb; b += 4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (real) v = __ldcg(reinterpret_cast<const float4*>(src + b));
          const float x4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float w0 = __shfl_sync(0xffffffffu, sw[0], b + i);
            const float w1 = __shfl_sync(0xffffffffu, sw[1], b + i);
            if (b + i < nKb) {
              fs[(0 * kMaxKb + b + i) * BT + r] = w0 * x4[i];
              fs[(1 * kMaxKb + b + i) * BT + r] = w1 * x4[i];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.sx_full[sb]);  // release: the scales are in place
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int st = j % NT;
        if (j >= NT && !f8_wait(sh, &sh.t_empty[st], (uint32_t)(((j / NT) - 1) & 1), a.status, 2, j)) {
          ok = false;
          break;
        }
        if (tc::elect_one()) {
          mbar_arrive_expect_tx(&sh.t_full[st], T_BYTES);
          tc::tma_load_2d(smem + OFF_T + st * T_BYTES, &tmap, ks * BK, ti.r0 + ti.m0, &sh.t_full[st]);
        }
        __syncwarp();
      }
    }
    if (lane == 0)
      for (int i = max(0, j - NT); i < j; ++i) mbar_wait(&sh.t_full[i % NT], (uint32_t)((i / NT) & 1));
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------ tcgen05.mma kind::f8f6f4
    // Per K block (two steps), per weight block b: once the promoters of b
    // have read its previous partial sums, 4 MMAs (2 steps x 2 halves of K)
    // into P_b, the first overwriting it, then a commit to p_full[b]; so the
    // tensor core works on one block while the other is promoted.  The
    // instruction descriptor has the same fields as for kind::f16: fp32 D,
    // A and B format code 0 (E4M3 here), both K-major.
    int j = 0, kbg = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += tstride) {
      const F8Tile ti = f8_tile(sh, a, t, GATEUP);
      const uint32_t idesc = tc::idesc_f16_f32(BW, ti.n);
      for (int kb = 0; kb < nKb && ok; ++kb, ++kbg, j += 2) {
        const int st0 = j % NT, sc0 = j % NCD, st1 = (j + 1) % NT, sc1 = (j + 1) % NCD;
        if (!f8_wait(sh, &sh.t_full[st0], (uint32_t)((j / NT) & 1), a.status, 6, j) ||
            !f8_wait(sh, &sh.c_full[sc0], (uint32_t)((j / NCD) & 1), a.status, 7, j) ||
            !f8_wait(sh, &sh.t_full[st1], (uint32_t)(((j + 1) / NT) & 1), a.status, 6, j + 1) ||
            !f8_wait(sh, &sh.c_full[sc1], (uint32_t)(((j + 1) / NCD) & 1), a.status, 7, j + 1)) {
          ok = false;
          break;
        }
        for (int blk = 0; blk < 2 && ok; ++blk) {
          if (kbg > 0 &&
              !f8_wait(sh, &sh.p_empty[blk], (uint32_t)((kbg - 1) & 1), a.status, 5, kbg)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          if (tc::elect_one()) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t b_addr = smem_base + OFF_T + (h ? st1 : st0) * T_BYTES;
              const uint32_t a_addr = smem_base + OFF_C + (h ? sc1 : sc0) * C_BYTES + blk * (BW * BK);
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                mma_f8_ss(tmem + COL_P + blk * BT, sw64_desc(a_addr + kk * 32),
                          sw64_desc(b_addr + kk * 32), idesc, (h | kk) ? 1u : 0u);
            }
            tc::commit(&sh.p_full[blk]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (tc::elect_one()) {
          // both blocks' MMAs have read the two steps' operands
          tc::commit(&sh.t_empty[st0]);
          tc::commit(&sh.c_empty[sc0]);
          tc::commit(&sh.t_empty[st1]);
          tc::commit(&sh.c_empty[sc1]);
        }
        __syncwarp();
      }
    }
    // drain: the newest commit completes once every MMA issued has
    if (lane == 0 && kbg > 0) mbar_wait(&sh.p_full[1], (uint32_t)((kbg - 1) & 1));
    __syncwarp();
  } else if (warp >= W_PRO0 && warp < W_PRO0 + kProWarps) {
    // ------------------------------------------------ promotion: R += Sw Sx P
    // Warp (blk, q): TMEM lanes 32 q .. 32 q + 31 of weight block blk (gate /
    // first 128 down rows, or up / the next 128); lane i holds the weight
    // scale of K block i of its row block, loaded a tile ahead.
    const int blk = (warp - W_PRO0) >> 2, q = warp & 3;
    const uint32_t t_p = tmem + ((uint32_t)(32 * q) << 16) + COL_P + (uint32_t)blk * BT;
    const uint32_t t_r = tmem + ((uint32_t)(32 * q) << 16) + COL_R + (uint32_t)blk * BT;
    int kbg = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += tstride, ++tl) {
      const F8Tile ti = f8_tile(sh, a, t, GATEUP);
      const int nchunks = (ti.n + 31) >> 5;
      const int sb = tl & 1;
      const float* fs = sx_buf + (sb * 2 + blk) * (kMaxKb * BT);
      if (!f8_wait(sh, &sh.sx_full[sb], (uint32_t)((tl >> 1) & 1), a.status, 13, tl)) break;
      for (int kb = 0; kb < nKb; ++kb, ++kbg) {
        if (!f8_wait(sh, &sh.p_full[blk], (uint32_t)(kbg & 1), a.status, 3, kbg) ||
            (kb == 0 && tl > 0 &&
             !f8_wait(sh, &sh.acc_empty, (uint32_t)((tl - 1) & 1), a.status, 4, tl))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t p[32], r[32];
          tc::ld_32x32b_x32(t_p + 32 * c, p);
          if (kb > 0) tc::ld_32x32b_x32(t_r + 32 * c, r);
          tc::wait_ld();
          if (c == nchunks - 1) {
            // all of this block's partial sums are read: the next block's
            // MMAs may overwrite them
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_empty[blk]);
          }
          // token 32 c + v's factor of block kb (16-byte broadcast reads)
          const float4* fc = reinterpret_cast<const float4*>(fs + kb * BT + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float4 s4 = fc[v4];
            const float f[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int v = 4 * v4 + i;
              const float pv = __uint_as_float(p[v]);
              r[v] = __float_as_uint(kb > 0 ? fmaf(pv, f[i], __uint_as_float(r[v])) : pv * f[i]);
            }
          }
          tc::st_32x32b_x32(t_r + 32 * c, r);
        }
        tc::wait_st();
      }
      if (!ok) break;
      // the tile's sums are complete; its scale buffer is free
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.acc_full);
        mbar_arrive(&sh.sx_empty[sb]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 11-18)
    // Lane quarter q of both sums: weight rows 32 q + lane; columns are the
    // tile's tokens.  gate/up: half eh takes the 32-token chunks eh, eh + 2;
    // down: half eh takes weight block eh.
    const int q = warp & 3, eh = (warp - W_EPI0) >> 2;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16) + COL_R;
    uint8_t* stg = smem + OFF_STG + (warp - W_EPI0) * STG_WARP_BYTES;
    if (GATEUP && !a.all_wait) griddep_wait();
    bool bad = false;
    int tl = 0;
    for (int t = blockIdx.x; t < n_tiles; t += tstride, ++tl) {
      const F8Tile ti = f8_tile(sh, a, t, GATEUP);
      tc::bulk_wait_read_all();
      __syncwarp();
      if (!f8_wait(sh, &sh.acc_full, (uint32_t)(tl & 1), a.status, 8, tl)) break;
      tc::fence_after_sync();
      const int nchunks = (ti.n + 31) >> 5;
      if (GATEUP) {
        // this warp's chunks: eh, eh + 2 (< nchunks); the last releases the sums
        const int last = eh < nchunks ? eh + 2 * ((nchunks - 1 - eh) >> 1) : -1;
        if (last < 0) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.acc_empty);
        }
        bool ok = true;
        for (int c = eh; c < 4 && ok; c += 2) {
          // every warp of the half takes part in each chunk pair's exchange,
          // real or not
          const bool real = c < nchunks;
          const int pi = c >> 1;
          float h[32];
          if (real) {
            uint32_t g[32], u[32];
            tc::ld_32x32b_x32(t_lane + 32 * c, g);
            tc::ld_32x32b_x32(t_lane + BT + 32 * c, u);
            tc::wait_ld();
            if (c == last) {
              tc::fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh.acc_empty);
            }
#pragma unroll
            for (int v = 0; v < 32; ++v) {
              const float gv = __uint_as_float(g[v]), uv = __uint_as_float(u[v]);
              const float sig = __fdividef(1.f, 1.f + __expf(-fminf(fmaxf(gv, -80.f), 80.f)));
              h[v] = gv * sig * uv;
            }
          } else {
#pragma unroll
            for (int v = 0; v < 32; ++v) h[v] = 0.f;
          }
          // token v's largest |hid| over this warp's 32 features -> lane v
          uint32_t mine = 0;
#pragma unroll
          for (int v = 0; v < 32; ++v) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(h[v]) & 0x7fffffffu);
            if (lane == v) mine = m;
          }
          // the slots' previous values have been read by all four warps
          if (tl > 0 && !f8_wait(sh, &sh.amx_free[eh][pi], (uint32_t)((tl - 1) & 1), a.status, 14, tl)) {
            ok = false;
            break;
          }
          sh.amax[eh][pi][q][lane] = mine;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.amx_full[eh][pi]);
          if (!f8_wait(sh, &sh.amx_full[eh][pi], (uint32_t)(tl & 1), a.status, 15, tl)) {
            ok = false;
            break;
          }
          // token 32 c + lane: its group (the tile's 128 features) scale
          uint32_t am = 0;
#pragma unroll
          for (int w = 0; w < 4; ++w) am = max(am, sh.amax[eh][pi][w][lane]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.amx_free[eh][pi]);
          if (!real) continue;
          const int nv = ti.rows - 32 * c;
          if (lane < nv && am >= 0x7f800000u) bad = true;
          const float amf = __uint_as_float(am);
          const bool zero = am == 0u;
          const float inv = zero ? 0.f : __fdiv_rn(448.f, amf);
          const size_t row = (size_t)(ti.r0 + ti.m0 + 32 * c + lane);
          if (q == 0 && lane < nv)
            a.hs[row * a.hs_ld + ti.n0 / kScaleBlock] = zero ? 0.f : __fdiv_rn(amf, 448.f);
          // codes, staged token-major (row v = token, byte lane = feature)
#pragma unroll
          for (int v = 0; v < 32; ++v) {
            const float iv = __shfl_sync(0xffffffffu, inv, v);
            stg[v * 32 + lane] = (uint8_t)f32_to_e4m3(h[v] * iv);
          }
          __syncwarp();
          if (lane < nv) {
            const uint4* src = reinterpret_cast<const uint4*>(stg + lane * 32);
            uint4* dst = reinterpret_cast<uint4*>(a.hid8 + row * a.rows_per_expert + ti.n0 + 32 * q);
            dst[0] = src[0];
            dst[1] = src[1];
          }
          __syncwarp();
        }
        if (!ok) break;
        // publish: this warp's hid codes and scales of the tile are stored
        __threadfence();
        __syncwarp();
        if (lane == 0) tc::red_release_gpu_add(a.slot_done + ti.slot, 1);
      } else {
        // block eh, rows col0 .. col0 + 31 of y's columns (this warp's
        // lanes) x tokens 32 c .. (the chunk's columns): staged in fp32
        // token-major, read back per token, fp16 y'' with y = y'' 2^s per
        // token and 32 columns (as in the fp16-operand GEMM)
        const int col0 = ti.n0 + eh * BW + 32 * q;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tc::ld_32x32b_x32(t_lane + eh * BT + 32 * c, v);
          const int nv = ti.rows - 32 * c;
          const size_t row = (size_t)(ti.r0 + ti.m0 + 32 * c + lane);
          tc::wait_ld();
          if (c == nchunks - 1) {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty);
          }
          tc::bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            *reinterpret_cast<uint32_t*>(stg + i * 128 + (((lane >> 2) ^ (i & 7)) << 4) +
                                         (lane & 3) * 4) = v[i];
          __syncwarp();
          float f[32];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float4 g = *reinterpret_cast<const float4*>(stg + lane * 128 + ((jj ^ (lane & 7)) << 4));
            f[4 * jj] = g.x;
            f[4 * jj + 1] = g.y;
            f[4 * jj + 2] = g.z;
            f[4 * jj + 3] = g.w;
          }
          __syncwarp();
          uint32_t m = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) m = max(m, __float_as_uint(f[i]) & 0x7fffffffu);
          if (lane < nv && m >= 0x7f800000u) bad = true;
          const int E = min(exp_of_bits(m), 127);
          const float sc = pow2f(kGroupTop - E);
          if (lane < nv) a.yexp[(size_t)(col0 >> 5) * a.yexp_rows + row] = (int16_t)(E - kGroupTop);
          uint4* dst = reinterpret_cast<uint4*>(a.y + row * a.rows_per_expert + col0);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint4 w4 = make_uint4(pack_f16x2(f[8 * jj] * sc, f[8 * jj + 1] * sc),
                                        pack_f16x2(f[8 * jj + 2] * sc, f[8 * jj + 3] * sc),
                                        pack_f16x2(f[8 * jj + 4] * sc, f[8 * jj + 5] * sc),
                                        pack_f16x2(f[8 * jj + 6] * sc, f[8 * jj + 7] * sc));
            if (nv >= 32)
              *reinterpret_cast<uint4*>(stg + lane * 64 + ((jj ^ ((lane >> 1) & 3)) << 4)) = w4;
            else if (lane < nv)
              dst[jj] = w4;
          }
          if (nv >= 32) {
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              tc::tma_store_2d(&tmap_y, col0, ti.r0 + ti.m0 + 32 * c, stg);
              tc::bulk_commit();
            }
            __syncwarp();
          }
        }
      }
    }
    if (bad && lane == 0) raise_status(a.status, MOE_DEV_NONFINITE);
    tc::bulk_wait_all();
    __syncwarp();
  }

  // ---- all roles done: free TMEM
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// E4M3 activation rows in expert order (the layer call's token -> row map):
// one warp per token quantises x[t] per group of 128 columns and writes the
// codes to each of its rows tok_slot_row[t k + j] >= 0 of x8 [P][K], the
// group scales to xs [P][xs_ld].  Lane l's piece i holds columns
// 8 (l + 32 i) .. + 7, so a group is one piece of 16 consecutive lanes.
constexpr int kF8GatherMaxPieces = 16;  // K <= 4096
__global__ void __launch_bounds__(256)
k_gather_tokens_f8(const uint16_t* __restrict__ x, int T, int K,
                   const int32_t* __restrict__ tok_slot_row, int k, uint8_t* __restrict__ x8,
                   float* __restrict__ xs, int xs_ld, int32_t* __restrict__ status) {
  griddep_wait();
  griddep_trigger();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;  // warp-uniform
  const int np = K / 256;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * K);
  uint2 codes[kF8GatherMaxPieces];
  float scale[kF8GatherMaxPieces];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kF8GatherMaxPieces; ++i) {
    if (i < np) {
      const uint4 v = __ldg(src + lane + 32 * i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t m = 0;  // largest bf16 magnitude bits of the piece, then of the group
#pragma unroll
      for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (m >= 0x7F80u) bad = true;
      const float amax = __uint_as_float(m << 16);
      const float inv = m ? __fdiv_rn(448.f, amax) : 0.f;
      scale[i] = m ? __fdiv_rn(amax, 448.f) : 0.f;
      uint32_t c[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = f32_to_e4m3(bf16_lo(w[j]) * inv), hi = f32_to_e4m3(bf16_hi(w[j]) * inv);
        c[j >> 1] |= (lo | (hi << 8)) << (16 * (j & 1));
      }
      codes[i] = make_uint2(c[0], c[1]);
    }
  }
  if (bad && lane == 0) raise_status(status, MOE_DEV_NONFINITE);
  const int my_row = lane < k ? tok_slot_row[(size_t)t * k + lane] : -1;
  for (int jj = 0; jj < k; ++jj) {
    const int row = __shfl_sync(0xffffffffu, my_row, jj);
    if (row < 0) continue;  // warp-uniform
    uint2* dst = reinterpret_cast<uint2*>(x8 + (size_t)row * K);
#pragma unroll
    for (int i = 0; i < kF8GatherMaxPieces; ++i) {
      if (i < np) {
        dst[lane + 32 * i] = codes[i];
        if ((lane & 15) == 0) xs[(size_t)row * xs_ld + 2 * i + (lane >> 4)] = scale[i];
      }
    }
  }
}

namespace {
// Code or E4M3 activation matrix [rows, K]: box 64 bytes of K x 128 rows,
// 64-byte swizzled.
cudaError_t f8_map(CUtensorMap* map, const uint8_t* base, long long rows, int K) {
  return make_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, K, BK, 128, 64);
}
}  // namespace

int act8_scale_ld(int K) { return ((K / kScaleBlock) + 3) & ~3; }

cudaError_t launch_expert_gemm_f8(const uint16_t* x, int T, const int32_t* expert_off,
                                  const int32_t* tok_slot_row, int k, int E, int P,
                                  const moe_fp8_ffn& w, int H, int I, const int32_t* tile_off,
                                  int32_t* slot_done, uint8_t* x8, float* xs, uint8_t* hid8,
                                  float* hs, uint16_t* y, int16_t* yexp, int yexp_rows,
                                  int32_t* status, cudaStream_t s, bool pdl) {
  static_assert(BT == kGemmTokenTile, "token tile of the permutation's tile prefix");
  if (H > kF8GatherMaxPieces * 256 || H / kScaleBlock > kMaxKb || I / kScaleBlock > kMaxKb ||
      H % 256 || I % kScaleBlock || !slot_done || !yexp)
    return cudaErrorInvalidValue;
  cudaError_t err;
  if ((err = ensure_smem((const void*)k_expert_gemm_f8<true>, SMEM_F8)) != cudaSuccess) return err;
  if ((err = ensure_smem((const void*)k_expert_gemm_f8<false>, SMEM_F8)) != cudaSuccess) return err;
  CUtensorMap gmap, umap, dmap, xmap, hmap, ymap;
  if ((err = f8_map(&gmap, w.gate.codes, (long long)E * I, H)) != cudaSuccess) return err;
  if ((err = f8_map(&umap, w.up.codes, (long long)E * I, H)) != cudaSuccess) return err;
  if ((err = f8_map(&dmap, w.down.codes, (long long)E * H, I)) != cudaSuccess) return err;
  if ((err = f8_map(&xmap, x8, P, H)) != cudaSuccess) return err;
  if ((err = f8_map(&hmap, hid8, P, I)) != cudaSuccess) return err;
  if ((err = make_tensor_map_2d(&ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, y, P, H, 32, 32, 64)) !=
      cudaSuccess)
    return err;
  err = launch_k(k_gather_tokens_f8, dim3(cdiv(T, 8)), dim3(256), 0, s, pdl, x, T, H, tok_slot_row,
                 k, x8, xs, act8_scale_ld(H), status);
  if (err != cudaSuccess) return err;
  uint64_t wait_ns = 0;
  if (const char* lim = getenv("MOE_FP8_WAIT_LIMIT_US")) {
    const long long us = atoll(lim);
    if (us > 0) wait_ns = (uint64_t)us * 1000ull;
  }
  const int max_ttiles = cdiv(P, BT) + min(E, P);
  const int nsm = num_sms();
  F8Args g{};
  g.expert_off = expert_off;
  g.tile_off = tile_off;
  g.E = E;
  g.K = H;
  g.rows_per_expert = I;
  g.s0 = w.gate.scales;
  g.s1 = w.up.scales;
  g.xs = xs;
  g.xs_ld = act8_scale_ld(H);
  g.n_wblocks = I / BW;
  g.slot_done = slot_done;
  g.status = status;
  g.hid8 = hid8;
  g.hs = hs;
  g.hs_ld = act8_scale_ld(I);
  g.wait_ns = wait_ns;
  err = launch_k(k_expert_gemm_f8<true>, dim3(min(nsm, max_ttiles * g.n_wblocks)), dim3(kThreads),
                 (size_t)SMEM_F8, s, pdl, gmap, umap, xmap, ymap, g);
  if (err != cudaSuccess) return err;
  F8Args d{};
  d.expert_off = expert_off;
  d.tile_off = tile_off;
  d.E = E;
  d.K = I;
  d.rows_per_expert = H;
  d.s0 = w.down.scales;
  d.xs = hs;
  d.xs_ld = act8_scale_ld(I);
  d.n_wblocks = H / (2 * BW);
  d.slot_done = slot_done;
  d.slot_need = (I / BW) * kEpiWarps;
  d.status = status;
  d.y = y;
  d.yexp = yexp;
  d.yexp_rows = yexp_rows;
  d.wait_ns = wait_ns;
  return launch_k(k_expert_gemm_f8<false>, dim3(min(nsm, max_ttiles * d.n_wblocks)),
                  dim3(kThreads), (size_t)SMEM_F8, s, pdl, dmap, dmap, hmap, ymap, d);
}

}  // namespace moe
