// Routed-expert FFN for many tokens per expert (prefill): a grouped GEMM on
// the 5th-generation tensor cores (colizig README, "Features": block-FP8
// weights; "MoE per-expert evaluation").
//
// One CTA computes one 128 x 256 output tile of one expert:
//   gate/up: rows = 128 permuted token rows of the expert, columns = 128 gate
//            features and the same 128 up features (one 128-row scale block
//            each), K = H; the epilogue forms hid = silu(g) * u in fp16.
//   down:    rows = 128 permuted rows, columns = 256 output features, K = I;
//            the epilogue writes y in fp32.
// Operands (fp16, K-major, 128-byte swizzle) live in shared memory, the fp32
// accumulator in TMEM (256 columns).  Per 64-wide K step:
//   - cp.async brings the step's activation rows (gathered by token for
//     gate/up, contiguous for down; rows past the expert's segment are
//     zero-filled) and the E4M3 code tile (256 rows x 64 bytes) into a 4-deep
//     ring, two steps ahead;
//   - all 8 warps decode the codes to fp16 and apply the block scale
//     (fp16(dec * fp16(scale))), writing the swizzled B tile (double buffer);
//   - thread 0 issues four tcgen05.mma (M=128, N=256, K=16) and commits to an
//     mbarrier; the MMA of step k runs while the warps decode step k+1.
// Precision: the same fp16 operands and fp32 accumulation as the GEMV path's
// down projection; x16 (fp16 x) comes from the router.
#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {
constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kThreadsTC = 256;
constexpr int NA = 4;  // activation / code ring depth
constexpr int DIST = 2;  // prefetch distance (steps ahead), <= NA - 2
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B8_BYTES = BN * BK;      // 16 KB
constexpr int B16_BYTES = BN * BK * 2; // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B8 = OFF_A + NA * A_BYTES;
constexpr int OFF_B16 = OFF_B8 + NA * B8_BYTES;
constexpr int SMEM_TC = OFF_B16 + 2 * B16_BYTES + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 256;
}  // namespace

template <bool GATEUP>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_expert_gemm_tc(const uint16_t* __restrict__ asrc, int K, int rows_per_expert,
                 const int32_t* __restrict__ expert_off, const int32_t* __restrict__ row_token,
                 const int32_t* __restrict__ tile_off, int E,
                 const uint8_t* __restrict__ w0, const float* __restrict__ s0,
                 const uint8_t* __restrict__ w1, const float* __restrict__ s1,
                 void* __restrict__ out, int out_ld, int32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t mma_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int row_src[BM];  // gate/up: token of each tile row; down: hid row (-1: none)
  __shared__ int abort_sh;
  griddep_wait();
  griddep_trigger();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- which tile
  const int slot = blockIdx.y;
  const int total = tile_off[E];
  if (slot >= total) return;
  int lo = 0, hi = E;  // largest e with tile_off[e] <= slot
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_off[mid] <= slot) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int r0 = expert_off[e];
  const int cnt = expert_off[e + 1] - r0;
  const int m0 = (slot - tile_off[e]) * BM;
  const int mrows = min(BM, cnt - m0);
  const int n0 = blockIdx.x * (GATEUP ? BN / 2 : BN);  // first feature (gate/up) or h
  const int nKb = cdiv(K, kScaleBlock);
  const int nRb = cdiv(rows_per_expert, kScaleBlock);

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t smem_base = smem_u32(smem);

  if (tid < BM) {
    const int m = tid;
    row_src[m] = m < mrows ? (GATEUP ? row_token[r0 + m0 + m] : r0 + m0 + m) : -1;
  }
  if (tid == 0) {
    mbar_init(&mma_bar[0], 1);
    mbar_init(&mma_bar[1], 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  // ---- B row sources: row r of the 256-row code tile
  auto wrow = [&](int r) -> const uint8_t* {
    if (GATEUP) {
      const uint8_t* base = r < 128 ? w0 : w1;
      return base + ((size_t)e * rows_per_expert + n0 + (r & 127)) * K;
    }
    return w0 + ((size_t)e * rows_per_expert + n0 + r) * K;
  };

  auto load_step = [&](int step) {
    const int k0 = step * BK;
    const int sa = step % NA;
    uint8_t* A = smem + OFF_A + sa * A_BYTES;
    uint8_t* B8 = smem + OFF_B8 + sa * B8_BYTES;
#pragma unroll
    for (int u = 0; u < (BM * 8) / kThreadsTC; ++u) {  // 4 x 16 B of activations
      const int q = tid + kThreadsTC * u;
      const int m = q >> 3, j = q & 7;
      const int src = row_src[m];
      const uint16_t* g = asrc + (size_t)(src < 0 ? 0 : src) * K + k0 + 8 * j;
      tc::cp_async16_zfill(A + tc::sw128_off(m, j), g, src >= 0);
    }
#pragma unroll
    for (int u = 0; u < (BN * 4) / kThreadsTC; ++u) {  // 4 x 16 B of codes
      const int q = tid + kThreadsTC * u;
      const int r = q >> 2, j = q & 3;
      cp_async16(B8 + r * 64 + 16 * j, wrow(r) + k0 + 16 * j);
    }
  };

  const int nK = K / BK;
  const uint32_t idesc = tc::idesc_f16_f32(BM, BN);
#pragma unroll
  for (int p = 0; p < DIST; ++p) {
    if (p < nK) load_step(p);
    cp_async_commit();
  }

  bool ok = true;
  int issued = 0;  // MMA steps issued (same count in every thread)
  for (int ks = 0; ks < nK; ++ks) {
    cp_async_wait<DIST - 1>();  // this thread's copies of step ks have landed
    if (tid == 0 && ks >= 2) {  // MMA(ks-2) done: its A stage and B16 buffer are free
      if (!mbar_wait(&mma_bar[ks & 1], (uint32_t)(((ks - 2) >> 1) & 1))) {
        abort_sh = 1;
        raise_status(status, MOE_DEV_WAIT_TIMEOUT);
      }
    }
    __syncthreads();  // all copies of step ks visible; verdict of thread 0 visible
    if (abort_sh) {
      ok = false;
      break;
    }
    if (ks + DIST < nK) load_step(ks + DIST);
    cp_async_commit();

    // decode the code tile of step ks into the fp16 B tile
    {
      const int k0 = ks * BK;
      const uint8_t* B8 = smem + OFF_B8 + (ks % NA) * B8_BYTES;
      uint8_t* B16 = smem + OFF_B16 + (ks & 1) * B16_BYTES;
      const int kb = k0 / kScaleBlock;
      float sc[2];
      if (GATEUP) {
        const size_t srow = (size_t)e * nRb + n0 / kScaleBlock;
        sc[0] = s0[srow * nKb + kb];
        sc[1] = s1[srow * nKb + kb];
      } else {
        const size_t srow = (size_t)e * nRb + n0 / kScaleBlock;
        sc[0] = s0[srow * nKb + kb];
        sc[1] = s0[(srow + 1) * nKb + kb];
      }
      const uint32_t s2[2] = {(uint32_t)f32_to_f16_bits(sc[0]) * 0x10001u,
                              (uint32_t)f32_to_f16_bits(sc[1]) * 0x10001u};
#pragma unroll
      for (int u = 0; u < (BN * 8) / kThreadsTC; ++u) {  // 8 items of 8 codes
        const int q = tid + kThreadsTC * u;
        const int r = q >> 3, j = q & 7;
        const uint2 c8 = *reinterpret_cast<const uint2*>(B8 + r * 64 + 8 * j);
        const uint32_t sv = s2[r >> 7];
        uint32_t h[4];
        h[0] = e4m3x2_to_f16x2(c8.x & 0xFFFFu);
        h[1] = e4m3x2_to_f16x2(c8.x >> 16);
        h[2] = e4m3x2_to_f16x2(c8.y & 0xFFFFu);
        h[3] = e4m3x2_to_f16x2(c8.y >> 16);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h[v]) : "r"(h[v]), "r"(sv));
        *reinterpret_cast<uint4*>(B16 + tc::sw128_off(r, j)) = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
    tc::fence_proxy_async();  // decoded B tile and copied A tile -> tensor-core reads
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t a_addr = smem_base + OFF_A + (ks % NA) * A_BYTES;
      const uint32_t b_addr = smem_base + OFF_B16 + (ks & 1) * B16_BYTES;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        tc::mma_f16(tmem, tc::sw128_desc(a_addr + kk * 32), tc::sw128_desc(b_addr + kk * 32),
                    idesc, (ks > 0 || kk > 0) ? 1u : 0u);
      tc::commit(&mma_bar[ks & 1]);
    }
    ++issued;
  }
  cp_async_wait<0>();  // no copy may still land in shared memory after this point

  // ---- wait (bounded) for the newest MMA issued: commits are cumulative
  if (tid == 0 && issued > 0) {
    const int last = issued - 1;
    if (!mbar_wait(&mma_bar[last & 1], (uint32_t)((last >> 1) & 1))) {
      abort_sh = 1;
      raise_status(status, MOE_DEV_WAIT_TIMEOUT);
    }
  }
  __syncthreads();
  tc::fence_after_sync();
  if (ok && !abort_sh) {
    const int quad = warp & 3, half = warp >> 2;
    const int m = quad * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    if (GATEUP) {
      uint16_t* hid = reinterpret_cast<uint16_t*>(out);
      bool overflow = false;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col = half * 64 + c2 * 32;
        uint32_t gr[32], ur[32];
        tc::ld_32x32b_x32(tl + col, gr);
        tc::ld_32x32b_x32(tl + 128 + col, ur);
        tc::wait_ld();
        if (m < mrows) {
          uint32_t pk[16];
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            const float g0 = __uint_as_float(gr[2 * v]), g1 = __uint_as_float(gr[2 * v + 1]);
            const float u0 = __uint_as_float(ur[2 * v]), u1 = __uint_as_float(ur[2 * v + 1]);
            const float h0 = g0 / (1.f + expf(-g0)) * u0;
            const float h1 = g1 / (1.f + expf(-g1)) * u1;
            overflow |= !(fabsf(h0) <= kF16Max) || !(fabsf(h1) <= kF16Max);
            pk[v] = (uint32_t)f32_to_f16_bits(h0) | ((uint32_t)f32_to_f16_bits(h1) << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(hid + (size_t)(r0 + m0 + m) * out_ld + n0 + col);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (overflow) raise_status(status, MOE_DEV_FP16_RANGE);
    } else {
      float* y = reinterpret_cast<float*>(out);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int col = half * 128 + c4 * 32;
        uint32_t v[32];
        tc::ld_32x32b_x32(tl + col, v);
        tc::wait_ld();
        if (m < mrows) {
          float4* dst = reinterpret_cast<float4*>(y + (size_t)(r0 + m0 + m) * out_ld + n0 + col);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Per-expert tile prefix: tile_off[e] = sum_{e' < e} ceil(cnt_e' / 128),
// tile_off[E] = total.  One CTA, E <= 1024.
__global__ void __launch_bounds__(1024)
k_tile_offsets(const int32_t* __restrict__ expert_off, int E, int32_t* __restrict__ tile_off) {
  __shared__ int32_t wsum[32];
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid < E ? cdiv(expert_off[tid + 1] - expert_off[tid], BM) : 0;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += v;
    }
    wsum[lane] = s;
  }
  __syncthreads();
  const int before = warp ? wsum[warp - 1] : 0;
  if (tid < E) tile_off[tid] = before + incl - c;
  if (tid == E - 1) tile_off[E] = before + incl;
}

bool expert_gemm_tc_ok(int H, int I) {
  return H % 256 == 0 && I % 128 == 0 && H >= 256 && I >= 128;
}

cudaError_t launch_expert_gemm_tc(const uint16_t* x16, const int32_t* expert_off,
                                  const int32_t* row_token, int E, int P, const moe_fp8_ffn& w,
                                  int H, int I, int32_t* tile_off, uint16_t* hid, float* y,
                                  int32_t* status, cudaStream_t s, bool pdl) {
  cudaError_t err;
  if ((err = ensure_smem((const void*)k_expert_gemm_tc<true>, SMEM_TC)) != cudaSuccess) return err;
  if ((err = ensure_smem((const void*)k_expert_gemm_tc<false>, SMEM_TC)) != cudaSuccess) return err;
  err = launch_k(k_tile_offsets, dim3(1), dim3(1024), 0, s, pdl, expert_off, E, tile_off);
  if (err != cudaSuccess) return err;
  const int max_tiles = cdiv(P, BM) + min(E, P);  // each expert adds at most one partial tile
  const dim3 blk(kThreadsTC);
  err = launch_k(k_expert_gemm_tc<true>, dim3(I / (BN / 2), max_tiles), blk, (size_t)SMEM_TC, s,
                 pdl, x16, H, I, expert_off, row_token, (const int32_t*)tile_off, E, w.gate.codes,
                 w.gate.scales, w.up.codes, w.up.scales, (void*)hid, I, status);
  if (err != cudaSuccess) return err;
  return launch_k(k_expert_gemm_tc<false>, dim3(H / BN, max_tiles), blk, (size_t)SMEM_TC, s, pdl,
                  (const uint16_t*)hid, I, H, expert_off, row_token, (const int32_t*)tile_off, E,
                  w.down.codes, w.down.scales, (const uint8_t*)nullptr, (const float*)nullptr,
                  (void*)y, H, status);
}

}  // namespace moe
