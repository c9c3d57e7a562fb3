// Routed-expert FFN for many tokens per expert (prefill): a grouped GEMM on
// the 5th-generation tensor cores (colizig README, "Features": block-FP8
// weights; "MoE per-expert evaluation").
//
// Output tiles are 128 rows x 256 columns of one expert:
//   gate/up: rows = 128 permuted token rows of the expert, columns = 128 gate
//            features and the same 128 up features (one 128-row scale block
//            each), K = H; the epilogue writes hid = silu(g) * u in fp16.
//   down:    rows = 128 permuted rows, columns = 256 output features, K = I;
//            the epilogue writes y in fp32.
// Operands are fp16, K-major, 128-byte swizzled in shared memory; the fp32
// accumulator lives in TMEM.  Persistent CTAs (one per SM) walk the tiles with
// warp-specialised roles that hand work to each other through mbarriers:
//   warp 0      TMA: the E4M3 code tile of each 64-wide K step (2-D tensor
//               maps over the stacked code matrices) into a 4-deep ring;
//   warps 1-2   gather the step's activation rows with cp.async (rows past the
//               expert's segment are zero-filled) into a 4-deep ring; a step is
//               published once its copies landed, after a proxy fence;
//   warps 3-10  decode codes to fp16 times the block scale
//               (fp16(dec * fp16(scale))) into a double-buffered B tile;
//   warp 11     one thread issues tcgen05.mma (M=128, N=256, K=16) into one of
//               two TMEM accumulators (512 columns) and commits to mbarriers;
//   warps 12-15 epilogue: tcgen05.ld from the finished accumulator while the
//               next tile accumulates in the other one.
// Every wait is bounded (about 2 s) and also gives up as soon as another
// role has given up, recording MOE_DEV_WAIT_TIMEOUT; the CTA then drains its
// copies and MMAs and frees its TMEM before it exits.
#include <cuda.h>

#include <mutex>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {
constexpr int BM = 128, BN = 256, BK = 64;
constexpr int NA = 4, NB = 4, NC = 2;  // ring depths: activations, codes, fp16 B tiles
// Steps an activation loader publishes behind the one it issues (<= NA - 2,
// so it never waits for a slot whose step it has not published yet).
constexpr int kALag = NA - 2 > 0 ? NA - 2 : 1;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B8_BYTES = BN * BK;       // 16 KB
constexpr int B16_BYTES = BN * BK * 2;  // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B8 = OFF_A + NA * A_BYTES;
constexpr int OFF_B16 = OFF_B8 + NB * B8_BYTES;
// down epilogue: per epilogue warp one 32-row x 32-column fp32 staging tile
// (4 KB, 128-byte swizzled) that a TMA store writes out
constexpr int EPI_BYTES = 4 * 4096;
constexpr int OFF_EPI = OFF_B16 + NC * B16_BYTES;
constexpr int SMEM_WS = OFF_EPI + EPI_BYTES + 1024;  // + alignment slack
constexpr int kLoadWarps = 2, kDecWarps = 8;
// warp roles: TMA, activation loaders, decoders, MMA issue, 4 epilogue warps
constexpr int W_TMA = 0, W_LOAD0 = 1, W_DEC0 = W_LOAD0 + kLoadWarps,
              W_MMA = W_DEC0 + kDecWarps;
constexpr int kWarps = W_MMA + 1 + 4;
constexpr int kThreadsWS = kWarps * 32;
constexpr int kLoadThreads = kLoadWarps * 32, kDecThreads = kDecWarps * 32;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column accumulators

struct GemmArgs {
  const uint16_t* asrc;  // gate/up: x16 [T, K]; down: hid [P, K]
  int K;                 // H for gate/up, I for down
  int rows_per_expert;   // I for gate/up, H for down
  const int32_t* expert_off;
  const int32_t* row_token;
  const int32_t* tile_off;  // m-tile prefix per expert, [E + 1]
  int E;
  const float* s0;  // gate (or down) scales
  const float* s1;  // up scales (gate/up only)
  void* out;        // hid fp16 [P, I] or y fp32 [P, H]
  int out_ld;
  int n_ntiles;  // column tiles per expert
  int32_t* status;
};

struct WsShared {
  uint64_t b8_full[NB], b8_empty[NB];
  uint64_t a_full[NA], a_empty[NA];
  uint64_t b16_full[NC], b16_empty[NC];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
  // Steps each role has completed, for the timeout record: [warp] for the
  // TMA warp (codes issued), the loader warps (activation steps published)
  // and the decoder warps (steps decoded); [kWarps] steps issued to the
  // tensor core, [kWarps + 1] tiles started by it, [kWarps + 2] tiles
  // finished by the epilogue.
  int prog[kWarps + 3];
  // copies of the per-expert tile prefix and row offsets (E + 1 entries),
  // so that finding a tile's expert costs shared-memory reads only
  int tile_off[kMaxExperts + 1];
  int expert_off[kMaxExperts + 1];
};

// Warp-uniform bounded wait: every lane polls the barrier together (the
// suspending try_wait, executed convergently), the lanes agree with a vote,
// and the warp gives up together once the budget is spent or another role
// has aborted.  Returns the same verdict in all lanes; on success every lane
// has itself observed the completed phase.  The first wait in the grid that
// runs out records where: status[1] = warp + 1, status[2] = barrier id,
// status[3] = step, status[4] = parity, status[5] = CTA, status[6..13] = how
// far each role of that CTA had got.
__device__ __forceinline__ bool warp_wait(WsShared& sh, uint64_t* bar, uint32_t parity,
                                          int32_t* status, int bar_id = 0, int step = 0) {
  constexpr unsigned kAll = 0xffffffffu;
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(kAll, done)) return true;
  const WaitBudget b = wait_budget();
  for (uint32_t n = 1;; ++n) {
    if (__any_sync(kAll, done)) {
      // the phase is complete: lanes that polled just before it completed
      // observe it now (bounded, although the phase cannot move on while
      // this warp has not consumed it)
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
      // [6] codes issued, [7..8] min/max activation steps published,
      // [9..10] min/max steps decoded, [11] steps issued to the tensor
      // core, [12] tiles it started, [13] tiles the epilogue finished
      const volatile int* pg = sh.prog;
      int lmin = pg[W_LOAD0], lmax = pg[W_LOAD0], dmin = pg[W_DEC0], dmax = pg[W_DEC0];
      for (int i = 1; i < kLoadWarps; ++i) {
        lmin = min(lmin, pg[W_LOAD0 + i]);
        lmax = max(lmax, pg[W_LOAD0 + i]);
      }
      for (int i = 1; i < kDecWarps; ++i) {
        dmin = min(dmin, pg[W_DEC0 + i]);
        dmax = max(dmax, pg[W_DEC0 + i]);
      }
      status[6] = pg[W_TMA];
      status[7] = lmin;
      status[8] = lmax;
      status[9] = dmin;
      status[10] = dmax;
      status[11] = pg[kWarps];
      status[12] = pg[kWarps + 1];
      status[13] = pg[kWarps + 2];
    }
  }
  __syncwarp();
  return false;
}

struct TileInfo {
  int e, r0, mrows, m0, n0;
};

// Tile t -> expert, rows and columns, from the shared-memory copies.
__device__ __forceinline__ TileInfo tile_info(const WsShared& sh, const GemmArgs& a, int t,
                                              bool gateup) {
  TileInfo ti;
  const int slot = t / a.n_ntiles, nt = t % a.n_ntiles;
  int lo = 0, hi = a.E;  // largest e with tile_off[e] <= slot
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh.tile_off[mid] <= slot) lo = mid; else hi = mid;
  }
  ti.e = lo;
  ti.r0 = sh.expert_off[lo];
  ti.m0 = (slot - sh.tile_off[lo]) * BM;
  ti.mrows = min(BM, sh.expert_off[lo + 1] - ti.r0 - ti.m0);
  ti.n0 = nt * (gateup ? BN / 2 : BN);
  return ti;
}

}  // namespace

template <bool GATEUP>
__global__ void __launch_bounds__(kThreadsWS, 1)
k_expert_gemm_ws(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                 const __grid_constant__ CUtensorMap tm2, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ WsShared sh;
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const GemmArgs& a = args;
  const int n_tiles = a.tile_off[a.E] * a.n_ntiles;
  if ((int)blockIdx.x >= n_tiles) return;  // uniform per CTA, before any barrier
  const int nK = a.K / BK;
  const int nKb = cdiv(a.K, kScaleBlock);
  const int nRb = cdiv(a.rows_per_expert, kScaleBlock);

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t smem_base = smem_u32(smem);

  if (tid == 0) {
    for (int s = 0; s < NB; ++s) {
      mbar_init(&sh.b8_full[s], 1);
      mbar_init(&sh.b8_empty[s], kDecWarps);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&sh.a_full[s], GATEUP ? kLoadWarps : 1);
      mbar_init(&sh.a_empty[s], 1);
    }
    for (int s = 0; s < NC; ++s) {
      mbar_init(&sh.b16_full[s], kDecWarps);
      mbar_init(&sh.b16_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.acc_full[s], 1);
      mbar_init(&sh.acc_empty[s], 4);
    }
    sh.abort_flag = 0;
    for (int i = 0; i < kWarps + 3; ++i) sh.prog[i] = 0;
    fence_mbar_init();
  }
  for (int i = tid; i <= a.E; i += kThreadsWS) {
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

  if (warp == W_TMA) {
    // ------------------------------------------------ E4M3 code tiles (TMA)
    int j = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(sh, a, t, GATEUP);
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sb = j % NB;
        if (j >= NB && !warp_wait(sh, &sh.b8_empty[sb], (uint32_t)(((j / NB) - 1) & 1), a.status, 1, j)) {
          ok = false;
          break;
        }
        // the decoders' reads of this slot (generic proxy) are ordered before
        // the copies that overwrite it (async proxy)
        tc::fence_proxy_async();
        if (lane == 0) {
          uint8_t* dst = smem + OFF_B8 + sb * B8_BYTES;
          mbar_arrive_expect_tx(&sh.b8_full[sb], B8_BYTES);
          const int row = ti.e * a.rows_per_expert + ti.n0;
          if (GATEUP) {
            tc::tma_load_2d(dst, &tm0, ks * BK, row, &sh.b8_full[sb]);
            tc::tma_load_2d(dst + 128 * BK, &tm1, ks * BK, row, &sh.b8_full[sb]);
          } else {
            tc::tma_load_2d(dst, &tm0, ks * BK, row, &sh.b8_full[sb]);
          }
          reinterpret_cast<volatile int*>(sh.prog)[W_TMA] = j + 1;
        }
        __syncwarp();
      }
    }
    // drain: the copies of the last NB steps issued must have landed
    if (lane == 0)
      for (int i = max(0, j - NB); i < j; ++i) mbar_wait(&sh.b8_full[i % NB], (uint32_t)((i / NB) & 1));
  } else if (!GATEUP && warp > W_LOAD0 && warp < W_LOAD0 + kLoadWarps) {
    // down: one TMA warp loads the rows; the other loader warps idle
  } else if (!GATEUP && warp == W_LOAD0) {
    // ------------------------------------------------ hid rows (TMA, down)
    // The down projection's rows are consecutive permuted rows: one
    // 128-byte-swizzled box of 64 columns x 128 rows per step (rows past the
    // expert's segment are computed and never stored; rows past P read 0).
    int j = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(sh, a, t, GATEUP);
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sa = j % NA;
        if (j >= NA && !warp_wait(sh, &sh.a_empty[sa], (uint32_t)(((j / NA) - 1) & 1), a.status, 2, j)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sh.a_full[sa], A_BYTES);
          tc::tma_load_2d(smem + OFF_A + sa * A_BYTES, &tm1, ks * BK, ti.r0 + ti.m0, &sh.a_full[sa]);
          reinterpret_cast<volatile int*>(sh.prog)[warp] = j + 1;
        }
        __syncwarp();
      }
    }
    // drain: the copies of the last NA steps issued must have landed
    if (lane == 0)
      for (int i = max(0, j - NA); i < j; ++i) mbar_wait(&sh.a_full[i % NA], (uint32_t)((i / NA) & 1));
    __syncwarp();
  } else if (GATEUP && warp >= W_LOAD0 && warp < W_LOAD0 + kLoadWarps) {
    // ------------------------------------------------ activation rows (cp.async)
    constexpr int RPT = (BM * 8) / kLoadThreads;  // 16-byte chunks per thread per step
    const int lt = tid - W_LOAD0 * 32;
    const int jj = lt & 7, mb = lt >> 3;  // chunk in row; rows mb + (kLoadThreads/8) u
    int j = 0;
    bool ok = true;
    // source rows of a tile (token rows for gate/up)
    auto rows_of = [&](int t, int (&src)[RPT]) {
      const TileInfo ti = tile_info(sh, a, t, GATEUP);
#pragma unroll
      for (int u = 0; u < RPT; ++u) {
        const int m = mb + (kLoadThreads / 8) * u;
        src[u] = m < ti.mrows ? a.row_token[ti.r0 + ti.m0 + m] : -1;
      }
    };
    int src_next[RPT];
    if ((int)blockIdx.x < n_tiles) rows_of(blockIdx.x, src_next);
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      int src[RPT];
#pragma unroll
      for (int u = 0; u < RPT; ++u) src[u] = src_next[u];
      // the next tile's token rows load while this tile streams
      if (t + (int)gridDim.x < n_tiles) rows_of(t + gridDim.x, src_next);
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sa = j % NA;
        if (j >= NA && !warp_wait(sh, &sh.a_empty[sa], (uint32_t)(((j / NA) - 1) & 1), a.status, 2, j)) {
          ok = false;
          break;
        }
        uint8_t* A = smem + OFF_A + sa * A_BYTES;
        const int k0 = ks * BK;
#pragma unroll
        for (int u = 0; u < RPT; ++u) {
          const int m = mb + (kLoadThreads / 8) * u;
          const uint16_t* g = a.asrc + (size_t)(src[u] < 0 ? 0 : src[u]) * a.K + k0 + 8 * jj;
          tc::cp_async16_zfill(A + tc::sw128_off(m, jj), g, src[u] >= 0);
        }
        cp_async_commit();
        // Publish step j - kALag: this thread's copies of it have landed (at
        // most kALag newer groups still pending, so kALag + 1 steps of
        // gathers stay in flight), then the proxy fence makes them visible
        // to tensor-core reads.
        // One arrival per loader warp, after every lane's wait and fence.
        if (j >= kALag) {
          cp_async_wait<kALag>();
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sh.a_full[(j - kALag) % NA]);
            reinterpret_cast<volatile int*>(sh.prog)[warp] = j - kALag + 1;
          }
        }
      }
    }
    // publish the last steps
    cp_async_wait<0>();
    tc::fence_proxy_async();
    __syncwarp();
    if (ok && lane == 0)
      for (int p = max(0, j - kALag); p < j; ++p) mbar_arrive(&sh.a_full[p % NA]);
  } else if (warp >= W_DEC0 && warp < W_DEC0 + kDecWarps) {
    // ------------------------------------------------ decode E4M3 -> fp16
    const int dt = tid - W_DEC0 * 32;
    int j = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(sh, a, t, GATEUP);
      const size_t srow = (size_t)ti.e * nRb + ti.n0 / kScaleBlock;
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sb = j % NB, c = j % NC;
        if (!warp_wait(sh, &sh.b8_full[sb], (uint32_t)((j / NB) & 1), a.status, 3, j) ||
            (j >= NC && !warp_wait(sh, &sh.b16_empty[c], (uint32_t)(((j / NC) - 1) & 1), a.status, 4, j))) {
          ok = false;
          break;
        }
        const int kb = ks * BK / kScaleBlock;
        const float sc0 = a.s0[srow * nKb + kb];
        const float sc1 = GATEUP ? a.s1[srow * nKb + kb] : a.s0[(srow + 1) * nKb + kb];
        const uint32_t s2[2] = {(uint32_t)f32_to_f16_bits(sc0) * 0x10001u,
                                (uint32_t)f32_to_f16_bits(sc1) * 0x10001u};
        const uint8_t* B8 = smem + OFF_B8 + sb * B8_BYTES;
        uint8_t* B16 = smem + OFF_B16 + c * B16_BYTES;
        constexpr int IPT = (BN * 4) / kDecThreads;  // items of 16 codes per thread
        uint4 c16[IPT];
#pragma unroll
        for (int u = 0; u < IPT; ++u) {
          const int q = dt + kDecThreads * u;
          c16[u] = *reinterpret_cast<const uint4*>(B8 + (q >> 2) * 64 + 16 * (q & 3));
        }
#pragma unroll
        for (int u = 0; u < IPT; ++u) {
          const int q = dt + kDecThreads * u;
          const int r = q >> 2, jp = 2 * (q & 3);
          const uint32_t sv = s2[r >> 7];
          const uint32_t w[4] = {c16[u].x, c16[u].y, c16[u].z, c16[u].w};
          uint32_t h[8];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            h[2 * v] = e4m3x2_to_f16x2(w[v] & 0xFFFFu);
            h[2 * v + 1] = e4m3x2_to_f16x2(w[v] >> 16);
          }
#pragma unroll
          for (int v = 0; v < 8; ++v)
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h[v]) : "r"(h[v]), "r"(sv));
          *reinterpret_cast<uint4*>(B16 + tc::sw128_off(r, jp)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(B16 + tc::sw128_off(r, jp + 1)) =
              make_uint4(h[4], h[5], h[6], h[7]);
        }
        tc::fence_proxy_async();  // decoded tile -> tensor-core reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh.b16_full[c]);
          mbar_arrive(&sh.b8_empty[sb]);
          reinterpret_cast<volatile int*>(sh.prog)[warp] = j + 1;
        }
      }
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------ tcgen05.mma issue
    const uint32_t idesc = tc::idesc_f16_f32(BM, BN);
    int j = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tl) {
      const int acc = tl & 1;
      if (tl >= 2 && !warp_wait(sh, &sh.acc_empty[acc], (uint32_t)(((tl >> 1) - 1) & 1), a.status, 5, tl)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t dcol = tmem + (uint32_t)(acc * BN);
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sa = j % NA, c = j % NC;
        if (!warp_wait(sh, &sh.a_full[sa], (uint32_t)((j / NA) & 1), a.status, 6, j) ||
            !warp_wait(sh, &sh.b16_full[c], (uint32_t)((j / NC) & 1), a.status, 7, j)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (lane == 0) {
          const uint32_t a_addr = smem_base + OFF_A + sa * A_BYTES;
          const uint32_t b_addr = smem_base + OFF_B16 + c * B16_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_f16(dcol, tc::sw128_desc(a_addr + kk * 32), tc::sw128_desc(b_addr + kk * 32),
                        idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          tc::commit(&sh.a_empty[sa]);
          tc::commit(&sh.b16_empty[c]);
          if (ks == nK - 1) tc::commit(&sh.acc_full[acc]);
          reinterpret_cast<volatile int*>(sh.prog)[kWarps] = j + 1;
          reinterpret_cast<volatile int*>(sh.prog)[kWarps + 1] = tl + 1;
        }
        __syncwarp();
      }
    }
    // drain: every MMA issued has completed once the newest commit has
    if (lane == 0 && j > 0) mbar_wait(&sh.a_empty[(j - 1) % NA], (uint32_t)(((j - 1) / NA) & 1));
  } else {
    // ------------------------------------------------ epilogue (warps 12-15)
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    int tl = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
      const int acc = tl & 1;
      if (!warp_wait(sh, &sh.acc_full[acc], (uint32_t)((tl >> 1) & 1), a.status, 8, tl)) break;
      tc::fence_after_sync();
      const TileInfo ti = tile_info(sh, a, t, GATEUP);
      const uint32_t tl_addr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
      if (GATEUP) {
        uint16_t* hid = reinterpret_cast<uint16_t*>(a.out);
        bool overflow = false;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          const int col = c4 * 32;
          uint32_t gr[32], ur[32];
          tc::ld_32x32b_x32(tl_addr + col, gr);
          tc::ld_32x32b_x32(tl_addr + 128 + col, ur);
          tc::wait_ld();
          if (m < ti.mrows) {
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
            uint4* dst = reinterpret_cast<uint4*>(
                hid + (size_t)(ti.r0 + ti.m0 + m) * a.out_ld + ti.n0 + col);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        if (overflow) raise_status(a.status, MOE_DEV_FP16_RANGE);
      } else {
        float* y = reinterpret_cast<float*>(a.out);
        // A warp whose 32 rows all belong to the tile's expert stages each
        // 32-column chunk in shared memory and writes it with one TMA store
        // (whole 128-byte row segments); a partial group stores directly.
        const bool whole = quad * 32 + 32 <= ti.mrows;
        uint8_t* stg = smem + OFF_EPI + quad * 4096;
#pragma unroll 1
        for (int c8 = 0; c8 < 8; ++c8) {
          const int col = c8 * 32;
          uint32_t v[32];
          tc::ld_32x32b_x32(tl_addr + col, v);
          tc::wait_ld();
          if (whole) {
            if (lane == 0) tc::bulk_wait_read_all();  // the previous store has read the tile
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              tc::tma_store_2d(&tm2, ti.n0 + col, ti.r0 + ti.m0 + quad * 32, stg);
              tc::bulk_commit();
            }
          } else if (m < ti.mrows) {
            float4* dst = reinterpret_cast<float4*>(
                y + (size_t)(ti.r0 + ti.m0 + m) * a.out_ld + ti.n0 + col);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acc_empty[acc]);
      if (lane == 0 && quad == 0) reinterpret_cast<volatile int*>(sh.prog)[kWarps + 2] = tl + 1;
    }
    if (!GATEUP && lane == 0) tc::bulk_wait_all();  // every TMA store is complete
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t get_encoder(EncodeTiled* out) {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                           &q);
    if (err == cudaSuccess && q != cudaDriverEntryPointSuccess) err = cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiled>(p);
  });
  *out = fn;
  return fn ? cudaSuccess : (err != cudaSuccess ? err : cudaErrorNotSupported);
}
}  // namespace

namespace {
// 2-D map over a row-major matrix [rows, cols] of esize-byte elements.
cudaError_t make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, int esize, const void* base,
                        long long rows, int cols, int box_cols, int box_rows, int swizzle_bytes) {
  EncodeTiled enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t make_u8_tensor_map(CUtensorMap* map, const uint8_t* base, long long rows, int cols,
                               int box_cols, int box_rows, bool swizzle128) {
  return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, box_cols, box_rows,
                     swizzle128 ? 128 : 0);
}

namespace {
// 2-D map over a stack of code matrices [rows_total, K] (uint8, row-major),
// box = 64 bytes of K x box_rows rows, no swizzle.
cudaError_t code_map(CUtensorMap* map, const uint8_t* codes, long long rows_total, int K,
                     int box_rows) {
  return make_u8_tensor_map(map, codes, rows_total, K, BK, box_rows, false);
}

}  // namespace

bool expert_gemm_tc_ok(int H, int I) {
  return H % 256 == 0 && I % 128 == 0 && H >= 256 && I >= 128;
}

cudaError_t launch_expert_gemm_tc(const uint16_t* x16, const int32_t* expert_off,
                                  const int32_t* row_token, int E, int P, const moe_fp8_ffn& w,
                                  int H, int I, int32_t* tile_off, uint16_t* hid, float* y,
                                  int32_t* status, cudaStream_t s, bool pdl) {
  cudaError_t err;
  if ((err = ensure_smem((const void*)k_expert_gemm_ws<true>, SMEM_WS)) != cudaSuccess) return err;
  if ((err = ensure_smem((const void*)k_expert_gemm_ws<false>, SMEM_WS)) != cudaSuccess) return err;
  CUtensorMap gmap, umap, dmap;
  if ((err = code_map(&gmap, w.gate.codes, (long long)E * I, H, 128)) != cudaSuccess) return err;
  if ((err = code_map(&umap, w.up.codes, (long long)E * I, H, 128)) != cudaSuccess) return err;
  if ((err = code_map(&dmap, w.down.codes, (long long)E * H, I, 256)) != cudaSuccess) return err;
  // hid [P, I] fp16, read by the down projection: 64 columns x 128 rows,
  // 128-byte swizzled (the K-major operand layout the MMA descriptors use)
  CUtensorMap hmap, ymap;
  if ((err = make_map_2d(&hmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hid, P, I, BK, BM, 128)) !=
      cudaSuccess)
    return err;
  // y [P, H] fp32, written by the down epilogue: 32 columns x 32 rows, swizzled
  if ((err = make_map_2d(&ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, P, H, 32, 32, 128)) !=
      cudaSuccess)
    return err;
  err = launch_k(k_tile_offsets, dim3(1), dim3(1024), 0, s, pdl, expert_off, E, tile_off);
  if (err != cudaSuccess) return err;
  // Host bound on the tile count: each expert adds at most one partial tile.
  const int max_mtiles = cdiv(P, BM) + min(E, P);
  const int nsm = num_sms();
  const dim3 blk(kThreadsWS);
  GemmArgs g{x16, H, I, expert_off, row_token, tile_off, E, w.gate.scales, w.up.scales,
             (void*)hid, I, I / (BN / 2), status};
  err = launch_k(k_expert_gemm_ws<true>, dim3(min(nsm, max_mtiles * g.n_ntiles)), blk,
                 (size_t)SMEM_WS, s, pdl, gmap, umap, ymap, g);
  if (err != cudaSuccess) return err;
  GemmArgs d{(const uint16_t*)hid, I, H, expert_off, row_token, tile_off, E, w.down.scales,
             nullptr, (void*)y, H, H / BN, status};
  return launch_k(k_expert_gemm_ws<false>, dim3(min(nsm, max_mtiles * d.n_ntiles)), blk,
                  (size_t)SMEM_WS, s, pdl, dmap, hmap, ymap, d);
}

}  // namespace moe
