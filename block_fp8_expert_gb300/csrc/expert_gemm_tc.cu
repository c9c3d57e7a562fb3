// Routed-expert FFN for many tokens per expert (prefill): a grouped GEMM on
// the 5th-generation tensor cores (colizig README, "Features": block-FP8
// weights; "MoE per-expert evaluation").
//
// The weights are the MMA's A operand and live in tensor memory; the tokens
// are its B operand (N = tokens) in shared memory.  A tile is one expert,
// up to 128 of its permuted token rows and two 128-row weight blocks:
//   gate/up: the gate rows n0..n0+127 and the same up rows, K = H; the
//            epilogue writes hid = silu(g) * u in fp16;
//   down:    output rows n0..n0+255 as two blocks of 128, K = I; the epilogue
//            writes y in fp32, or fp16 with one exponent per 32 columns.
// Range: every operand and intermediate is normalised by an exact power of
// two, so the fp16 formats hold any block-scale and activation magnitude:
//   x'  = x 2^-a per token row (a = floor(log2 rms(x)), by the gather);
//   W'  = dec(code) * (S / 2^p), p = floor(log2) of the largest scale of the
//         expert's gate (or up) matrix, or of the down row block;
//   hid'= silu(g) u / 2^(a + pg + a + pu + c), c = floor(log2 H) + 4: the
//         accumulators give it as sigma(g) D0 D1 2^-c, independent of every
//         scale and of the activations' magnitude;
//   y   = D 2^(pd + pg + pu + c + 2a).
// A hid' value beyond fp16's range, or a token whose 32 features of one
// epilogue warp all fall below 2^-12 (where fp16's spacing would cost
// precision), raises MOE_DEV_FP16_RANGE; a non-finite scale, activation or
// result raises MOE_DEV_NONFINITE.
// Two accumulators D0, D1 (128 lanes = weight rows x N columns = tokens, fp32)
// use TMEM columns 0..255; columns 256..511 hold four stages of decoded
// weights (two 128 x 64 fp16 blocks per 64-wide K step).  N is the tile's row
// count rounded up to 16, so a ragged last tile of an expert costs only its
// rows.  A tile list holds the gate/up tiles, then the down tiles; a down
// tile's token rows wait only for its own token tile's gate/up tiles (a
// per-token-tile counter).  With few tiles per SM (decode batches) one
// launch runs the whole list (kBoth), so an SM streams down codes as soon as
// its last gate/up tile's codes are in, instead of leaving the SM to a second
// launch; otherwise the gate/up tiles (kGateUp) and the down tiles (kDown)
// are two launches, the second's CTAs starting on SMs the first has left.
// Persistent CTAs (one per SM) walk a static sequence of the list (TileSeq).
// Warp-specialised roles hand work to each other through mbarriers:
//   warp 0      TMA: the step's two E4M3 code blocks (64-byte swizzled) into
//               a ring in shared memory;
//   warp 1      TMA: the step's token rows into a ring in shared memory, one
//               128-byte-swizzled box of 128 consecutive rows of the
//               permuted activations (gate/up: x gathered into expert order
//               by k_gather_rows; down: hid);
//   warp 2      one elected thread issues tcgen05.mma (M = 128, N, K = 16),
//               A from TMEM, and commits to mbarriers;
//   warps 3-10  decode codes to fp16 times the block scale
//               (fp16(dec * fp16(scale))) and store them into a TMEM stage;
//               warp w serves TMEM lanes 32 (w % 4) .. + 31 of one block;
//   warps 11-18 epilogue: tcgen05.ld from the accumulators, SwiGLU, stores;
//               warp w reads TMEM lanes 32 (w % 4) .. + 31, half of the
//               tile's columns (gate/up) or one of the two blocks (down).
// Every wait is bounded (about 2 s) and also gives up as soon as another
// role has given up, recording MOE_DEV_WAIT_TIMEOUT; the CTA then drains its
// copies and MMAs and frees its TMEM before it exits.
#include <cuda.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {
constexpr int BT = 128;  // token rows per tile (MMA N, at most)
constexpr int BW = 128;  // weight rows per block (MMA M)
constexpr int BK = 64;   // K per step
constexpr int NT = 5, NCD = 5, NA = 4;  // ring depths: tokens, codes, TMEM weight stages
constexpr int T_BYTES = BT * BK * 2;    // 16 KB
constexpr int C_BYTES = 2 * BW * BK;    // 16 KB: two code blocks of 8 KB
constexpr int OFF_T = 0;
constexpr int OFF_C = OFF_T + NT * T_BYTES;
// Epilogue staging, 4 KB per epilogue warp: gate/up stages its half of a hid
// tile, [64 tokens][32 features] fp16, written one 64-byte row per bulk copy;
// down stages one fp32 tile [32 tokens][32 features] (128-byte swizzled) at a
// time, each written by one TMA store.
constexpr int STG_WARP_BYTES = 4096;
constexpr int OFF_STG = OFF_C + NCD * C_BYTES;
constexpr int kDecWarps = 8, kEpiWarps = 8;
constexpr int STG_BYTES = kEpiWarps * STG_WARP_BYTES;  // 32 KB
constexpr int SMEM_WS = OFF_STG + STG_BYTES + 1024;  // + alignment slack
// warp roles: code TMA, token TMA, MMA issue, decoders, epilogue
constexpr int W_CODES = 0, W_TOK = 1, W_MMA = 2, W_DEC0 = 3, W_EPI0 = W_DEC0 + kDecWarps;
constexpr int kWarps = W_EPI0 + kEpiWarps;
constexpr int kThreadsWS = kWarps * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_D1 = BT;       // D0 at column 0, D1 at 128
constexpr uint32_t COL_A = 2 * BT;    // weight stages from column 256
constexpr uint32_t A_STAGE_COLS = 64;  // two blocks x 32 columns (64 fp16 of K)
static_assert(COL_A + NA * A_STAGE_COLS <= TMEM_COLS, "TMEM budget");
static_assert(kDecWarps == 8 && kEpiWarps == 8, "two blocks (or halves) x four lane quarters");

// The expert FFN's two GEMMs as one tile list: every gate/up tile (a token
// tile x 128 gate rows and the same up rows, K = H), then every down tile (a
// token tile x 256 output rows, K = I), each part in token-tile ("slot")
// order.  A launch runs all of it or one part (FfnMode).
enum FfnMode { kBoth = 0, kGateUp = 1, kDown = 2 };

struct FfnArgs {
  const int32_t* expert_off;
  const int32_t* tile_off;  // token-tile prefix per expert, [E + 1]
  int E;
  int H, I;
  const float* gs;  // gate, up and down block scales
  const float* us;
  const float* ds;
  uint16_t* hid;    // [P, I] fp16: the gate/up output, the down input
  void* y;          // [P, H]: fp32, or fp16 when yexp is set
  int all_wait;     // 1: the previous kernel wrote the tile offsets (every warp waits)
  // Per token tile: completed gate/up epilogue-warp tiles.  Each gate/up
  // weight-block tile adds kEpiWarps once its hid rows are stored; a down
  // tile's token warp waits for slot_need before it loads the slot's rows.
  int32_t* slot_done;
  int slot_need;
  int32_t* status;
  // Range normalisation (see the top of this file)
  const int32_t* xexp;  // a of each permuted row: its activations are x' 2^a
  int hid_shift;        // c
  // fp16 y only: exponent s per 32 columns and row (y = y'' 2^s),
  // [H / 32][yexp_rows]; NULL: y is fp32
  int16_t* yexp;
  int yexp_rows;
  // bounded waits give up after this many nanoseconds (0: the default);
  // a diagnostic setting (MOE_FP8_WAIT_LIMIT_US)
  uint64_t wait_ns;
};


struct WsShared {
  uint64_t c_full[NCD], c_empty[NCD];
  uint64_t t_full[NT], t_empty[NT];
  uint64_t a_full[NA], a_empty[NA];
  uint64_t acc_full, acc_empty;
  uint32_t tmem_base;
  int abort_flag;
  uint64_t wait_ns;  // the role waits' budget (FfnArgs::wait_ns)
  // Steps each role has completed, for the timeout record: [warp] for the
  // TMA warps (steps issued) and the decoder warps (steps decoded),
  // [kWarps] steps issued to the tensor core, [kWarps + 1] tiles started by
  // it, [kWarps + 2] tiles finished by the epilogue.
  int prog[kWarps + 3];
  // copies of the per-expert tile prefix and row offsets (E + 1 entries),
  // so that finding a tile's expert costs shared-memory reads only
  int tile_off[kMaxExperts + 1];
  int expert_off[kMaxExperts + 1];
  // down epilogue: each warp's row exponents a of the current tile
  int8_t ax[kEpiWarps][BT];
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
  const WaitBudget b = wait_budget(sh.wait_ns);
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
      // [6] code steps issued, [7] token steps issued, [8..9] min/max steps
      // decoded, [10] steps issued to the tensor core, [11] tiles it
      // started, [12] tiles the epilogue finished
      const volatile int* pg = sh.prog;
      int dmin = pg[W_DEC0], dmax = pg[W_DEC0];
      for (int i = 1; i < kDecWarps; ++i) {
        dmin = min(dmin, pg[W_DEC0 + i]);
        dmax = max(dmax, pg[W_DEC0 + i]);
      }
      status[6] = pg[W_CODES];
      status[7] = pg[W_TOK];
      status[8] = dmin;
      status[9] = dmax;
      status[10] = pg[kWarps];
      status[11] = pg[kWarps + 1];
      status[12] = pg[kWarps + 2];
    }
  }
  __syncwarp();
  return false;
}

// Waits for N barrier phases: one round of non-blocking probes issued back to
// back (their latencies overlap), then, if any phase is still open, the
// bounded warp-uniform wait on each in turn.
template <int N>
__device__ __forceinline__ bool warp_wait_all(WsShared& sh, uint64_t* const (&bar)[N],
                                              const uint32_t (&parity)[N], int32_t* status,
                                              const int (&bar_id)[N], int step) {
  bool done = true;
#pragma unroll
  for (int i = 0; i < N; ++i) done &= mbar_test_wait(bar[i], parity[i]);
  if (__all_sync(0xffffffffu, done)) return true;
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (!warp_wait(sh, bar[i], parity[i], status, bar_id[i], step)) return false;
  return true;
}

struct TileInfo {
  int e, r0, m0, rows, n, n0;  // n = rows rounded up to 16 (the MMA's N)
  int slot;                    // token tile index (tile_off[e] + m0 / 128)
  bool gu;                     // a gate/up tile (else down)
  int K, nK;                   // the contraction length and its 64-wide steps
};

// List entry t -> phase, expert, token rows and weight rows, from the
// shared-memory copies of the offsets (n_gu: gate/up tiles in the list).
template <int MODE>
__device__ __forceinline__ TileInfo tile_info(const WsShared& sh, const FfnArgs& a, int t,
                                              int n_gu) {
  TileInfo ti;
  ti.gu = MODE == kBoth ? t < n_gu : MODE == kGateUp;
  const int u = ti.gu ? t : t - n_gu;
  const int nwb = ti.gu ? a.I / BW : a.H / (2 * BW);  // weight tiles per token tile
  const int slot = u / nwb, wb = u - slot * nwb;
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
  ti.n0 = wb * (ti.gu ? BW : 2 * BW);
  ti.K = ti.gu ? a.H : a.I;
  ti.nK = ti.K / BK;
  return ti;
}

// This CTA's tiles, in order: gate/up tiles i, i + G, ... (the first r of
// the G CTAs hold one more when G does not divide them), then down tiles.
// A gate/up tile costs about m = round(H / I) down tiles (the same 256 x N
// shape with K = H rather than I), so the r CTAs with the extra gate/up tile
// sit out the first m rounds of down tiles; every other round goes to all G.
// Every role of the CTA walks the same sequence.
struct TileSeq {
  int i, G, n_gu, n_dn, r, m, k = 0, jj = 0;
  bool in_gu = true;
  __device__ TileSeq(int i_, int G_, int n_gu_, int n_dn_, int m_)
      : i(i_), G(G_), n_gu(n_gu_), n_dn(n_dn_), r(n_gu_ % G_), m(m_) {}
  __device__ int next() {  // a list index, or -1 after the last
    if (in_gu) {
      const int t = i + k * G;
      if (t < n_gu) {
        ++k;
        return t;
      }
      in_gu = false;
    }
    const int d = i >= r ? (jj < m ? jj * (G - r) + (i - r) : m * (G - r) + (jj - m) * G + i)
                         : m * (G - r) + jj * G + i;
    if (d >= n_dn) return -1;
    ++jj;
    return n_gu + d;
  }
};

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kThreadsWS, 1)
k_expert_ffn_ws(const __grid_constant__ CUtensorMap cm_g, const __grid_constant__ CUtensorMap cm_u,
                const __grid_constant__ CUtensorMap cm_d, const __grid_constant__ CUtensorMap tm_x,
                const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_y,
                const FfnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ WsShared sh;
  // Only the token warp and the epilogue wait for the previous kernel (they
  // read its output: the expert-order activation rows and their exponents).
  // Everything else reads data written two or more launches back (tile and
  // row offsets, weights), so on SMs the previous kernel
  // has already left the codes are fetched and decoded while it finishes.
  if (args.all_wait) griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const FfnArgs& a = args;
  const int n_slots = a.tile_off[a.E];
  const int n_gu = MODE == kDown ? 0 : n_slots * (a.I / BW);
  const int n_all = n_gu + (MODE == kGateUp ? 0 : n_slots * (a.H / (2 * BW)));
  // uniform per CTA, before any barrier
  if ((int)blockIdx.x >= n_all) return;
  const int G = (int)gridDim.x;
  const int m_skip = (a.H + a.I / 2) / a.I;
  auto seq = [&]() { return TileSeq((int)blockIdx.x, G, n_gu, n_all - n_gu, m_skip); };

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t smem_base = smem_u32(smem);

  if (tid == 0) {
    for (int s = 0; s < NCD; ++s) {
      mbar_init(&sh.c_full[s], 1);
      mbar_init(&sh.c_empty[s], kDecWarps);
    }
    for (int s = 0; s < NT; ++s) {
      mbar_init(&sh.t_full[s], 1);
      mbar_init(&sh.t_empty[s], 1);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&sh.a_full[s], kDecWarps);
      mbar_init(&sh.a_empty[s], 1);
    }
    mbar_init(&sh.acc_full, 1);
    mbar_init(&sh.acc_empty, kEpiWarps);
    sh.abort_flag = 0;
    sh.wait_ns = a.wait_ns;
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

  if (warp == W_CODES) {
    // ------------------------------------------------ E4M3 code blocks (TMA)
    int j = 0;
    bool ok = true;
    TileSeq sq = seq();
    for (int t = sq.next(); t >= 0 && ok; t = sq.next()) {
      const TileInfo ti = tile_info<MODE>(sh, a, t, n_gu);
      const int row = ti.e * (ti.gu ? a.I : a.H) + ti.n0;
      for (int ks = 0; ks < ti.nK; ++ks, ++j) {
        const int sc = j % NCD;
        if (j >= NCD && !warp_wait(sh, &sh.c_empty[sc], (uint32_t)(((j / NCD) - 1) & 1), a.status, 1, j)) {
          ok = false;
          break;
        }
        tc::fence_proxy_async();
        if (tc::elect_one()) {
          uint8_t* dst = smem + OFF_C + sc * C_BYTES;
          mbar_arrive_expect_tx(&sh.c_full[sc], C_BYTES);
          if (ti.gu) {
            tc::tma_load_2d(dst, &cm_g, ks * BK, row, &sh.c_full[sc]);
            tc::tma_load_2d(dst + BW * BK, &cm_u, ks * BK, row, &sh.c_full[sc]);
          } else {
            tc::tma_load_2d(dst, &cm_d, ks * BK, row, &sh.c_full[sc]);
            tc::tma_load_2d(dst + BW * BK, &cm_d, ks * BK, row + BW, &sh.c_full[sc]);
          }
          reinterpret_cast<volatile int*>(sh.prog)[W_CODES] = j + 1;
        }
        __syncwarp();
      }
    }
    if (lane == 0)
      for (int i = max(0, j - NCD); i < j; ++i) mbar_wait(&sh.c_full[i % NCD], (uint32_t)((i / NCD) & 1));
    __syncwarp();
  } else if (warp == W_TOK) {
    // ------------------------------------------------ token rows (TMA)
    // One box of 128 consecutive permuted rows per step (rows past the tile
    // are never stored; rows past the matrix read 0): x' for gate/up (after
    // the previous kernel, which wrote it, has completed), hid for down
    // (after the slot's gate/up tiles have stored it).
    bool waited = a.all_wait != 0;
    int j = 0;
    bool ok = true;
    TileSeq sq = seq();
    for (int t = sq.next(); t >= 0 && ok; t = sq.next()) {
      const TileInfo ti = tile_info<MODE>(sh, a, t, n_gu);
      if (ti.gu) {
        if (!waited) griddep_wait();
        waited = true;
      } else {
        // every gate/up weight-block tile of the slot has stored its hid
        // rows (bounded warp-uniform poll, then the acquired data is ordered
        // before the async-proxy loads below)
        const WaitBudget b = wait_budget(sh.wait_ns);
        bool done = false;
        for (uint32_t i = 0; !done; ++i) {
          done = __all_sync(0xffffffffu, tc::ld_acquire_gpu(a.slot_done + ti.slot) >= a.slot_need);
          if (!done && (i & 31) == 31) {
            const bool give_up =
                *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0 || budget_spent(b);
            if (__any_sync(0xffffffffu, give_up)) break;
          }
        }
        if (!done) {
          if (lane == 0 && !sh.abort_flag) {
            sh.abort_flag = 1;
            raise_status(a.status, MOE_DEV_WAIT_TIMEOUT);
            // where: the token warp's wait for a token tile's hid rows
            // (barrier id 9), the tile's slot and its completion count
            if (a.status && atomicCAS(a.status + 1, 0, 1 + W_TOK) == 0) {
              a.status[2] = 9;
              a.status[3] = ti.slot;
              a.status[4] = tc::ld_acquire_gpu(a.slot_done + ti.slot);
              a.status[5] = (int)blockIdx.x;
            }
          }
          __syncwarp();
          ok = false;
          break;
        }
        tc::fence_proxy_async_global();
      }
      const CUtensorMap* tm = ti.gu ? &tm_x : &tm_h;
      for (int ks = 0; ks < ti.nK; ++ks, ++j) {
        const int st = j % NT;
        if (j >= NT && !warp_wait(sh, &sh.t_empty[st], (uint32_t)(((j / NT) - 1) & 1), a.status, 2, j)) {
          ok = false;
          break;
        }
        if (tc::elect_one()) {
          mbar_arrive_expect_tx(&sh.t_full[st], T_BYTES);
          tc::tma_load_2d(smem + OFF_T + st * T_BYTES, tm, ks * BK, ti.r0 + ti.m0, &sh.t_full[st]);
          reinterpret_cast<volatile int*>(sh.prog)[warp] = j + 1;
        }
        __syncwarp();
      }
    }
    // drain: the copies of the last NT steps issued must have landed
    if (lane == 0)
      for (int i = max(0, j - NT); i < j; ++i) mbar_wait(&sh.t_full[i % NT], (uint32_t)((i / NT) & 1));
    __syncwarp();
  } else if (warp >= W_DEC0 && warp < W_DEC0 + kDecWarps) {
    // ------------------------------------------------ decode E4M3 -> fp16 -> TMEM
    // This warp: block blk (0: gate / first 128 down rows, 1: up / next 128),
    // weight rows 32 q .. 32 q + 31 of it = its TMEM lane quarter; the lane
    // owns one weight row and writes its 64 fp16 of K as 32 columns.
    const int blk = (warp - W_DEC0) >> 2, q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16) + COL_A + (uint32_t)blk * 32;
    // 64-byte swizzle of the code block: 16-byte chunk u of row r sits at
    // chunk u ^ ((r >> 1) & 3)
    const int swz = (r >> 1) & 3;
    // Block scales: lane i holds the decoder scale of K block i of the
    // tile's weight block (nKb <= 32), published with the tile's list entry
    // by the code warp, so that no step waits for global memory.
    bool bad = false;
    auto scale_of = [&](int t) -> float {
      const TileInfo ti = tile_info<MODE>(sh, a, t, n_gu);
      const float* sp = ti.gu ? (blk ? a.us : a.gs) : a.ds;
      const int nKb = cdiv(ti.K, kScaleBlock);
      const int nRb = cdiv(ti.gu ? a.I : a.H, kScaleBlock);
      const size_t srow = (size_t)ti.e * nRb + ti.n0 / kScaleBlock + (ti.gu ? 0 : blk);
      const float sc = lane < nKb ? sp[srow * nKb + lane] : 0.f;
      const int p = ti.gu ? warp_max_exp_of(sp + (size_t)ti.e * nRb * nKb, nRb * nKb, lane, bad)
                          : warp_max_exp(__float_as_uint(sc) & 0x7fffffffu, bad);
      return sc * pow2f(-p);
    };
    TileSeq sq = seq();
    int t = sq.next();
    float scale_next = t >= 0 ? scale_of(t) : 0.f;
    int j = 0;
    bool ok = true;
    for (int t_next; t >= 0 && ok; t = t_next) {
      const float scale_tile = scale_next;
      t_next = sq.next();
      if (t_next >= 0) scale_next = scale_of(t_next);
      const int nK = tile_info<MODE>(sh, a, t, n_gu).nK;
      for (int ks = 0; ks < nK; ++ks, ++j) {
        const int sc = j % NCD, sa = j % NA;
        const float scale = __shfl_sync(0xffffffffu, scale_tile, ks * BK / kScaleBlock);
        if (!warp_wait(sh, &sh.c_full[sc], (uint32_t)((j / NCD) & 1), a.status, 3, j) ||
            (j >= NA && !warp_wait(sh, &sh.a_empty[sa], (uint32_t)(((j / NA) - 1) & 1), a.status, 4, j))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();  // the MMAs that read this stage are complete
        const uint8_t* row = smem + OFF_C + sc * C_BYTES + blk * (BW * BK) + r * BK;
        uint4 c16[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) c16[u] = *reinterpret_cast<const uint4*>(row + 16 * (u ^ swz));
        const uint32_t s2 = (uint32_t)f32_to_f16_bits(scale) * 0x10001u;
        uint32_t h[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w[4] = {c16[u].x, c16[u].y, c16[u].z, c16[u].w};
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            h[8 * u + 2 * v] = e4m3x2_to_f16x2(w[v] & 0xFFFFu);
            h[8 * u + 2 * v + 1] = e4m3x2_to_f16x2(w[v] >> 16);
          }
        }
#pragma unroll
        for (int v = 0; v < 32; ++v) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h[v]) : "r"(h[v]), "r"(s2));
        tc::st_32x32b_x32(t_lane + (uint32_t)sa * A_STAGE_COLS, h);
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh.a_full[sa]);
          mbar_arrive(&sh.c_empty[sc]);
          reinterpret_cast<volatile int*>(sh.prog)[warp] = j + 1;
        }
      }
    }
    if (bad && lane == 0) raise_status(a.status, MOE_DEV_NONFINITE);
  } else if (warp == W_MMA) {
    // ------------------------------------------------ tcgen05.mma issue
    int j = 0, tl = 0;
    bool ok = true;
    TileSeq sq = seq();
    for (int t = sq.next(); t >= 0 && ok; t = sq.next(), ++tl) {
      const TileInfo ti = tile_info<MODE>(sh, a, t, n_gu);
      const int nK = ti.nK;
      const uint32_t idesc = tc::idesc_f16_f32(BW, ti.n);
      if (tl >= 1 && !warp_wait(sh, &sh.acc_empty, (uint32_t)((tl - 1) & 1), a.status, 5, tl)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // Two steps per round (nK is even: K is a multiple of 128): one wait for
      // both steps' operands, then their 16 MMAs back to back, so that the
      // tensor pipe's queue stays ahead of the barrier round trips.
      for (int ks = 0; ks < nK; ks += 2, j += 2) {
        const int st0 = j % NT, sa0 = j % NA, st1 = (j + 1) % NT, sa1 = (j + 1) % NA;
        uint64_t* const bars[4] = {&sh.t_full[st0], &sh.a_full[sa0], &sh.t_full[st1],
                                   &sh.a_full[sa1]};
        const uint32_t par[4] = {(uint32_t)((j / NT) & 1), (uint32_t)((j / NA) & 1),
                                 (uint32_t)(((j + 1) / NT) & 1), (uint32_t)(((j + 1) / NA) & 1)};
        const int ids[4] = {6, 7, 6, 7};
        if (!warp_wait_all(sh, bars, par, a.status, ids, j)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (tc::elect_one()) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int st = h ? st1 : st0, sa = h ? sa1 : sa0;
            const uint32_t b_addr = smem_base + OFF_T + st * T_BYTES;
            const uint32_t a_col = tmem + COL_A + (uint32_t)sa * A_STAGE_COLS;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t bdesc = tc::sw128_desc(b_addr + kk * 32);
              const uint32_t acc = (ks + h > 0 || kk > 0) ? 1u : 0u;
              tc::mma_f16_ts(tmem, a_col + kk * 8, bdesc, idesc, acc);
              tc::mma_f16_ts(tmem + COL_D1, a_col + 32 + kk * 8, bdesc, idesc, acc);
            }
            tc::commit(&sh.t_empty[st]);
            tc::commit(&sh.a_empty[sa]);
          }
          if (ks + 2 == nK) tc::commit(&sh.acc_full);
          reinterpret_cast<volatile int*>(sh.prog)[kWarps] = j + 2;
          reinterpret_cast<volatile int*>(sh.prog)[kWarps + 1] = tl + 1;
        }
        __syncwarp();
      }
    }
    // drain: every MMA issued has completed once the newest commit has
    if (lane == 0 && j > 0) mbar_wait(&sh.a_empty[(j - 1) % NA], (uint32_t)(((j - 1) / NA) & 1));
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (warps 11-18)
    // Lane quarter q of both accumulators: weight rows 32 q + lane; columns
    // are the tile's tokens.  Half eh of the epilogue warps takes the 32-token
    // chunks c = eh, eh + 2 (gate/up) or block eh (down).
    const int q = warp & 3, eh = (warp - W_EPI0) >> 2;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16);
    uint8_t* stg = smem + OFF_STG + (warp - W_EPI0) * STG_WARP_BYTES;
    // block scales per expert of one gate/up matrix, and of the down matrix:
    // [rows / 128][K / 128]
    const int nKb_g = cdiv(a.H, kScaleBlock), nRb_g = cdiv(a.I, kScaleBlock);
    const int n_gu_scales = nRb_g * nKb_g;
    const int nKb_d = cdiv(a.I, kScaleBlock), nRb_d = cdiv(a.H, kScaleBlock);
    const float inv_c = pow2f(-a.hid_shift);
    // the row exponents are read ahead of the accumulators: after the kernel
    // that wrote them has completed
    if (MODE != kDown && !a.all_wait) griddep_wait();
    bool bad = false;
    int tl = 0;
    TileSeq sq = seq();
    for (int t = sq.next(); t >= 0; t = sq.next(), ++tl) {
      const TileInfo ti = tile_info<MODE>(sh, a, t, n_gu);
      // the tile's powers of two (scales only: computed before the wait)
      int p0 = 0;  // gate/up: pg; down: pd + pg + pu + c
      if (ti.gu) {
        p0 = warp_max_exp_of(a.gs + (size_t)ti.e * n_gu_scales, n_gu_scales, lane, bad);
      } else {
        const size_t srow = (size_t)ti.e * nRb_d + ti.n0 / kScaleBlock + eh;
        const float sc = lane < nKb_d ? a.ds[srow * nKb_d + lane] : 0.f;
        p0 = warp_max_exp(__float_as_uint(sc) & 0x7fffffffu, bad) +
             warp_max_exp_of(a.gs + (size_t)ti.e * n_gu_scales, n_gu_scales, lane, bad) +
             warp_max_exp_of(a.us + (size_t)ti.e * n_gu_scales, n_gu_scales, lane, bad) +
             a.hid_shift;
      }
      // a of the tile's tokens, lane i holding token 32 c + i's for each
      // chunk c this warp takes (gate/up: c = eh, eh + 2; down: c = 0 .. 3),
      // all requested at once.  gate/up reads them before the accumulators
      // are ready (its epilogue warps waited for the kernel that wrote them);
      // down after its accumulator wait, which follows the token warp's
      // acquire of the tile's hid rows (the rows' writer had waited for them).
      // (|a| <= 126: one byte each; gate/up packs its two into a register,
      // down parks its four in the warp's shared bytes, chunk u at 32 u + lane)
      uint32_t axp = 0;
      int8_t* axs = sh.ax[warp - W_EPI0];
      auto load_ax = [&](int c0, int dc, int cnt) {
        int v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + dc * u;
          v[u] = (u < cnt && lane < ti.rows - 32 * c) ? __ldg(a.xexp + ti.r0 + ti.m0 + 32 * c + lane) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (ti.gu) axp |= ((uint32_t)v[u] & 0xffu) << (8 * u);
          else axs[32 * u + lane] = (int8_t)v[u];
        }
      };
      auto ax_of = [&](int u) {
        return ti.gu ? (int)(int8_t)(axp >> (8 * u)) : (int)axs[32 * u + lane];
      };
      if (ti.gu) load_ax(eh, 2, 2);
      // this warp's copies of the previous tile have read its staging
      tc::bulk_wait_read_all();
      __syncwarp();
      if (!warp_wait(sh, &sh.acc_full, (uint32_t)(tl & 1), a.status, 8, tl)) break;
      tc::fence_after_sync();
      const int nchunks = (ti.n + 31) >> 5;
      if (!ti.gu) load_ax(0, 1, 4);
      if (ti.gu) {
        bool overflow = false, underflow = false;
#pragma unroll 1
        for (int c = eh; c < nchunks; c += 2) {
          uint32_t gr[32], ur[32];
          tc::ld_32x32b_x32(t_lane + 32 * c, gr);
          tc::ld_32x32b_x32(t_lane + COL_D1 + 32 * c, ur);
          const int nv = ti.rows - 32 * c;  // columns of real tokens in this chunk
          const int ax = ax_of((c - eh) >> 1);
          tc::wait_ld();
          uint8_t* rows = stg + (c >> 1) * (32 * 64);
          uint32_t small = 0, nonzero = 0;
#pragma unroll
          for (int v = 0; v < 32; ++v) {
            const float d0 = __uint_as_float(gr[v]), d1 = __uint_as_float(ur[v]);
            // g = d0 2^(pg + a) decides the gate; the rest is normalised:
            // hid' = sigma(g) d0 d1 2^-c
            const int av = __shfl_sync(0xffffffffu, ax, v);
            const float g = d0 * pow2f(min(max(p0 + av, -126), 127));
            const float sig = __fdividef(1.f, 1.f + __expf(-fminf(fmaxf(g, -80.f), 80.f)));
            const float h = sig * d0 * d1 * inv_c;
            overflow |= v < nv && !(fabsf(h) <= kF16Max);
            small |= (uint32_t)(fabsf(h) < 0x1p-12f) << v;
            nonzero |= (uint32_t)(h != 0.f) << v;
            *reinterpret_cast<uint16_t*>(rows + v * 64 + lane * 2) = f32_to_f16_bits(h);
          }
          // a token (column) whose 32 features here are all tiny but not all
          // zero would lose precision to fp16's subnormal spacing
          const uint32_t valid = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
          if (__reduce_and_sync(0xffffffffu, small) & __reduce_or_sync(0xffffffffu, nonzero) & valid)
            underflow = true;
        }
        if (overflow || underflow) raise_status(a.status, MOE_DEV_FP16_RANGE);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.acc_empty);
        // staged rows -> bulk copies (async proxy): features 32 q .. + 31 of
        // each of this half's token rows, 64 bytes
        tc::fence_proxy_async();
        __syncwarp();
        uint16_t* hid = a.hid + (size_t)(ti.r0 + ti.m0) * a.I + ti.n0 + 32 * q;
        for (int i = lane; i < 64; i += 32) {
          const int c = 2 * (i >> 5) + eh, m = 32 * c + (i & 31);  // token row of staged row i
          if (m < ti.rows) tc::bulk_store(hid + (size_t)m * a.I, stg + i * 64, 64);
        }
        tc::bulk_commit();
        if (a.slot_done) {
          // publish: this warp's hid rows of the tile are stored
          tc::bulk_wait_all();
          tc::fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            tc::red_release_gpu_add(a.slot_done + ti.slot, 1);
          }
        }
      } else {
        // Chunk c of block eh: features col0 .. col0 + 31 (this warp's
        // lanes) x tokens 32 c .. 32 c + 31 (the chunk's columns).  The chunk
        // is staged in fp32 token-major (row = token, 128 bytes, 16-byte
        // groups swizzled by token % 8: conflict-free both ways), then lane r
        // reads back token 32 c + r's 32 values, so the token's power of two
        // and the group exponent of its 32 values are lane-local.  A chunk of
        // 32 real tokens leaves by one TMA store from the staging tile; a
        // ragged chunk's real rows by plain stores.
        const int col0 = ti.n0 + eh * BW + 32 * q;  // first of this warp's 32 columns
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tc::ld_32x32b_x32(t_lane + eh * COL_D1 + 32 * c, v);
          const int nv = ti.rows - 32 * c;
          const size_t row = (size_t)(ti.r0 + ti.m0 + 32 * c + lane);  // this lane's token row
          const int ax = ax_of(c);
          tc::wait_ld();
          if (c == nchunks - 1) {
            // this warp's reads of the accumulators are done
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty);
          }
          // the previous store from the staging tile has read it
          tc::bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            *reinterpret_cast<uint32_t*>(stg + i * 128 + (((lane >> 2) ^ (i & 7)) << 4) +
                                         (lane & 3) * 4) = v[i];
          __syncwarp();
          float f[32];  // token 32 c + lane: its features col0 .. col0 + 31
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 g = *reinterpret_cast<const float4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
            f[4 * j] = g.x;
            f[4 * j + 1] = g.y;
            f[4 * j + 2] = g.z;
            f[4 * j + 3] = g.w;
          }
          __syncwarp();  // every lane has read its row before the tile is reused
          if (a.yexp) {
            // fp16 y'' with y = y'' 2^s, s per token and 32 columns
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) m = max(m, __float_as_uint(f[i]) & 0x7fffffffu);
            if (lane < nv && m >= 0x7f800000u) bad = true;
            const int E = min(exp_of_bits(m), 127);
            const float sc = pow2f(kGroupTop - E);
            if (lane < nv)
              a.yexp[(size_t)(col0 >> 5) * a.yexp_rows + row] = (int16_t)(E - kGroupTop + p0 + 2 * ax);
            // row r of 32 fp16 (64 bytes): into the staging tile at r * 64,
            // 16-byte groups swizzled by (r >> 1) & 3 (the 64-byte TMA
            // swizzle), or straight to its row when the chunk is ragged
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.y) +
                                                  row * a.H + col0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 w4 = make_uint4(pack_f16x2(f[8 * j] * sc, f[8 * j + 1] * sc),
                                          pack_f16x2(f[8 * j + 2] * sc, f[8 * j + 3] * sc),
                                          pack_f16x2(f[8 * j + 4] * sc, f[8 * j + 5] * sc),
                                          pack_f16x2(f[8 * j + 6] * sc, f[8 * j + 7] * sc));
              if (nv >= 32)
                *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = w4;
              else if (lane < nv)
                dst[j] = w4;
            }
            if (nv >= 32) {
              tc::fence_proxy_async();
              __syncwarp();
              if (lane == 0) {  // bulk groups are per thread: always the same lane
                tc::tma_store_2d(&tm_y, col0, ti.r0 + ti.m0 + 32 * c, stg);
                tc::bulk_commit();
              }
              __syncwarp();
            }
          } else {
            // fp32 y = D 2^(pd + pg + pu + c + 2a), in two exact steps
            const int n = min(max(p0 + 2 * ax, -252), 252), h1 = n / 2;
            const float s1 = pow2f(h1), s2 = pow2f(n - h1);
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) +
                                                    row * a.H + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 w4 = make_float4(f[4 * j] * s1 * s2, f[4 * j + 1] * s1 * s2,
                                            f[4 * j + 2] * s1 * s2, f[4 * j + 3] * s1 * s2);
              if (nv >= 32)
                *reinterpret_cast<float4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = w4;
              else if (lane < nv)
                dst[j] = w4;
            }
            if (nv >= 32) {
              tc::fence_proxy_async();
              __syncwarp();
              if (lane == 0) {
                tc::tma_store_2d(&tm_y, col0, ti.r0 + ti.m0 + 32 * c, stg);
                tc::bulk_commit();
              }
              __syncwarp();
            }
          }
        }
      }
      if (lane == 0 && q == 0 && eh == 0) reinterpret_cast<volatile int*>(sh.prog)[kWarps + 2] = tl + 1;
    }
    if (bad && lane == 0) raise_status(a.status, MOE_DEV_NONFINITE);
    tc::bulk_wait_all();  // every bulk copy and TMA store of this warp is complete
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

// Per-expert token-tile prefix: tile_off[e] = sum_{e' < e} ceil(cnt_e' / 128),
// tile_off[E] = total.  One CTA, E <= 1024.
__global__ void __launch_bounds__(1024)
k_tile_offsets(const int32_t* __restrict__ expert_off, int E, int32_t* __restrict__ tile_off,
               int32_t* __restrict__ slot_done, int max_slots) {
  __shared__ int32_t wsum[32];
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid < E ? cdiv(expert_off[tid + 1] - expert_off[tid], BT) : 0;
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
  // the gate/up -> down completion counters of this call start at zero
  if (slot_done)
    for (int i = tid; i < max_slots; i += blockDim.x) slot_done[i] = 0;
}

// Activation rows normalised for the GEMM: a row of x becomes
//   a  = floor(log2 rms(x[t]))  (0 for an all-zero row),
//   x' = fp16(x[t] 2^-a),
// exact (bf16 has fewer mantissa bits than fp16; |x'| < 2 sqrt(K) <= 128,
// and only values under 2^-14 rms lose bits).  a depends on x[t] alone, so
// every copy of a token's row gets the same a.  An infinite or NaN activation
// raises MOE_DEV_NONFINITE.  K % 256 == 0, K <= 4096: one warp holds a row in
// registers, kGatherMaxPieces 16-byte pieces per lane at most.
constexpr int kGatherMaxPieces = 16;

// One warp: x[t] -> v (fp16 x', in place) and returns a (warp-uniform).
__device__ __forceinline__ int normalise_row(const uint16_t* __restrict__ x, int t, int K, int lane,
                                             uint4 (&v)[kGatherMaxPieces],
                                             int32_t* __restrict__ status) {
  const int np = K / 256;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * K);
  uint32_t m = 0;  // largest bf16 magnitude bits
#pragma unroll
  for (int i = 0; i < kGatherMaxPieces; ++i) {
    if (i < np) {
      v[i] = __ldg(src + lane + 32 * i);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if (m >= 0x7F80u && lane == 0) raise_status(status, MOE_DEV_NONFINITE);
  // sum of squares of x / 2^ea (no overflow: every term is below 4), in a
  // fixed order; lane 0's total decides a for the whole row
  const int ea = min(exp_of_bits(m << 16), 126);
  const float fa = pow2f(-ea);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kGatherMaxPieces; ++i) {
    if (i < np) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = bf16_lo(w[j]) * fa, hi = bf16_hi(w[j]) * fa;
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  int ae = 0;
  if (m != 0 && m < 0x7F80u) {
    const float rms = sqrtf(ss / (float)K);  // in [2^-6, 2]: a normal float
    ae = min(max(ea + (int)(__float_as_uint(rms) >> 23) - 127, -126), 126);
  }
  ae = __shfl_sync(0xffffffffu, ae, 0);
  const float f = pow2f(-ae);
#pragma unroll
  for (int i = 0; i < kGatherMaxPieces; ++i) {
    if (i < np) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      v[i] = make_uint4(pack_f16x2(bf16_lo(w[0]) * f, bf16_hi(w[0]) * f),
                        pack_f16x2(bf16_lo(w[1]) * f, bf16_hi(w[1]) * f),
                        pack_f16x2(bf16_lo(w[2]) * f, bf16_hi(w[2]) * f),
                        pack_f16x2(bf16_lo(w[3]) * f, bf16_hi(w[3]) * f));
    }
  }
  return ae;
}

__device__ __forceinline__ void store_row(uint16_t* __restrict__ dst_row, int K, int lane,
                                          const uint4 (&v)[kGatherMaxPieces]) {
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
  for (int i = 0; i < kGatherMaxPieces; ++i)
    if (i < K / 256) dst[lane + 32 * i] = v[i];
}

// Rows in expert order from the permutation's row -> token map: xp[p] = x'
// of token row_token[p], xexp[p] = its a, for the routed rows p <
// expert_off[E]; a token index outside [0, T) gives a zero row with a = 0.
// One warp per row.
__global__ void __launch_bounds__(256)
k_gather_rows(const uint16_t* __restrict__ x, int T, const int32_t* __restrict__ row_token,
              const int32_t* __restrict__ expert_off, int E, int P, int K,
              uint16_t* __restrict__ xp, int32_t* __restrict__ xexp,
              int32_t* __restrict__ status) {
  griddep_wait();
  griddep_trigger();
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (p >= min(P, expert_off[E])) return;  // warp-uniform
  const int t = row_token[p];
  uint4 v[kGatherMaxPieces];
  int a = 0;
  if (t < 0 || t >= T) {
#pragma unroll
    for (int i = 0; i < kGatherMaxPieces; ++i) v[i] = make_uint4(0, 0, 0, 0);
  } else {
    a = normalise_row(x, t, K, lane, v, status);
  }
  store_row(xp + (size_t)p * K, K, lane, v);
  if (lane == 0) xexp[p] = a;
}

// The same from the token side (the layer call, which has the permutation's
// token -> row map): one warp per token normalises x[t] once and writes it
// to each of its rows tok_slot_row[t k + j] >= 0 and, when xs is set, to
// row t of xs (the shared expert's rows, in token order).
__global__ void __launch_bounds__(256)
k_gather_tokens(const uint16_t* __restrict__ x, int T, int K,
                const int32_t* __restrict__ tok_slot_row, int k, uint16_t* __restrict__ xp,
                int32_t* __restrict__ xexp, uint16_t* __restrict__ xs,
                int32_t* __restrict__ sxexp, int32_t* __restrict__ status) {
  griddep_wait();
  griddep_trigger();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;  // warp-uniform
  uint4 v[kGatherMaxPieces];
  const int a = normalise_row(x, t, K, lane, v, status);
  const int my_row = lane < k ? tok_slot_row[(size_t)t * k + lane] : -1;
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, my_row, j);
    if (row < 0) continue;  // warp-uniform
    store_row(xp + (size_t)row * K, K, lane, v);
    if (lane == 0) xexp[row] = a;
  }
  if (xs) {
    store_row(xs + (size_t)t * K, K, lane, v);
    if (lane == 0) sxexp[t] = a;
  }
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

// 2-D map over a row-major matrix [rows, cols] of esize-byte elements.
cudaError_t make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, int esize, const void* base,
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

namespace {
// 2-D map over a stack of code matrices [rows_total, K] (uint8, row-major):
// box = 64 bytes of K x 128 rows, 64-byte swizzle (conflict-free reads of a
// row's four 16-byte chunks by the lanes that own consecutive rows).
cudaError_t code_map(CUtensorMap* map, const uint8_t* codes, long long rows_total, int K) {
  return make_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes, rows_total, K, BK, BW, 64);
}
}  // namespace

bool expert_gemm_tc_ok(int H, int I) {
  // K / 128 <= 32 block scales per weight row block (one per decoder lane)
  return H % 256 == 0 && I % 128 == 0 && H >= 256 && I >= 128 && H <= 32 * kScaleBlock &&
         I <= 32 * kScaleBlock;
}

cudaError_t launch_expert_gemm_tc(const uint16_t* x, int T, const int32_t* expert_off,
                                  const int32_t* row_token, uint16_t* x_perm, int32_t* xexp,
                                  int E, int P, const moe_fp8_ffn& w, int H, int I,
                                  int32_t* tile_off, int32_t* slot_done, uint16_t* hid, void* y,
                                  int16_t* yexp, int yexp_rows, int32_t* status, cudaStream_t s,
                                  bool pdl, bool tile_off_ready, const GemmGather& gather) {
  static_assert(BT == kGemmTokenTile, "token tile of the permutation's tile prefix");
  if (!x_perm || !xexp || H > kGatherMaxPieces * 256) return cudaErrorInvalidValue;
  cudaError_t err;
  if (!slot_done) return cudaErrorInvalidValue;
  if ((err = ensure_smem((const void*)k_expert_ffn_ws<kBoth>, SMEM_WS)) != cudaSuccess ||
      (err = ensure_smem((const void*)k_expert_ffn_ws<kGateUp>, SMEM_WS)) != cudaSuccess ||
      (err = ensure_smem((const void*)k_expert_ffn_ws<kDown>, SMEM_WS)) != cudaSuccess)
    return err;
  CUtensorMap gmap, umap, dmap, xmap, hmap, ymap;
  if ((err = code_map(&gmap, w.gate.codes, (long long)E * I, H)) != cudaSuccess) return err;
  if ((err = code_map(&umap, w.up.codes, (long long)E * I, H)) != cudaSuccess) return err;
  if ((err = code_map(&dmap, w.down.codes, (long long)E * H, I)) != cudaSuccess) return err;
  // Normalised activations in expert order [P, H] fp16 and hid [P, I] fp16:
  // 64 columns x 128 rows per box, 128-byte swizzled (the K-major operand
  // layout of the MMA)
  if ((err = make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x_perm, P, H, BK, BT,
                                128)) != cudaSuccess)
    return err;
  if ((err = make_tensor_map_2d(&hmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hid, P, I, BK, BT, 128)) !=
      cudaSuccess)
    return err;
  // y [P, H], written by the down epilogue: 32 columns x 32 rows; fp32 rows of
  // 128 bytes (128-byte swizzle) or fp16 rows of 64 bytes (64-byte swizzle)
  if ((err = yexp ? make_tensor_map_2d(&ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, y, P, H, 32, 32,
                                       64)
                  : make_tensor_map_2d(&ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, P, H, 32, 32,
                                       128)) != cudaSuccess)
    return err;
  // Tile offsets first, then the gather: the GEMMs' warps other than the
  // token warp read the offsets without waiting for their previous kernel.
  // Host bound on the tile count: each expert adds at most one partial tile.
  const int max_ttiles = cdiv(P, BT) + min(E, P);
  if (!tile_off_ready) {
    err = launch_k(k_tile_offsets, dim3(1), dim3(1024), 0, s, pdl, expert_off, E, tile_off,
                   slot_done, max_ttiles);
    if (err != cudaSuccess) return err;
  }
  bool prev_wrote_offsets = !tile_off_ready;  // the GEMM's previous kernel
  if (gather.tok_slot_row) {
    err = launch_k(k_gather_tokens, dim3(cdiv(T, 8)), dim3(256), 0, s, pdl, x, T, H,
                   gather.tok_slot_row, gather.k, x_perm, xexp, gather.shared_rows,
                   gather.shared_xexp, status);
    prev_wrote_offsets = false;
  } else if (!gather.rows_ready) {
    err = launch_k(k_gather_rows, dim3(cdiv(P, 8)), dim3(256), 0, s, pdl, x, T, row_token,
                   expert_off, E, P, H, x_perm, xexp, status);
    prev_wrote_offsets = false;
  }
  if (err != cudaSuccess) return err;
  int log2H = 0;
  while ((2 << log2H) <= H) ++log2H;
  // Diagnostics (read on every call): a shorter limit for the bounded waits
  // (MOE_FP8_WAIT_LIMIT_US), and down tiles that wait for one more
  // completed gate/up tile per token tile than exist, so that its wait runs
  // out (MOE_FP8_TEST_STALL=down; the failure-path test).
  uint64_t wait_ns = 0;
  if (const char* lim = getenv("MOE_FP8_WAIT_LIMIT_US")) {
    const long long us = atoll(lim);
    if (us > 0) wait_ns = (uint64_t)us * 1000ull;
  }
  const char* stall = getenv("MOE_FP8_TEST_STALL");
  const bool stall_down = stall && strcmp(stall, "down") == 0;
  FfnArgs f{};
  f.expert_off = expert_off;
  f.tile_off = tile_off;
  f.E = E;
  f.H = H;
  f.I = I;
  f.gs = w.gate.scales;
  f.us = w.up.scales;
  f.ds = w.down.scales;
  f.hid = hid;
  f.y = y;
  // every warp waits when the previous kernel wrote the tile offsets
  f.all_wait = prev_wrote_offsets ? 1 : 0;
  f.slot_done = slot_done;
  f.slot_need = (I / BW) * kEpiWarps + (stall_down ? 1 : 0);
  f.status = status;
  f.xexp = xexp;
  f.hid_shift = log2H + 4;
  f.yexp = yexp;
  f.yexp_rows = yexp_rows;
  f.wait_ns = wait_ns;
  // One launch for both GEMMs when gate/up tiles fill every SM and the list
  // is short (at most 16 tiles per SM, bounded from the shapes): measured,
  // it saves the second launch's start on every SM (decode T = 32 / 64 / 96
  // of the Qwen3 shape: -7.6 / -3.8 / -7 us).  With more tiles per SM the
  // single kernel's larger code costs more than that, and a grid that
  // gate/up alone does not fill (the shared expert) gains nothing from it,
  // so gate/up and down launch apart.  MOE_FP8_GEMM_LAUNCHES=1 or =2 forces
  // either (diagnostics and tests).
  const int nsm = num_sms();
  const int gu_tiles = max_ttiles * (I / BW), dn_tiles = max_ttiles * (H / (2 * BW));
  bool one = gu_tiles >= nsm && gu_tiles + dn_tiles <= 16 * nsm;
  if (const char* v = getenv("MOE_FP8_GEMM_LAUNCHES")) {
    if (strcmp(v, "1") == 0) one = true;
    if (strcmp(v, "2") == 0) one = false;
  }
  if (one)
    return launch_k(k_expert_ffn_ws<kBoth>, dim3(min(nsm, gu_tiles + dn_tiles)), dim3(kThreadsWS),
                    (size_t)SMEM_WS, s, pdl, gmap, umap, dmap, xmap, hmap, ymap, f);
  err = launch_k(k_expert_ffn_ws<kGateUp>, dim3(min(nsm, gu_tiles)), dim3(kThreadsWS),
                 (size_t)SMEM_WS, s, pdl, gmap, umap, dmap, xmap, hmap, ymap, f);
  if (err != cudaSuccess) return err;
  f.all_wait = 0;  // the gate/up launch is the previous kernel: waited for per token tile
  return launch_k(k_expert_ffn_ws<kDown>, dim3(min(nsm, dn_tiles)), dim3(kThreadsWS),
                  (size_t)SMEM_WS, s, pdl, gmap, umap, dmap, xmap, hmap, ymap, f);
}

}  // namespace moe
