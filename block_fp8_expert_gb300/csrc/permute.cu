// Permutation of the T*k (token, slot) pairs into expert-contiguous rows:
// a stable counting sort of the flattened pair index q = t*k + j by expert.
// Inside one expert, ascending q is ascending t (a token never picks the same
// expert twice), which is the order the layer's rows use.
//
// Three launches, no atomics that decide an order:
//   count   per block of kPermBlock pairs: per-expert counts and each pair's
//           rank among the block's pairs of the same expert (warp match +
//           per-warp prefix);
//   scan    one CTA: per-expert totals, exclusive prefix over blocks, the
//           expert offsets (exclusive scan over experts) and the list of
//           experts that received rows;
//   scatter row = off[e] + block prefix + rank.
#include "moe_internal.h"

namespace moe {

constexpr int kPermBlock = 256;  // pairs per count/scatter CTA (8 warps)
static_assert(kPermBlock == kPermPairsPerBlock, "scratch sizing assumes 256 pairs per block");

__global__ void __launch_bounds__(kPermBlock)
k_perm_count(const int32_t* __restrict__ topk_idx, int P, int E,
             int32_t* __restrict__ rank, int32_t* __restrict__ block_cnt,
             int32_t* __restrict__ status) {
  extern __shared__ int32_t cnt_w[];  // [8][E]
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 8 * E; i += kPermBlock) cnt_w[i] = 0;
  __syncthreads();
  const int q = blockIdx.x * kPermBlock + tid;
  int e = -2;  // -2: past the end, -1: invalid index
  if (q < P) {
    e = topk_idx[q];
    if (e < 0 || e >= E) {
      raise_status(status, MOE_DEV_BAD_EXPERT_INDEX);
      e = -1;
    }
  }
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank_w == 0) cnt_w[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = tid; x < E; x += kPermBlock) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = cnt_w[w * E + x];
      cnt_w[w * E + x] = run;
      run += c;
    }
    block_cnt[(size_t)blockIdx.x * E + x] = run;
  }
  __syncthreads();
  if (q < P) rank[q] = e >= 0 ? cnt_w[warp * E + e] + rank_w : -1;
}

// One CTA of 1024 threads; E <= 1024.  Each expert's column of block counts
// is split among G = 1024 / E threads (contiguous runs of blocks): each sums
// its run (independent loads), the runs' sums are prefixed in shared memory,
// and each thread writes its run's block bases.  Then the scan over experts
// gives the offsets, the active list and, when tile_off is set, the
// tensor-core GEMM's token-tile prefix (tile_off[e] = sum over e' < e of
// ceil(count / kGemmTokenTile)); counters[0, n_counters) are zeroed.
__global__ void __launch_bounds__(1024)
k_perm_scan(const int32_t* __restrict__ block_cnt, int nblocks, int E,
            int32_t* __restrict__ block_base, int32_t* __restrict__ expert_off,
            int32_t* __restrict__ active, int32_t* __restrict__ tile_off,
            int32_t* __restrict__ counters, int n_counters) {
  __shared__ int32_t part[1024];
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t warp_act[32];
  __shared__ int32_t warp_til[32];
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = min(32, 1024 / E);  // threads per expert
  const int e = tid % E, g = tid / E;
  const bool mine = g < G;
  const int b0 = mine ? (int)((long long)g * nblocks / G) : 0;
  const int b1 = mine ? (int)((long long)(g + 1) * nblocks / G) : 0;
  int run = 0;
#pragma unroll 8
  for (int b = b0; b < b1; ++b) run += block_cnt[(size_t)b * E + e];
  part[tid] = run;
  __syncthreads();
  int before = 0, total = 0;
  if (mine)
    for (int h = 0; h < G; ++h) {
      const int v = part[h * E + e];
      if (h < g) before += v;
      total += v;
    }
  run = before;
#pragma unroll 8
  for (int b = b0; b < b1; ++b) {
    const int c = block_cnt[(size_t)b * E + e];
    block_base[(size_t)b * E + e] = run;
    run += c;
  }
  if (counters)
    for (int i = tid; i < n_counters; i += 1024) counters[i] = 0;
  // exclusive scans over experts (threads tid < E: expert tid) of the totals,
  // of the non-empty flags and of the token-tile counts
  if (tid >= E) total = 0;
  const int ntile = (total + kGemmTokenTile - 1) / kGemmTokenTile;
  int incl = total, act = total > 0 ? 1 : 0, til = ntile;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int w = __shfl_up_sync(0xffffffffu, act, o);
    const int u = __shfl_up_sync(0xffffffffu, til, o);
    if (lane >= o) {
      incl += v;
      act += w;
      til += u;
    }
  }
  if (lane == 31) {
    warp_sum[warp] = incl;
    warp_act[warp] = act;
    warp_til[warp] = til;
  }
  __syncthreads();
  if (warp == 0) {
    int sv = warp_sum[lane], av = warp_act[lane], tv = warp_til[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, sv, o);
      const int w = __shfl_up_sync(0xffffffffu, av, o);
      const int u = __shfl_up_sync(0xffffffffu, tv, o);
      if (lane >= o) {
        sv += v;
        av += w;
        tv += u;
      }
    }
    warp_sum[lane] = sv;  // inclusive over warps
    warp_act[lane] = av;
    warp_til[lane] = tv;
  }
  __syncthreads();
  const int wbefore = warp ? warp_sum[warp - 1] : 0;
  const int abefore = warp ? warp_act[warp - 1] : 0;
  const int tbefore = warp ? warp_til[warp - 1] : 0;
  if (tid < E) {
    expert_off[tid] = wbefore + incl - total;
    if (total > 0) active[1 + abefore + act - 1] = tid;
    if (tile_off) tile_off[tid] = tbefore + til - ntile;
  }
  if (tid == E - 1) {
    expert_off[E] = wbefore + incl;
    active[0] = abefore + act;
    if (tile_off) tile_off[E] = tbefore + til;
  }
}

__global__ void __launch_bounds__(kPermBlock)
k_perm_scatter(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ rank,
               const int32_t* __restrict__ block_base, const int32_t* __restrict__ expert_off,
               int P, int E, int k, int32_t* __restrict__ row_token,
               int32_t* __restrict__ tok_slot_row, int32_t* __restrict__ row_pair) {
  griddep_wait();
  griddep_trigger();
  const int q = blockIdx.x * kPermBlock + threadIdx.x;
  if (q >= P) return;
  const int r = rank[q];
  if (r < 0) {
    tok_slot_row[q] = -1;
    return;
  }
  const int e = topk_idx[q];
  const int row = expert_off[e] + block_base[(size_t)blockIdx.x * E + e] + r;
  row_token[row] = q / k;
  tok_slot_row[q] = row;
  if (row_pair) row_pair[row] = q;
}

// Active-expert list from offsets alone (for callers of the expert FFN that
// did not run the permutation here).  One CTA; E <= 1024.
__global__ void __launch_bounds__(1024)
k_active_from_offsets(const int32_t* __restrict__ expert_off, int E,
                      int32_t* __restrict__ active, int32_t* __restrict__ status) {
  __shared__ int32_t warp_act[32];
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kStatusWords && status) status[tid] = 0;  // first kernel of an expert-FFN call
  const int ne = (tid < E && expert_off[tid + 1] > expert_off[tid]) ? 1 : 0;
  int act = ne;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, act, o);
    if (lane >= o) act += a;
  }
  if (lane == 31) warp_act[warp] = act;
  __syncthreads();
  if (warp == 0) {
    int a = warp_act[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, a, o);
      if (lane >= o) a += w;
    }
    warp_act[lane] = a;
  }
  __syncthreads();
  const int before = warp ? warp_act[warp - 1] : 0;
  if (ne) active[1 + before + act - 1] = tid;
  if (tid == 1023) active[0] = warp_act[31];
}

cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, int32_t* rank,
                           int32_t* block_cnt, int32_t* block_base, int32_t* expert_off,
                           int32_t* row_token, int32_t* tok_slot_row, int32_t* row_pair,
                           int32_t* active, int32_t* status, cudaStream_t s, bool pdl,
                           int32_t* tile_off, int32_t* counters, int n_counters) {
  const int P = T * k;
  const int nb = cdiv(P, kPermBlock);
  cudaError_t e;
  if (nb > 0) {
    const size_t smem = sizeof(int32_t) * 8 * E;
    e = launch_k(k_perm_count, dim3(nb), dim3(kPermBlock), smem, s, pdl, topk_idx, P, E, rank,
                 block_cnt, status);
    if (e != cudaSuccess) return e;
  }
  e = launch_k(k_perm_scan, dim3(1), dim3(1024), 0, s, pdl, (const int32_t*)block_cnt, nb, E,
               block_base, expert_off, active, tile_off, counters, n_counters);
  if (e != cudaSuccess || nb == 0) return e;
  return launch_k(k_perm_scatter, dim3(nb), dim3(kPermBlock), 0, s, pdl, topk_idx,
                  (const int32_t*)rank, (const int32_t*)block_base, (const int32_t*)expert_off, P,
                  E, k, row_token, tok_slot_row, row_pair);
}

cudaError_t launch_active_from_offsets(const int32_t* expert_off, int E, int32_t* active,
                                       int32_t* status, cudaStream_t s, bool pdl) {
  return launch_k(k_active_from_offsets, dim3(1), dim3(1024), 0, s, pdl, expert_off, E, active,
                  status);
}

}  // namespace moe
