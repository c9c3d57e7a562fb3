// Router: logits l = x Wr^T (+ b), then per token the top-k experts and their
// renormalised weights (colizig README, model table: experts with top-k
// routing).  The renormalised weight p_j / sum_sel p equals the softmax over
// the k selected logits, because the full softmax's normaliser cancels; the
// kernels compute it that way and never form the E probabilities.
#include <climits>

#include "moe_internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// logits on the tensor cores.  fp32 router weights are split into three bf16
// parts (w = hi + mid + lo to within 2^-24 |w|); bf16 activations are exact,
// so three bf16 MMAs accumulating in fp32 give fp32-accurate logits.
// grid (ceil(E/16), KS, ceil(T/(8*NT))): a CTA owns 16 experts, one of KS
// slices of K = H and 8*NT tokens; its 4 warps take the slice's 64-column
// chunks round-robin.  Partial sums go to part[ks][t][e]; the top-k kernels
// add the KS slices in a fixed order (deterministic).
// When xn is set, the CTAs of expert tile 0 also write the activations for
// the streamed expert kernels: xn = fp16(x 2^(14 - e)) and xe = e, one e per
// token and 64 columns (the largest magnitude of the 64 lands in
// [2^14, 2^15); exact, see bf16x16_to_f16_norm).
// ---------------------------------------------------------------------------
constexpr int kRouteWarps = 4;
constexpr int kMaxKSlices = 8;  // K-slices of the router logits (route_kslices)

// One 64-column chunk of the router logits for one warp: lane (g, c) holds
// experts ea = e0 + g and eb = e0 + g + 8, columns kk .. kk + 15 of the
// chunk (kk = k0 + 16 c), and the activations of tokens trow[nt].
template <int NT>
struct RouterChunk {
  float wa[16], wb[16];
  uint4 xa[NT][2];
  __device__ __forceinline__ void load(const uint16_t* __restrict__ x,
                                       const float* __restrict__ Wr, int H, int E, int ea,
                                       int eb, const int (&trow)[NT], int kk) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 fa = ea < E ? __ldg(reinterpret_cast<const float4*>(Wr + (size_t)ea * H + kk) + v)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 fb = eb < E ? __ldg(reinterpret_cast<const float4*>(Wr + (size_t)eb * H + kk) + v)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      wa[4 * v + 0] = fa.x; wa[4 * v + 1] = fa.y; wa[4 * v + 2] = fa.z; wa[4 * v + 3] = fa.w;
      wb[4 * v + 0] = fb.x; wb[4 * v + 1] = fb.y; wb[4 * v + 2] = fb.z; wb[4 * v + 3] = fb.w;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (trow[nt] >= 0) {
        const uint16_t* xp = x + (size_t)trow[nt] * H + kk;
        xa[nt][0] = ldg16(xp);
        xa[nt][1] = ldg16(xp + 8);
      } else {
        xa[nt][0] = xa[nt][1] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  // the streamed kernels' activations: the quad of lanes 4g .. 4g + 3 holds
  // token trow's 64 columns k0 .. k0 + 63 (all lanes take part in the quad's
  // shuffles)
  __device__ __forceinline__ void write_xn(uint16_t* __restrict__ xn, int8_t* __restrict__ xe,
                                           int H, const int (&trow)[NT], int k0, int c) const {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint4 v[2] = {xa[nt][0], xa[nt][1]};
      bool bad = false;  // a non-finite x shows in the expert kernels' results
      const int ex = bf16x16_to_f16_norm(v, bad);
      if (trow[nt] >= 0) {
        uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)trow[nt] * H + k0 + 16 * c);
        dst[0] = v[0];
        dst[1] = v[1];
        if (c == 0) xe[(size_t)trow[nt] * (H / 64) + k0 / 64] = (int8_t)min(ex, 127);
      }
    }
  }
  // acc += the chunk's products: the three bf16 parts of Wr, smallest first
  __device__ __forceinline__ void mma(float (&acc)[NT][4]) const {
    // bf16x2 registers of the three parts, element pairs (2m, 2m+1)
    uint32_t ah[8], am[8], al[8], bh[8], bm[8], bl[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t h0, m0, l0, h1, m1, l1;
      split3_bf16(wa[2 * m], h0, m0, l0);
      split3_bf16(wa[2 * m + 1], h1, m1, l1);
      ah[m] = h0 | (h1 << 16); am[m] = m0 | (m1 << 16); al[m] = l0 | (l1 << 16);
      split3_bf16(wb[2 * m], h0, m0, l0);
      split3_bf16(wb[2 * m + 1], h1, m1, l1);
      bh[m] = h0 | (h1 << 16); bm[m] = m0 | (m1 << 16); bl[m] = l0 | (l1 << 16);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t xr[8] = {xa[nt][0].x, xa[nt][0].y, xa[nt][0].z, xa[nt][0].w,
                              xa[nt][1].x, xa[nt][1].y, xa[nt][1].z, xa[nt][1].w};
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint32_t b[2] = {xr[2 * st], xr[2 * st + 1]};
        const uint32_t A0[4] = {al[2 * st], bl[2 * st], al[2 * st + 1], bl[2 * st + 1]};
        const uint32_t A1[4] = {am[2 * st], bm[2 * st], am[2 * st + 1], bm[2 * st + 1]};
        const uint32_t A2[4] = {ah[2 * st], bh[2 * st], ah[2 * st + 1], bh[2 * st + 1]};
        mma_bf16_16x8x16(acc[nt], A0, b);
        mma_bf16_16x8x16(acc[nt], A1, b);
        mma_bf16_16x8x16(acc[nt], A2, b);
      }
    }
  }
};

template <int NT>
__global__ void __launch_bounds__(kRouteWarps * 32)
k_router_mma(const uint16_t* __restrict__ x, const float* __restrict__ Wr, int T, int H, int E,
             int kslice, float* __restrict__ part, uint16_t* __restrict__ xn,
             int8_t* __restrict__ xe, int32_t* __restrict__ status) {
  __shared__ float red[kRouteWarps][NT][4][32];
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  // The router runs first in a layer call: it clears the status words that
  // later kernels of the call may raise.
  if (status && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && tid < kStatusWords)
    status[tid] = 0;
  const int e0 = blockIdx.x * 16;
  const int t0 = blockIdx.z * NT * 8;
  const int kbeg = blockIdx.y * kslice, kend = min(H, kbeg + kslice);
  const int ea = e0 + g, eb = e0 + g + 8;
  const bool write_xn = xn != nullptr && blockIdx.x == 0;  // CTA-uniform
  int trow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) trow[nt] = (t0 + nt * 8 + g < T) ? t0 + nt * 8 + g : -1;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;

  // up to kAhead chunks' loads in flight (4 for one 8-token group, fewer
  // for more tokens: their activations take the registers), then the
  // chunks' MMAs in ascending k0, as one chunk at a time would
  constexpr int kAhead = NT == 1 ? 4 : NT == 2 ? 2 : 1;
  for (int k0 = kbeg + warp * 64; k0 < kend; k0 += kAhead * kRouteWarps * 64) {
    RouterChunk<NT> ch[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int ku = k0 + u * kRouteWarps * 64;
      if (ku < kend) ch[u].load(x, Wr, H, E, ea, eb, trow, ku + 16 * c);
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int ku = k0 + u * kRouteWarps * 64;
      if (ku < kend) {
        if (write_xn) ch[u].write_xn(xn, xe, H, trow, ku, c);
        ch[u].mma(acc);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int q = 0; q < 4; ++q) red[warp][nt][q][lane] = acc[nt][q];
  __syncthreads();
  for (int o = tid; o < NT * 128; o += kRouteWarps * 32) {
    const int nt = o >> 7, q = (o >> 5) & 3, L = o & 31;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) v += red[w][nt][q][L];
    const int e = e0 + (L >> 2) + 8 * (q >> 1);
    const int t = t0 + nt * 8 + 2 * (L & 3) + (q & 1);
    if (e < E && t < T) part[((size_t)blockIdx.y * T + t) * E + e] = v;
  }
}

// ---------------------------------------------------------------------------
// top-k + renormalisation of one token by one warp: EPL logits per lane.
// Lane j < k ends up holding slot j (expert index and weight).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int EPL>
__device__ __forceinline__ void warp_topk(const float* __restrict__ part, int KS,
                                          const float* __restrict__ bias, int T, int E, int k,
                                          int t, int lane, int& my_idx, float& my_w) {
  // All partial logits of this lane first (independent loads), then the sums
  // in slice order.
  float v[EPL];
  if (EPL * kMaxKSlices <= 32) {
    // every load in flight at once, then the sums in slice order
    float p[kMaxKSlices][EPL];
#pragma unroll
    for (int ks = 0; ks < kMaxKSlices; ++ks)
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        p[ks][i] = (ks < KS && e < E) ? __ldcg(&part[((size_t)ks * T + t) * E + e]) : 0.f;
      }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      v[i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kMaxKSlices; ++ks) v[i] += p[ks][i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) v[i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kMaxKSlices; ++ks) {
      if (ks < KS) {
        float p[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int e = lane + 32 * i;
          p[i] = e < E ? __ldcg(&part[((size_t)ks * T + t) * E + e]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) v[i] += p[i];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? (bias ? v[i] + bias[e] : v[i]) : -INFINITY;
  }
  // Order-preserving integer keys (exact: -0 is first folded into +0; the
  // map is its own inverse, so a key gives back its logit).  Each lane keeps
  // the best of its not-yet-taken experts (largest key, lowest index); a
  // round is two redux.sync reductions over the lanes' heads (largest key,
  // then the lowest expert index holding it), and only the winning lane
  // rescans its own experts.  The round results are warp-uniform, so lane j
  // keeps the j-th selection without a shuffle.
  int key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int b = __float_as_int(v[i] + 0.0f);
    key[i] = (lane + 32 * i < E) ? (b ^ ((b >> 31) & 0x7FFFFFFF)) : INT_MIN;
  }
  uint32_t taken = 0;
  int hk = INT_MIN, he = 0x7fffffff, hs = 0;
  auto rescan = [&]() {
    hk = INT_MIN;
    he = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && key[i] > hk) {  // first (lowest e) of equal keys
        hk = key[i];
        he = e;
        hs = i;
      }
    }
  };
  rescan();
  int my_key = INT_MIN;
  my_idx = 0;
  for (int j = 0; j < k; ++j) {
    const int wk = __reduce_max_sync(0xffffffffu, hk);
    const int wi = __reduce_min_sync(0xffffffffu, hk == wk ? he : 0x7fffffff);
    if (lane == j) {
      my_key = wk;
      my_idx = wi;
    }
    if (he == wi) {
      taken |= 1u << hs;
      rescan();
    }
  }
  const float my_val = __int_as_float(my_key ^ ((my_key >> 31) & 0x7FFFFFFF));
  const float vmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < k ? expf(my_val - vmax) : 0.f;
  float s = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  my_w = ex / s;
}

// Gated shared expert: sigmoid(x[t] . g) for token t by one warp (H % 8 ==
// 0), fp32 products summed per lane in order, then over the lanes; lane 0's
// value is the result (returned in every lane).
__device__ __forceinline__ float warp_shared_gate(const uint16_t* __restrict__ x,
                                                  const float* __restrict__ g, int H, int t,
                                                  int lane) {
  float s = 0.f;
  for (int h = lane * 8; h < H; h += 256) {
    const uint4 v = ldg16(x + (size_t)t * H + h);
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(g + h));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(g + h + 4));
    s = fmaf(bf16_lo(v.x), g0.x, s);
    s = fmaf(bf16_hi(v.x), g0.y, s);
    s = fmaf(bf16_lo(v.y), g0.z, s);
    s = fmaf(bf16_hi(v.y), g0.w, s);
    s = fmaf(bf16_lo(v.z), g1.x, s);
    s = fmaf(bf16_hi(v.z), g1.y, s);
    s = fmaf(bf16_lo(v.w), g1.z, s);
    s = fmaf(bf16_hi(v.w), g1.w, s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  s = __shfl_sync(0xffffffffu, s, 0);
  return 1.f / (1.f + expf(-s));
}

// The gate inputs of the layer call's top-k kernels (sgate == NULL: none).
struct SharedGate {
  const uint16_t* x = nullptr;
  const float* g = nullptr;
  int H = 0;
  float* sgate = nullptr;  // [T] out
};

template <int EPL>
__global__ void __launch_bounds__(256)
k_router_topk(const float* __restrict__ part, int KS, const float* __restrict__ bias, int T,
              int E, int k, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
              const SharedGate sg) {
  griddep_wait();
  griddep_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  int idx;
  float w;
  warp_topk<EPL>(part, KS, bias, T, E, k, t, lane, idx, w);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = idx;
    topk_w[(size_t)t * k + lane] = w;
  }
  if (sg.sgate) {
    const float gt = warp_shared_gate(sg.x, sg.g, sg.H, t, lane);
    if (lane == 0) sg.sgate[t] = gt;
  }
}

// ---------------------------------------------------------------------------
// Small batches: top-k and the whole permutation in ONE CTA of 1024 threads
// (T*k <= kSmallPairs, E <= 1024), replacing four launches.  Same results as
// k_router_topk followed by the three permutation kernels: pairs are ranked
// inside each expert in ascending pair index q = t*k + j (ascending t).
//   1. warp per token: top-k, written to global and to shared memory;
//   2. per-expert counts (order-free shared atomics), exclusive scan ->
//      expert_off and the active-expert list;
//   3. rounds of 1024 pairs: warp match ranks, per-warp counts, prefix over
//      warps, row = off[e] + pairs of e in earlier rounds + prefix + rank.
// Also writes the shared expert's identity permutation when asked, and
// row_pair[row] = q (the pair of each permuted row).
// ---------------------------------------------------------------------------
constexpr int kSmallPairs = 4096;
// From this many tokens on, top-k runs as its own multi-CTA launch before the
// one-CTA permutation (below it, the single fused CTA is faster).
constexpr int kSplitTopkTokens = 16;

size_t small_route_smem(int E) {
  return sizeof(int32_t) * (kSmallPairs + 3 * 1024 + 1 + 96) + sizeof(uint16_t) * 32 * (size_t)E;
}

template <int EPL>
__global__ void __launch_bounds__(1024, 1)
k_topk_permute_small(const float* __restrict__ part, int KS, const float* __restrict__ bias,
                     int T, int E, int k, int32_t* __restrict__ topk_idx,
                     float* __restrict__ topk_w, int32_t* __restrict__ expert_off,
                     int32_t* __restrict__ row_token, int32_t* __restrict__ tok_slot_row,
                     int32_t* __restrict__ row_pair, int32_t* __restrict__ active,
                     int32_t* __restrict__ sh_off, int32_t* __restrict__ sh_rows,
                     int32_t* __restrict__ sh_active, int32_t* __restrict__ tile_off,
                     int32_t* __restrict__ counters, int n_counters, const SharedGate sg) {
  extern __shared__ int32_t sm[];
  int32_t* s_idx = sm;                   // [kSmallPairs] expert of pair q
  int32_t* s_cnt = s_idx + kSmallPairs;  // [1024] counts, then rows taken so far
  int32_t* s_tot = s_cnt + 1024;         // [1024] this round's count per expert
  int32_t* s_off = s_tot + 1024;         // [1025] expert offsets
  int32_t* s_wsum = s_off + 1025;        // [32]
  int32_t* s_wact = s_wsum + 32;         // [32]
  int32_t* s_wtil = s_wact + 32;         // [32]
  uint16_t* s_cw = reinterpret_cast<uint16_t*>(s_wtil + 32);  // [32][E] per-warp counts
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = T * k;

  // 1. top-k (EPL = 0: already selected by k_router_topk, read it back)
  if constexpr (EPL == 0) {
    for (int q = tid; q < P; q += 1024) s_idx[q] = topk_idx[q];
  } else {
    for (int t = warp; t < T; t += 32) {
      int idx;
      float w;
      warp_topk<EPL>(part, KS, bias, T, E, k, t, lane, idx, w);
      if (lane < k) {
        topk_idx[(size_t)t * k + lane] = idx;
        topk_w[(size_t)t * k + lane] = w;
        s_idx[t * k + lane] = idx;
      }
      if (sg.sgate) {
        const float gt = warp_shared_gate(sg.x, sg.g, sg.H, t, lane);
        if (lane == 0) sg.sgate[t] = gt;
      }
    }
  }
  s_cnt[tid] = 0;
  if (sh_rows) {  // shared expert: every token, in order
    for (int t = tid; t < T; t += 1024) sh_rows[t] = t;
    if (tid == 0) {
      sh_off[0] = 0;
      sh_off[1] = T;
      sh_active[0] = T > 0 ? 1 : 0;
      sh_active[1] = 0;
    }
  }
  __syncthreads();
  // 2. counts, offsets, active list
  for (int q = tid; q < P; q += 1024) atomicAdd(&s_cnt[s_idx[q]], 1);
  __syncthreads();
  // (and, for the tensor-core GEMM, the token-tile prefix: tile_off[e] =
  // sum over e' < e of ceil(count / kGemmTokenTile))
  const int c = tid < E ? s_cnt[tid] : 0;
  const int nt = cdiv(c, kGemmTokenTile);
  int incl = c, act = c > 0 ? 1 : 0, tin = nt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int a = __shfl_up_sync(0xffffffffu, act, o);
    const int b = __shfl_up_sync(0xffffffffu, tin, o);
    if (lane >= o) {
      incl += v;
      act += a;
      tin += b;
    }
  }
  if (lane == 31) {
    s_wsum[warp] = incl;
    s_wact[warp] = act;
    s_wtil[warp] = tin;
  }
  __syncthreads();
  if (warp == 0) {
    int s = s_wsum[lane], a = s_wact[lane], b = s_wtil[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, s, o);
      const int w = __shfl_up_sync(0xffffffffu, a, o);
      const int u = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) {
        s += v;
        a += w;
        b += u;
      }
    }
    s_wsum[lane] = s;
    s_wact[lane] = a;
    s_wtil[lane] = b;
  }
  __syncthreads();
  {
    const int before = warp ? s_wsum[warp - 1] : 0;
    const int before_a = warp ? s_wact[warp - 1] : 0;
    const int before_t = warp ? s_wtil[warp - 1] : 0;
    if (tid < E) {
      const int o = before + incl - c;
      s_off[tid] = o;
      expert_off[tid] = o;
      if (c > 0) active[1 + before_a + act - 1] = tid;
      if (tile_off) tile_off[tid] = before_t + tin - nt;
    }
    if (tid == E - 1) {
      s_off[E] = before + incl;
      expert_off[E] = before + incl;
      active[0] = before_a + act;
      if (tile_off) tile_off[E] = before_t + tin;
    }
  }
  // the expert kernels' counters of this call (the GEMM's gate/up -> down
  // completion counters, or the fused combine's tickets) start at zero
  if (counters)
    for (int i = tid; i < n_counters; i += 1024) counters[i] = 0;
  __syncthreads();
  s_cnt[tid] = 0;  // rows of each expert placed by earlier rounds
  // 3. rank rounds of 1024 pairs
  for (int r0 = 0; r0 < P; r0 += 1024) {
    const int q = r0 + tid;
    const int e = q < P ? s_idx[q] : -1;
    for (int i = tid; i < 32 * E; i += 1024) s_cw[i] = 0;
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank_w == 0) s_cw[warp * E + e] = (uint16_t)__popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += 1024) {  // exclusive prefix over the 32 warps
      int run = 0;
      for (int w = 0; w < 32; ++w) {
        const int cw = s_cw[w * E + x];
        s_cw[w * E + x] = (uint16_t)run;
        run += cw;
      }
      s_tot[x] = run;
    }
    __syncthreads();
    if (e >= 0) {
      const int row = s_off[e] + s_cnt[e] + s_cw[warp * E + e] + rank_w;
      row_token[row] = q / k;
      tok_slot_row[q] = row;
      if (row_pair) row_pair[row] = q;
    }
    __syncthreads();
    for (int x = tid; x < E; x += 1024) s_cnt[x] += s_tot[x];
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Tiny batches (T*k <= 64, T < kSplitTopkTokens): warp t does token t's
// top-k as above, then warp 0 alone builds the whole permutation with
// shuffles: every pair (q = t k + j) is ranked by (expert, q) against all
// others, which is the expert-major, ascending-token order; the per-expert
// counts (shared-memory atomics, order-free) give the offsets, the active
// list and the GEMM's token-tile prefix (an expert has at most 64 rows here:
// one token tile).  Same results as k_topk_permute_small.
// ---------------------------------------------------------------------------
constexpr int kTinyPairs = 64;

template <int EPL>
__global__ void __launch_bounds__(512, 1)
k_topk_permute_tiny(const float* __restrict__ part, int KS, const float* __restrict__ bias,
                    int T, int E, int k, int32_t* __restrict__ topk_idx,
                    float* __restrict__ topk_w, int32_t* __restrict__ expert_off,
                    int32_t* __restrict__ row_token, int32_t* __restrict__ tok_slot_row,
                    int32_t* __restrict__ row_pair, int32_t* __restrict__ active,
                    int32_t* __restrict__ sh_off, int32_t* __restrict__ sh_rows,
                    int32_t* __restrict__ sh_active, int32_t* __restrict__ tile_off,
                    int32_t* __restrict__ counters, int n_counters, const SharedGate sg) {
  __shared__ int32_t s_idx[kTinyPairs];
  __shared__ int32_t s_cnt[kMaxExperts];
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = T * k;
  for (int t = warp; t < T; t += (int)(blockDim.x >> 5)) {
    int idx;
    float w;
    warp_topk<EPL>(part, KS, bias, T, E, k, t, lane, idx, w);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = idx;
      topk_w[(size_t)t * k + lane] = w;
      s_idx[t * k + lane] = idx;
    }
    if (sg.sgate) {
      const float gt = warp_shared_gate(sg.x, sg.g, sg.H, t, lane);
      if (lane == 0) sg.sgate[t] = gt;
    }
  }
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  if (warp != 0) return;  // no block-wide barrier follows
  constexpr unsigned kAll = 0xffffffffu;
  // this lane's pairs: q = lane and lane + 32; key (expert, q) is unique
  const int q0 = lane, q1 = lane + 32;
  const int e0 = q0 < P ? s_idx[q0] : -1, e1 = q1 < P ? s_idx[q1] : -1;
  const int key0 = e0 >= 0 ? e0 * kTinyPairs + q0 : INT_MAX;
  const int key1 = e1 >= 0 ? e1 * kTinyPairs + q1 : INT_MAX;
  int r0 = 0, r1 = 0;
#pragma unroll 4
  for (int src = 0; src < 32; ++src) {
    const int a = __shfl_sync(kAll, key0, src), b = __shfl_sync(kAll, key1, src);
    r0 += (a < key0) + (b < key0);
    r1 += (a < key1) + (b < key1);
  }
  if (e0 >= 0) {
    atomicAdd(&s_cnt[e0], 1);
    row_token[r0] = q0 / k;
    tok_slot_row[q0] = r0;
    if (row_pair) row_pair[r0] = q0;
  }
  if (e1 >= 0) {
    atomicAdd(&s_cnt[e1], 1);
    row_token[r1] = q1 / k;
    tok_slot_row[q1] = r1;
    if (row_pair) row_pair[r1] = q1;
  }
  __syncwarp();
  // lane l owns experts [l B, l B + B): sums, then exclusive scans over lanes
  const int B = (E + 31) / 32;
  int tot = 0, act = 0;
  for (int i = 0; i < B; ++i) {
    const int e = lane * B + i;
    if (e < E) {
      tot += s_cnt[e];
      act += s_cnt[e] > 0 ? 1 : 0;
    }
  }
  int it = tot, ia = act;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int vt = __shfl_up_sync(kAll, it, o), va = __shfl_up_sync(kAll, ia, o);
    if (lane >= o) {
      it += vt;
      ia += va;
    }
  }
  int off = it - tot, ai = ia - act;
  for (int i = 0; i < B; ++i) {
    const int e = lane * B + i;
    if (e < E) {
      expert_off[e] = off;
      if (tile_off) tile_off[e] = ai;  // one token tile per hit expert
      if (s_cnt[e] > 0) active[1 + ai++] = e;
      off += s_cnt[e];
    }
  }
  if (lane == 31) {
    expert_off[E] = it;
    active[0] = ia;
    if (tile_off) tile_off[E] = ia;
  }
  if (sh_rows) {  // shared expert: every token, in order
    for (int t = lane; t < T; t += 32) sh_rows[t] = t;
    if (lane == 0) {
      sh_off[0] = 0;
      sh_off[1] = T;
      sh_active[0] = T > 0 ? 1 : 0;
      sh_active[1] = 0;
    }
  }
  // the expert kernels' counters of this call start at zero
  if (counters)
    for (int i = lane; i < n_counters; i += 32) counters[i] = 0;
}

int route_kslices(int T, int H, int E) {
  if (router_tc_ok(T, H, E)) {
    // tensor-core path: split K until the CTAs fill about one wave
    const int tiles = cdiv(T, 128) * (E / 128);
    int ks = 1;
    while (ks < kMaxKSlices && tiles * ks * 2 <= num_sms() && (H / (2 * ks)) % 64 == 0) ks *= 2;
    return ks;
  }
  // Split K across CTAs when few tokens leave too few CTAs to stream Wr: with
  // 8 slices each of the 4 warps of a CTA owns one 64-column chunk (H = 2048).
  // The top-k lane sums every slice of its experts; slices x experts per lane
  // stay <= 32 so all of those loads are in flight at once.
  int ks = T <= 64 ? kMaxKSlices : 1;
  int epl = 1;
  while (epl < cdiv(E, 32)) epl <<= 1;
  while (ks > 1 && ks * epl > 32) ks >>= 1;
  while (ks > 1 && (H / ks) % 64 != 0) ks >>= 1;
  return ks;
}

cudaError_t launch_router_logits(const uint16_t* x, const float* Wr, int T, int H, int E,
                                 float* part, uint16_t* planes, uint16_t* xn, int8_t* xe,
                                 int32_t* status, cudaStream_t s, bool pdl) {
  const int KS = route_kslices(T, H, E);
  if (router_tc_ok(T, H, E))
    return launch_router_logits_tc(x, Wr, T, H, E, KS, part, planes, xn, xe, status, s, pdl);
  const int kslice = H / KS;
  const dim3 blk(kRouteWarps * 32);
  if (T <= 8)
    return launch_k(k_router_mma<1>, dim3(cdiv(E, 16), KS, cdiv(T, 8)), blk, 0, s, pdl, x, Wr,
                    T, H, E, kslice, part, xn, xe, status);
  if (T <= 64)
    return launch_k(k_router_mma<2>, dim3(cdiv(E, 16), KS, cdiv(T, 16)), blk, 0, s, pdl, x, Wr,
                    T, H, E, kslice, part, xn, xe, status);
  return launch_k(k_router_mma<4>, dim3(cdiv(E, 16), KS, cdiv(T, 32)), blk, 0, s, pdl, x, Wr,
                  T, H, E, kslice, part, xn, xe, status);
}

cudaError_t launch_route(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                         int E, int k, float* part, uint16_t* planes, int32_t* topk_idx,
                         float* topk_w, uint16_t* xn, int8_t* xe, int32_t* status,
                         cudaStream_t s, bool pdl, const float* shared_gate, float* sgate) {
  if (T == 0) return cudaSuccess;
  SharedGate sg;
  if (sgate) {
    sg.x = x;
    sg.g = shared_gate;
    sg.H = H;
    sg.sgate = sgate;
  }
  cudaError_t err = launch_router_logits(x, Wr, T, H, E, part, planes, xn, xe, status, s, pdl);
  if (err != cudaSuccess) return err;
  const int KS = route_kslices(T, H, E);
  const int epl = cdiv(E, 32);
  const dim3 g2(cdiv(T, 8)), blk(256);
#define MOE_TOPK(EPLV) \
  launch_k(k_router_topk<EPLV>, g2, blk, 0, s, pdl, part, KS, bias, T, E, k, topk_idx, topk_w, sg)
  if (epl <= 1) return MOE_TOPK(1);
  if (epl <= 2) return MOE_TOPK(2);
  if (epl <= 4) return MOE_TOPK(4);
  if (epl <= 8) return MOE_TOPK(8);
  if (epl <= 16) return MOE_TOPK(16);
  return MOE_TOPK(32);
#undef MOE_TOPK
}

bool small_route_permute_ok(int T, int E, int k) {
  return (long long)T * k <= kSmallPairs && E <= 1024;
}

cudaError_t launch_route_permute_small(const uint16_t* x, const float* Wr, const float* bias,
                                       int T, int H, int E, int k, float* part,
                                       uint16_t* planes, int32_t* topk_idx, float* topk_w,
                                       int32_t* expert_off,
                                       int32_t* row_token, int32_t* tok_slot_row,
                                       int32_t* row_pair, int32_t* active, int32_t* sh_off,
                                       int32_t* sh_rows, int32_t* sh_active, uint16_t* xn,
                                       int8_t* xe, int32_t* tile_off, int32_t* counters,
                                       int n_counters, int32_t* status, cudaStream_t s, bool pdl,
                                       const float* shared_gate, float* sgate) {
  cudaError_t err = launch_router_logits(x, Wr, T, H, E, part, planes, xn, xe, status, s, pdl);
  SharedGate sg;
  if (sgate) {
    sg.x = x;
    sg.g = shared_gate;
    sg.H = H;
    sg.sgate = sgate;
  }
  if (err != cudaSuccess) return err;
  const int KS = route_kslices(T, H, E);
  const size_t smem = small_route_smem(E);
  const int epl = cdiv(E, 32);
  if (T >= kSplitTopkTokens) {
    // top-k spread over T/8 CTAs (a warp per token), then the permutation
    // alone in one CTA: one launch more, but the selections no longer queue
    // on a single SM
    const dim3 g2(cdiv(T, 8)), blk(256);
#define MOE_TOPK(EPLV) \
  launch_k(k_router_topk<EPLV>, g2, blk, 0, s, pdl, part, KS, bias, T, E, k, topk_idx, topk_w, sg)
    err = epl <= 1 ? MOE_TOPK(1) : epl <= 2 ? MOE_TOPK(2) : epl <= 4 ? MOE_TOPK(4)
        : epl <= 8 ? MOE_TOPK(8) : epl <= 16 ? MOE_TOPK(16) : MOE_TOPK(32);
#undef MOE_TOPK
    if (err != cudaSuccess) return err;
    err = ensure_smem((const void*)k_topk_permute_small<0>, (int)small_route_smem(1024));
    if (err != cudaSuccess) return err;
    return launch_k(k_topk_permute_small<0>, dim3(1), dim3(1024), smem, s, pdl, part, KS, bias,
                    T, E, k, topk_idx, topk_w, expert_off, row_token, tok_slot_row, row_pair,
                    active, sh_off, sh_rows, sh_active, tile_off, counters, n_counters, sg);
  }
  if ((long long)T * k <= kTinyPairs) {
    const dim3 blk(32 * T);  // T < kSplitTopkTokens: at most 480 threads
#define MOE_TINY(EPLV)                                                                        \
  return launch_k(k_topk_permute_tiny<EPLV>, dim3(1), blk, 0, s, pdl, part, KS, bias, T, E, k, \
                  topk_idx, topk_w, expert_off, row_token, tok_slot_row, row_pair, active,     \
                  sh_off, sh_rows, sh_active, tile_off, counters, n_counters, sg)
    if (epl <= 1) MOE_TINY(1);
    if (epl <= 2) MOE_TINY(2);
    if (epl <= 4) MOE_TINY(4);
    if (epl <= 8) MOE_TINY(8);
    if (epl <= 16) MOE_TINY(16);
    MOE_TINY(32);
#undef MOE_TINY
  }
#define MOE_SMALL(EPLV)                                                                      \
  do {                                                                                       \
    err = ensure_smem((const void*)k_topk_permute_small<EPLV>, (int)small_route_smem(1024)); \
    if (err != cudaSuccess) return err;                                                      \
    return launch_k(k_topk_permute_small<EPLV>, dim3(1), dim3(1024), smem, s, pdl, part, KS, \
                    bias, T, E, k, topk_idx, topk_w, expert_off, row_token, tok_slot_row,    \
                    row_pair, active, sh_off, sh_rows, sh_active, tile_off, counters,        \
                    n_counters, sg);                                                         \
  } while (0)
  if (epl <= 1) MOE_SMALL(1);
  if (epl <= 2) MOE_SMALL(2);
  if (epl <= 4) MOE_SMALL(4);
  if (epl <= 8) MOE_SMALL(8);
  if (epl <= 16) MOE_SMALL(16);
  MOE_SMALL(32);
#undef MOE_SMALL
}

}  // namespace moe
