// Router: logits l = x Wr^T (+ b), then per token the top-k experts and their
// renormalised weights (colizig README, model table: experts with top-k
// routing).  The renormalised weight p_j / sum_sel p equals the softmax over
// the k selected logits, because the full softmax's normaliser cancels; the
// kernel computes it that way and never forms the E probabilities.
#include "moe_internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// logits: one warp per expert, 8 tokens per CTA row of the grid
// ---------------------------------------------------------------------------
constexpr int kRouteTok = 8;    // tokens per CTA
constexpr int kRouteWarps = 4;  // experts per CTA

__global__ void __launch_bounds__(kRouteWarps * 32)
k_router_logits(const uint16_t* __restrict__ x, const float* __restrict__ Wr,
                const float* __restrict__ bias, int T, int H, int E,
                float* __restrict__ logits, int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  // The router runs first in a layer call: it clears the status word that
  // later kernels of the call may raise.
  if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *status = 0;
  const int e = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  const int t0 = blockIdx.y * kRouteTok;
  if (e >= E) return;
  const int nt = min(kRouteTok, T - t0);
  float acc[kRouteTok];
#pragma unroll
  for (int t = 0; t < kRouteTok; ++t) acc[t] = 0.f;
  const float* wrow = Wr + (size_t)e * H;
  for (int h = lane * 4; h < H; h += 128) {
    const float4 w4 = __ldg(reinterpret_cast<const float4*>(wrow + h));
#pragma unroll
    for (int t = 0; t < kRouteTok; ++t) {
      if (t < nt) {
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * H + h));
        acc[t] = fmaf(bf16_lo(xv.x), w4.x, acc[t]);
        acc[t] = fmaf(bf16_hi(xv.x), w4.y, acc[t]);
        acc[t] = fmaf(bf16_lo(xv.y), w4.z, acc[t]);
        acc[t] = fmaf(bf16_hi(xv.y), w4.w, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRouteTok; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
  if (lane == 0) {
    const float b = bias ? bias[e] : 0.f;
#pragma unroll
    for (int t = 0; t < kRouteTok; ++t)
      if (t < nt) logits[(size_t)(t0 + t) * E + e] = acc[t] + b;
  }
}

// ---------------------------------------------------------------------------
// top-k + renormalisation: one warp per token, EPL logits per lane
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int EPL>
__global__ void __launch_bounds__(256)
k_router_topk(const float* __restrict__ logits, int T, int E, int k,
              int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* lrow = logits + (size_t)t * E;
  float v[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? lrow[e] : -INFINITY;
  }
  uint32_t taken = 0;
  float my_val = -INFINITY;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    // best not-yet-taken candidate of this lane
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_val = bv;
      my_idx = bi;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < k ? expf(my_val - vmax) : 0.f;
  float s = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = my_idx;
    topk_w[(size_t)t * k + lane] = ex / s;
  }
}

cudaError_t launch_route(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                         int E, int k, float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 g1(cdiv(E, kRouteWarps), cdiv(T, kRouteTok));
  k_router_logits<<<g1, kRouteWarps * 32, 0, s>>>(x, Wr, bias, T, H, E, logits, status);
  const int g2 = cdiv(T, 8);
  const int epl = cdiv(E, 32);
  if (epl <= 1)
    k_router_topk<1><<<g2, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  else if (epl <= 2)
    k_router_topk<2><<<g2, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  else if (epl <= 4)
    k_router_topk<4><<<g2, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  else if (epl <= 8)
    k_router_topk<8><<<g2, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  else if (epl <= 16)
    k_router_topk<16><<<g2, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  else
    k_router_topk<32><<<g2, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w);
  return cudaGetLastError();
}

}  // namespace moe
