// Combine: out[t] = sum_j w[t,j] y_perm[tok_slot_row[t*k+j]] (+ shared_y[t]),
// summed in fp32 in slot order j, rounded once to bf16.  The expert outputs
// are fp32 (the C ABI's moe_combine) or fp16 (inside moe_layer_forward).
#include "moe_internal.h"

namespace moe {

// One thread per 16 bytes of each of a token's expert rows: 4 fp32 or 8 fp16
// outputs.
template <typename YT>
__global__ void __launch_bounds__(256)
k_combine(const YT* __restrict__ y_perm, const int32_t* __restrict__ tok_slot_row,
          const float* __restrict__ topk_w, const YT* __restrict__ shared_y, int T, int H,
          int k, uint16_t* __restrict__ out) {
  constexpr int V = 16 / sizeof(YT);
  griddep_wait();
  griddep_trigger();
  const int HV = H / V;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * HV) return;
  const int t = (int)(i / HV), h = (int)(i % HV) * V;
  combine_v<YT, V>(y_perm, tok_slot_row, topk_w, shared_y, t, h, H, k, out);
}

// The layer call's combine, k <= KMAX (8 or 16): the slot rows and weights
// come from the routing, which had completed before the expert kernels'
// first wait, so they are loaded before this kernel waits for the expert
// outputs; the arithmetic is combine_v's (shared row first, then fmaf over
// the slots in order j, eight rows in flight at a time, one bf16 rounding).
template <typename YT, int KMAX>
__global__ void __launch_bounds__(256)
k_combine_early(const YT* __restrict__ y_perm, const int32_t* __restrict__ tok_slot_row,
                const float* __restrict__ topk_w, const YT* __restrict__ shared_y, int T, int H,
                int k, uint16_t* __restrict__ out) {
  constexpr int V = 16 / sizeof(YT);
  const int HV = H / V;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * HV) return;
  const int t = (int)(i / HV), h = (int)(i % HV) * V;
  int row[KMAX];
  float w[KMAX];
#pragma unroll
  for (int u = 0; u < KMAX; ++u) {
    row[u] = u < k ? tok_slot_row[(size_t)t * k + u] : -1;
    w[u] = u < k ? topk_w[(size_t)t * k + u] : 0.f;
  }
  griddep_wait();
  griddep_trigger();
  float acc[V], r[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = r[v] = 0.f;
  if (shared_y) load_v(shared_y + (size_t)t * H + h, acc);
#pragma unroll
  for (int j0 = 0; j0 < KMAX; j0 += 8) {
    float y[8][V];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[j0 + u] >= 0) {
        load_v(y_perm + (size_t)row[j0 + u] * H + h, y[u]);
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) y[u][v] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[j0 + u] < 0) continue;
#pragma unroll
      for (int v = 0; v < V; ++v) r[v] = fmaf(w[j0 + u], y[u][v], r[v]);
    }
  }
  uint32_t o[V / 2];
#pragma unroll
  for (int v = 0; v < V / 2; ++v) o[v] = pack_bf16x2(acc[2 * v] + r[2 * v], acc[2 * v + 1] + r[2 * v + 1]);
  if constexpr (V == 8)
    *reinterpret_cast<uint4*>(out + (size_t)t * H + h) = make_uint4(o[0], o[1], o[2], o[3]);
  else
    *reinterpret_cast<uint2*>(out + (size_t)t * H + h) = make_uint2(o[0], o[1]);
}

cudaError_t launch_combine_layer(const void* y_perm, bool y_half, const int32_t* tok_slot_row,
                                 const float* topk_w, const void* shared_y, int T, int H, int k,
                                 uint16_t* out, cudaStream_t s) {
  if (k > 16)
    return launch_combine(y_perm, y_half, tok_slot_row, topk_w, shared_y, T, H, k, out, s, true);
  const long long n = (long long)T * (H / (y_half ? 8 : 4));
  if (n == 0) return cudaSuccess;
  const dim3 grid((unsigned)((n + 255) / 256));
  const uint16_t* yh = static_cast<const uint16_t*>(y_perm);
  const uint16_t* sh = static_cast<const uint16_t*>(shared_y);
  const float* yf = static_cast<const float*>(y_perm);
  const float* sf = static_cast<const float*>(shared_y);
  if (k <= 8)
    return y_half ? launch_k(k_combine_early<uint16_t, 8>, grid, dim3(256), 0, s, true, yh,
                             tok_slot_row, topk_w, sh, T, H, k, out)
                  : launch_k(k_combine_early<float, 8>, grid, dim3(256), 0, s, true, yf,
                             tok_slot_row, topk_w, sf, T, H, k, out);
  return y_half ? launch_k(k_combine_early<uint16_t, 16>, grid, dim3(256), 0, s, true, yh,
                           tok_slot_row, topk_w, sh, T, H, k, out)
                : launch_k(k_combine_early<float, 16>, grid, dim3(256), 0, s, true, yf,
                           tok_slot_row, topk_w, sf, T, H, k, out);
}

cudaError_t launch_combine(const void* y_perm, bool y_half, const int32_t* tok_slot_row,
                           const float* topk_w, const void* shared_y, int T, int H, int k,
                           uint16_t* out, cudaStream_t s, bool pdl) {
  const long long n = (long long)T * (H / (y_half ? 8 : 4));
  if (n == 0) return cudaSuccess;
  const dim3 grid((unsigned)((n + 255) / 256));
  if (y_half)
    return launch_k(k_combine<uint16_t>, grid, dim3(256), 0, s, pdl,
                    static_cast<const uint16_t*>(y_perm), tok_slot_row, topk_w,
                    static_cast<const uint16_t*>(shared_y), T, H, k, out);
  return launch_k(k_combine<float>, grid, dim3(256), 0, s, pdl, static_cast<const float*>(y_perm),
                  tok_slot_row, topk_w, static_cast<const float*>(shared_y), T, H, k, out);
}

}  // namespace moe
