// Combine: out[t] = sum_j w[t,j] y_perm[tok_slot_row[t*k+j]] (+ shared_y[t]),
// summed in fp32 in slot order j, rounded once to bf16.
#include "moe_internal.h"

namespace moe {

__global__ void __launch_bounds__(256)
k_combine(const float* __restrict__ y_perm, const int32_t* __restrict__ tok_slot_row,
          const float* __restrict__ topk_w, const float* __restrict__ shared_y, int T, int H,
          int k, uint16_t* __restrict__ out) {
  griddep_wait();
  griddep_trigger();
  const int H4 = H / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * H4) return;
  const int t = (int)(i / H4), h = (int)(i % H4) * 4;
  float4 acc = shared_y ? __ldg(reinterpret_cast<const float4*>(shared_y + (size_t)t * H + h))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
  // Slots in groups of 8: row indices and weights first, then the 8 row
  // gathers, so the loads of a group are in flight together.
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += 8) {
    int row[8];
    float w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      row[u] = j < k ? tok_slot_row[(size_t)t * k + j] : -1;
      w[u] = j < k ? topk_w[(size_t)t * k + j] : 0.f;
    }
    float4 y[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      y[u] = row[u] >= 0 ? __ldg(reinterpret_cast<const float4*>(y_perm + (size_t)row[u] * H + h))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[u] < 0) continue;
      r.x = fmaf(w[u], y[u].x, r.x);
      r.y = fmaf(w[u], y[u].y, r.y);
      r.z = fmaf(w[u], y[u].z, r.z);
      r.w = fmaf(w[u], y[u].w, r.w);
    }
  }
  acc.x += r.x;
  acc.y += r.y;
  acc.z += r.z;
  acc.w += r.w;
  uint2 o;
  o.x = pack_bf16x2(acc.x, acc.y);
  o.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(out + (size_t)t * H + h) = o;
}

cudaError_t launch_combine(const float* y_perm, const int32_t* tok_slot_row, const float* topk_w,
                           const float* shared_y, int T, int H, int k, uint16_t* out,
                           cudaStream_t s, bool pdl) {
  const long long n = (long long)T * (H / 4);
  if (n == 0) return cudaSuccess;
  return launch_k(k_combine, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, pdl, y_perm,
                  tok_slot_row, topk_w, shared_y, T, H, k, out);
}

}  // namespace moe
