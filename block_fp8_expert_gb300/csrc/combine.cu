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
