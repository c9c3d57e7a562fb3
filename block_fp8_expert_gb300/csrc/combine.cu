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
  combine4(y_perm, tok_slot_row, topk_w, shared_y, t, h, H, k, out);
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
