// Combine: out[t] = sum_j w[t,j] y_perm[tok_slot_row[t*k+j]] (+ shared_y[t]),
// summed in fp32 in slot order j, rounded once to bf16.  The expert outputs
// are fp32 (the C ABI's moe_combine) or, inside moe_layer_forward, fp16 y''
// with one power-of-two exponent per row and 32 columns (y = y'' 2^s).
#include "moe_internal.h"

namespace moe {

// One thread per 16 bytes of each of a token's fp32 expert rows (4 outputs).
__global__ void __launch_bounds__(256)
k_combine(const float* __restrict__ y_perm, const int32_t* __restrict__ tok_slot_row,
          const float* __restrict__ topk_w, const float* __restrict__ shared_y, int T, int H,
          int k, uint16_t* __restrict__ out) {
  griddep_wait();
  griddep_trigger();
  const int HV = H / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * HV) return;
  const int t = (int)(i / HV), h = (int)(i % HV) * 4;
  combine_v<float, 4>(y_perm, tok_slot_row, topk_w, shared_y, t, h, H, k, out);
}

// The layer call's combine, k <= KMAX (8, 16 or 32), one thread per 8
// outputs of a token.  The slot rows and weights come from the routing,
// which had completed before the expert kernels' first wait, so they are
// loaded before this kernel waits for the expert outputs.  Each term is
// fmaf(w 2^s, y'', r): w 2^s is exact, so this rounds w y + r once, the
// same arithmetic as an fp32 y; the shared row (y''_s 2^s_s, exact) comes
// first, then the slots in order j, eight rows in flight at a time, one bf16
// rounding.  yexp is [H / 32][P], syexp [H / 32][sstride].
template <int KMAX>
__global__ void __launch_bounds__(256)
k_combine_layer(const uint16_t* __restrict__ y, const int16_t* __restrict__ yexp, int P,
                const int32_t* __restrict__ tok_slot_row, const float* __restrict__ topk_w,
                const uint16_t* __restrict__ sy, const int16_t* __restrict__ syexp, int sstride,
                const float* __restrict__ sgate, int T, int H, int k,
                uint16_t* __restrict__ out) {
  const int HV = H / 8;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * HV) return;
  const int t = (int)(i / HV), h = (int)(i % HV) * 8, grp = h >> 5;
  int row[KMAX];
  float w[KMAX];
#pragma unroll
  for (int u = 0; u < KMAX; ++u) {
    row[u] = u < k ? tok_slot_row[(size_t)t * k + u] : -1;
    w[u] = u < k ? topk_w[(size_t)t * k + u] : 0.f;
  }
  griddep_wait();
  griddep_trigger();
  float acc[8], r[8];
#pragma unroll
  for (int v = 0; v < 8; ++v) acc[v] = r[v] = 0.f;
  if (sy) {
    load_v(sy + (size_t)t * H + h, acc);
    float f = ldexp2f(1.f, syexp[(size_t)grp * sstride + t]);
    if (sgate) f *= sgate[t];  // gated shared expert
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[v] *= f;  // exact unless it leaves fp32's range
  }
#pragma unroll
  for (int j0 = 0; j0 < KMAX; j0 += 8) {
    // eight rows in flight, kept packed (8 fp16 in 16 bytes) until used
    uint4 yr[8];
    int ys[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[j0 + u] >= 0) {
        yr[u] = __ldg(reinterpret_cast<const uint4*>(y + (size_t)row[j0 + u] * H + h));
        ys[u] = yexp[(size_t)grp * P + row[j0 + u]];
      } else {
        yr[u] = make_uint4(0, 0, 0, 0);
        ys[u] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[j0 + u] < 0) continue;
      const float wf = ldexp2f(w[j0 + u], ys[u]);
      float yv[8];
      unpack_f16x8(yr[u], yv);
#pragma unroll
      for (int v = 0; v < 8; ++v) r[v] = fmaf(wf, yv[v], r[v]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) o[v] = pack_bf16x2(acc[2 * v] + r[2 * v], acc[2 * v + 1] + r[2 * v + 1]);
  *reinterpret_cast<uint4*>(out + (size_t)t * H + h) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_combine_layer(const uint16_t* y, const int16_t* yexp, int P,
                                 const int32_t* tok_slot_row, const float* topk_w,
                                 const uint16_t* sy, const int16_t* syexp, int sstride,
                                 const float* sgate, int T, int H, int k, uint16_t* out,
                                 cudaStream_t s) {
  const long long n = (long long)T * (H / 8);
  if (n == 0) return cudaSuccess;
  const dim3 grid((unsigned)((n + 255) / 256)), blk(256);
  if (k <= 8)
    return launch_k(k_combine_layer<8>, grid, blk, 0, s, true, y, yexp, P, tok_slot_row, topk_w,
                    sy, syexp, sstride, sgate, T, H, k, out);
  if (k <= 16)
    return launch_k(k_combine_layer<16>, grid, blk, 0, s, true, y, yexp, P, tok_slot_row, topk_w,
                    sy, syexp, sstride, sgate, T, H, k, out);
  return launch_k(k_combine_layer<32>, grid, blk, 0, s, true, y, yexp, P, tok_slot_row, topk_w, sy,
                  syexp, sstride, sgate, T, H, k, out);
}

cudaError_t launch_combine(const float* y_perm, const int32_t* tok_slot_row, const float* topk_w,
                           const float* shared_y, int T, int H, int k, uint16_t* out,
                           cudaStream_t s, bool pdl) {
  const long long n = (long long)T * (H / 4);
  if (n == 0) return cudaSuccess;
  const dim3 grid((unsigned)((n + 255) / 256));
  return launch_k(k_combine, grid, dim3(256), 0, s, pdl, y_perm, tok_slot_row, topk_w, shared_y,
                  T, H, k, out);
}

}  // namespace moe
