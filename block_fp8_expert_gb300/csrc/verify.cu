// Runtime cross-check of a layer call on sampled tokens (colizig README, CLI
// reference: --cuda-verify, which checks the CUDA path against the CPU path).
// Here the check runs on the GPU, on an arithmetic path independent of the
// layer kernels: plain fp32 dot products with the E4M3 codes decoded by bit
// fields and multiplied by their block scale, no tensor cores and no
// power-of-two normalisation; SwiGLU with expf; the combine in fp32.  For
// each sampled token it recomputes the layer output from the routing the
// layer call produced (topk_idx / topk_w) and reports the worst
// |out - ref| / (1e-2 (|ref| + rms(ref))), rms over the sampled outputs.
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kVerifyWarps = 8;
constexpr int kVerifyMaxTokens = 64;

// E4M3 (no infinities) from its bit fields: s eeee mmm.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float v;
  if (e == 0)
    v = (float)m * 0x1p-9f;  // 2^-6 * m / 8
  else if (e == 15 && m == 7)
    v = __int_as_float(0x7fc00000);  // NaN
  else
    v = (float)(8 + m) * pow2f((int)e - 10);  // 2^(e-7) (1 + m / 8)
  return (c & 0x80u) ? -v : v;
}

// Pair p of the sample: token tokens[p / S], slot p % S (S = k, or k + 1
// with the shared expert as the last slot).
struct VPair {
  int t;       // token
  int e;       // expert (-1: the shared expert)
  float w;     // routing weight (shared: its gate factor or 1)
};

__device__ __forceinline__ VPair vpair(int p, int S, int k, bool has_shared,
                                       const int32_t* tokens, const int32_t* topk_idx,
                                       const float* topk_w) {
  VPair r;
  r.t = tokens[p / S];
  const int j = p % S;
  if (has_shared && j == k) {
    r.e = -1;
    r.w = 1.f;
  } else {
    r.e = topk_idx[(size_t)r.t * k + j];
    r.w = topk_w[(size_t)r.t * k + j];
  }
  return r;
}

// hid[p, i] = silu(g) * u for pair p, one warp per (pair, feature i).
__global__ void __launch_bounds__(kVerifyWarps * 32)
k_verify_gateup(const uint16_t* __restrict__ x, const int32_t* __restrict__ tokens,
                const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int k,
                int S, bool has_shared, moe_fp8_ffn routed, moe_fp8_ffn shared, int H, int I,
                int Is, int E, int T, int npairs, float* __restrict__ hid,
                int32_t* __restrict__ bad) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kVerifyWarps + (threadIdx.x >> 5);
  const int Imax = I > Is ? I : Is;
  if (wid >= (long long)npairs * Imax) return;
  const int p = (int)(wid / Imax), i = (int)(wid % Imax);
  const VPair q = vpair(p, S, k, has_shared, tokens, topk_idx, topk_w);
  const bool sh = q.e < 0;
  const int Ie = sh ? Is : I;
  if (i >= Ie) return;
  if (q.t < 0 || q.t >= T || (!sh && (q.e >= E || q.e < 0))) {  // nothing to recompute
    if (lane == 0) atomicOr(bad, 1);
    return;
  }
  const moe_fp8_mat& G = sh ? shared.gate : routed.gate;
  const moe_fp8_mat& U = sh ? shared.up : routed.up;
  const int ee = sh ? 0 : q.e;
  const int nHb = cdiv(H, kScaleBlock), nIb = cdiv(Ie, kScaleBlock);
  const uint8_t* gr = G.codes + ((size_t)ee * Ie + i) * H;
  const uint8_t* ur = U.codes + ((size_t)ee * Ie + i) * H;
  const float* gs = G.scales + ((size_t)ee * nIb + i / kScaleBlock) * nHb;
  const float* us = U.scales + ((size_t)ee * nIb + i / kScaleBlock) * nHb;
  const uint16_t* xr = x + (size_t)q.t * H;
  float g = 0.f, u = 0.f;
  for (int h = lane; h < H; h += 32) {
    const float xv = __uint_as_float((uint32_t)xr[h] << 16);
    g = fmaf(e4m3_value(gr[h]) * gs[h / kScaleBlock], xv, g);
    u = fmaf(e4m3_value(ur[h]) * us[h / kScaleBlock], xv, u);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    g += __shfl_xor_sync(0xffffffffu, g, o);
    u += __shfl_xor_sync(0xffffffffu, u, o);
  }
  if (lane == 0) hid[(size_t)p * Imax + i] = g / (1.f + expf(-g)) * u;
}

// y[p, h] = sum_i hid[p, i] Wd[h, i], one warp per (pair, output h).
__global__ void __launch_bounds__(kVerifyWarps * 32)
k_verify_down(const int32_t* __restrict__ tokens, const int32_t* __restrict__ topk_idx,
              const float* __restrict__ topk_w, int k, int S, bool has_shared,
              moe_fp8_ffn routed, moe_fp8_ffn shared, int H, int I, int Is, int E, int T,
              int npairs, const float* __restrict__ hid, float* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kVerifyWarps + (threadIdx.x >> 5);
  if (wid >= (long long)npairs * H) return;
  const int p = (int)(wid / H), h = (int)(wid % H);
  const VPair q = vpair(p, S, k, has_shared, tokens, topk_idx, topk_w);
  const bool sh = q.e < 0;
  if (q.t < 0 || q.t >= T || (!sh && q.e >= E)) return;  // flagged by the gate/up kernel
  const int Ie = sh ? Is : I, Imax = I > Is ? I : Is;
  const moe_fp8_mat& Dm = sh ? shared.down : routed.down;
  const int ee = sh ? 0 : q.e;
  const int nHb = cdiv(H, kScaleBlock), nIb = cdiv(Ie, kScaleBlock);
  const uint8_t* dr = Dm.codes + ((size_t)ee * H + h) * Ie;
  const float* ds = Dm.scales + ((size_t)ee * nHb + h / kScaleBlock) * nIb;
  const float* hp = hid + (size_t)p * Imax;
  float acc = 0.f;
  for (int i = lane; i < Ie; i += 32)
    acc = fmaf(e4m3_value(dr[i]) * ds[i / kScaleBlock], hp[i], acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) y[(size_t)p * H + h] = acc;
}

// ref[n, h] = sum_j w_j y[pair(n, j), h] (+ gate * shared), then one CTA
// reduces: rms(ref), and the worst |out - ref| / (1e-2 (|ref| + rms)).
__global__ void __launch_bounds__(1024)
k_verify_compare(const uint16_t* __restrict__ x, const int32_t* __restrict__ tokens,
                 const float* __restrict__ topk_w, int k, int S, bool has_shared,
                 const float* __restrict__ shared_gate, int H, int T, int n,
                 const float* __restrict__ y, const uint16_t* __restrict__ out,
                 float* __restrict__ ref, const int32_t* __restrict__ bad,
                 float* __restrict__ result) {
  __shared__ float red[32];
  __shared__ float s_gate[kVerifyMaxTokens];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // gate factors of the sampled tokens (warp per token)
  for (int m = warp; m < n; m += 32) {
    float f = 1.f;
    if (has_shared && shared_gate && tokens[m] >= 0 && tokens[m] < T) {
      const uint16_t* xr = x + (size_t)tokens[m] * H;
      float z = 0.f;
      for (int h = lane; h < H; h += 32)
        z = fmaf(__uint_as_float((uint32_t)xr[h] << 16), shared_gate[h], z);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      f = 1.f / (1.f + expf(-z));
    }
    if (lane == 0) s_gate[m] = f;
  }
  __syncthreads();
  float ss = 0.f;
  for (long long o = tid; o < (long long)n * H; o += blockDim.x) {
    const int m = (int)(o / H), h = (int)(o % H);
    const int t = tokens[m];
    if (t < 0 || t >= T) continue;  // flagged by the gate/up kernel
    float r = 0.f;
    for (int j = 0; j < k; ++j)
      r = fmaf(topk_w[(size_t)t * k + j], y[((size_t)m * S + j) * H + h], r);
    if (has_shared) r = fmaf(s_gate[m], y[((size_t)m * S + k) * H + h], r);
    ref[o] = r;
    ss = fmaf(r, r, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    red[0] = sqrtf(s / (float)((long long)n * H));
  }
  __syncthreads();
  const float rms = red[0];
  __syncthreads();
  float worst = 0.f, worst_abs = 0.f;
  for (long long o = tid; o < (long long)n * H; o += blockDim.x) {
    const int m = (int)(o / H), h = (int)(o % H);
    if (tokens[m] < 0 || tokens[m] >= T) continue;
    const float got = __uint_as_float((uint32_t)out[(size_t)tokens[m] * H + h] << 16);
    const float err = fabsf(got - ref[o]);
    const float ratio = err / (1e-2f * (fabsf(ref[o]) + rms));
    // NaN compares false: make it the worst
    worst = (ratio <= worst) ? worst : (ratio == ratio ? ratio : INFINITY);
    worst_abs = fmaxf(worst_abs, err);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    worst_abs = fmaxf(worst_abs, __shfl_xor_sync(0xffffffffu, worst_abs, o));
  }
  if (lane == 0) red[warp] = worst;
  __syncthreads();
  if (tid == 0) {
    float wv = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) wv = fmaxf(wv, red[w]);
    result[0] = *bad ? INFINITY : wv;  // an expert index outside [0, E): no reference
    result[2] = rms;
  }
  __syncthreads();
  if (lane == 0) red[warp] = worst_abs;
  __syncthreads();
  if (tid == 0) {
    float wv = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) wv = fmaxf(wv, red[w]);
    result[1] = wv;
  }
}

}  // namespace

int verify_max_tokens() { return kVerifyMaxTokens; }

size_t verify_workspace(const moe_dims& d, int n) {
  const size_t S = (size_t)d.k + (d.I_shared ? 1 : 0), Imax = d.I > d.I_shared ? d.I : d.I_shared;
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  return up((size_t)n * S * Imax * 4) + up((size_t)n * S * d.H * 4) + up((size_t)n * d.H * 4) + 256;
}

cudaError_t launch_verify(const uint16_t* x, const moe_fp8_ffn& routed, const moe_fp8_ffn* shared,
                          const float* shared_gate, const moe_dims& d, const uint16_t* out,
                          const int32_t* topk_idx, const float* topk_w, const int32_t* tokens,
                          int n, float* result, void* ws, cudaStream_t s) {
  const bool has_shared = d.I_shared > 0;
  const int S = d.k + (has_shared ? 1 : 0), Imax = d.I > d.I_shared ? d.I : d.I_shared;
  const int npairs = n * S;
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  char* w = static_cast<char*>(ws);
  float* hid = reinterpret_cast<float*>(w);
  float* y = reinterpret_cast<float*>(w + up((size_t)npairs * Imax * 4));
  float* ref = reinterpret_cast<float*>(w + up((size_t)npairs * Imax * 4) + up((size_t)npairs * d.H * 4));
  int32_t* bad = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ref) + up((size_t)n * d.H * 4));
  cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const moe_fp8_ffn sh = shared ? *shared : moe_fp8_ffn{};
  const long long w1 = (long long)npairs * Imax, w2 = (long long)npairs * d.H;
  e = launch_k(k_verify_gateup, dim3((unsigned)((w1 + kVerifyWarps - 1) / kVerifyWarps)),
               dim3(kVerifyWarps * 32), 0, s, false, x, tokens, topk_idx, topk_w, d.k, S,
               has_shared, routed, sh, d.H, d.I, d.I_shared, d.E, d.T, npairs, hid, bad);
  if (e != cudaSuccess) return e;
  e = launch_k(k_verify_down, dim3((unsigned)((w2 + kVerifyWarps - 1) / kVerifyWarps)),
               dim3(kVerifyWarps * 32), 0, s, false, tokens, topk_idx, topk_w, d.k, S,
               has_shared, routed, sh, d.H, d.I, d.I_shared, d.E, d.T, npairs, (const float*)hid,
               y);
  if (e != cudaSuccess) return e;
  return launch_k(k_verify_compare, dim3(1), dim3(1024), 0, s, false, x, tokens, topk_w, d.k, S,
                  has_shared, shared_gate, d.H, d.T, n, (const float*)y, out, ref,
                  (const int32_t*)bad,
                  result);
}

}  // namespace moe
