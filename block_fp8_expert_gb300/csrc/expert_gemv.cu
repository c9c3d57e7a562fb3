// Routed-expert FFN for few tokens per expert (decode): a grouped GEMV that
// streams only the selected experts' E4M3 bytes (colizig README, "Features":
// block-FP8 weights, fused decode+FMA dot products; "MoE per-expert
// evaluation").
//
// Weight bytes go from HBM straight into registers with 16-byte loads (no
// shared-memory round trip), are decoded there, and feed warp-level bf16
// tensor-core MMAs whose N side is the expert's tokens (8 per MMA).  The
// tensor core here is only a cheap multiply-accumulate for 1..16 tokens; the
// kernel's bound is the weight stream.
//
// K permutation: an MMA's 16 logical K positions are fed from physical
// columns so that a thread owns 16 consecutive bytes of a weight row: for
// thread (g = lane/4, c = lane%4) and MMA step s of a 64-column chunk, the
// logical pairs (2c, 2c+1) and (2c+8, 2c+9) are physical columns
// 16c + 4s + {0,1} and 16c + 4s + {2,3}.  The activations use the same map,
// so every product pairs the right weight with the right activation.
//
// Block scale: weights are decoded as dec(code) * 2^-112 (exact); each
// 64-column chunk lies inside one 128x128 scale block, so the chunk's MMA sum
// is multiplied by scale * 2^112 and added to an fp32 accumulator.
#include "moe_internal.h"

namespace moe {

constexpr int kGemvWarps = 8;

// One 64-column chunk: 16 weight rows (g, g+8) x NT*8 tokens.  F16: weights
// decoded exactly to fp16 and activations in fp16; otherwise weights decoded
// to bf16 * 2^-112 and activations in bf16.
template <int NT, bool F16>
__device__ __forceinline__ void chunk_mma(const uint4& w_lo, const uint4& w_hi,
                                          const uint4 (&xa)[NT][2], float (&part)[NT][4]) {
  uint32_t wl[8], wh[8];
  if (F16) {
    decode16_f16(w_lo, wl);
    decode16_f16(w_hi, wh);
  } else {
    decode16_scaled(w_lo, wl);
    decode16_scaled(w_hi, wh);
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t xr[8] = {xa[nt][0].x, xa[nt][0].y, xa[nt][0].z, xa[nt][0].w,
                            xa[nt][1].x, xa[nt][1].y, xa[nt][1].z, xa[nt][1].w};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t a[4] = {wl[2 * s], wh[2 * s], wl[2 * s + 1], wh[2 * s + 1]};
      const uint32_t b[2] = {xr[2 * s], xr[2 * s + 1]};
      if (F16)
        mma_f16_16x8x16(part[nt], a, b);
      else
        mma_bf16_16x8x16(part[nt], a, b);
    }
  }
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU.  grid (I/16, max active experts), 8 warps split K = H.
// hid[r, i] = silu(g) * u in fp16 for every row r of the expert.
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32)
k_gateup_gemv(const uint16_t* __restrict__ x, int H, int I,
              const int32_t* __restrict__ expert_off, const int32_t* __restrict__ row_token,
              const int32_t* __restrict__ active,
              const uint8_t* __restrict__ gcodes, const float* __restrict__ gscales,
              const uint8_t* __restrict__ ucodes, const float* __restrict__ uscales,
              uint16_t* __restrict__ hid, int32_t* __restrict__ status) {
  __shared__ float red[kGemvWarps][NT][2][4][32];
  __shared__ int tok[NT * 8];
  const int a = blockIdx.y;
  if (a >= active[0]) return;
  const int e = active[1 + a];
  const int r0 = expert_off[e];
  const int ne = expert_off[e + 1] - r0;
  const int i0 = blockIdx.x * 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int nch = H / 64;
  const int nHb = cdiv(H, kScaleBlock);
  const size_t wrow = ((size_t)e * I + i0 + g) * H;
  const uint8_t* gp = gcodes + wrow + 16 * c;
  const uint8_t* up = ucodes + wrow + 16 * c;
  const size_t r8 = (size_t)8 * H;
  const float* gs = gscales + ((size_t)e * cdiv(I, kScaleBlock) + i0 / kScaleBlock) * nHb;
  const float* us = uscales + ((size_t)e * cdiv(I, kScaleBlock) + i0 / kScaleBlock) * nHb;

  for (int n0 = 0; n0 < ne; n0 += NT * 8) {
    if (tid < NT * 8) tok[tid] = (n0 + tid < ne) ? row_token[r0 + n0 + tid] : -1;
    __syncthreads();
    int trow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) trow[nt] = tok[nt * 8 + g];
    float accg[NT][4], accu[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) accg[nt][q] = accu[nt][q] = 0.f;

#pragma unroll 2
    for (int ch = warp; ch < nch; ch += kGemvWarps) {
      const int k0 = ch * 64;
      const uint4 g_lo = ldg_stream16(gp + k0), g_hi = ldg_stream16(gp + r8 + k0);
      const uint4 u_lo = ldg_stream16(up + k0), u_hi = ldg_stream16(up + r8 + k0);
      uint4 xa[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (trow[nt] >= 0) {
          const uint16_t* xp = x + (size_t)trow[nt] * H + k0 + 16 * c;
          xa[nt][0] = ldg16(xp);
          xa[nt][1] = ldg16(xp + 8);
        } else {
          xa[nt][0] = xa[nt][1] = make_uint4(0, 0, 0, 0);
        }
      }
      const float sg = gs[k0 / kScaleBlock] * kPow2_112;
      const float su = us[k0 / kScaleBlock] * kPow2_112;
      float pg[NT][4], pu[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) pg[nt][q] = pu[nt][q] = 0.f;
      chunk_mma<NT, false>(g_lo, g_hi, xa, pg);
      chunk_mma<NT, false>(u_lo, u_hi, xa, pu);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          accg[nt][q] = fmaf(pg[nt][q], sg, accg[nt][q]);
          accu[nt][q] = fmaf(pu[nt][q], su, accu[nt][q]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        red[warp][nt][0][q][lane] = accg[nt][q];
        red[warp][nt][1][q][lane] = accu[nt][q];
      }
    __syncthreads();
    // One output (row, token) per thread: tid = nt*128 + q*32 + L.
    if (tid < NT * 128) {
      const int nt = tid >> 7, q = (tid >> 5) & 3, L = tid & 31;
      float gv = 0.f, uv = 0.f;
#pragma unroll
      for (int w = 0; w < kGemvWarps; ++w) {
        gv += red[w][nt][0][q][L];
        uv += red[w][nt][1][q][L];
      }
      const int row = (L >> 2) + 8 * (q >> 1);
      const int n = n0 + nt * 8 + 2 * (L & 3) + (q & 1);
      if (n < ne) {
        const float hv = gv / (1.f + expf(-gv)) * uv;
        if (!(fabsf(hv) <= kF16Max)) raise_status(status, MOE_DEV_FP16_RANGE);
        hid[(size_t)(r0 + n) * I + i0 + row] = f32_to_f16_bits(hv);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// down projection.  grid (H/128, max active experts); warp w owns output rows
// [h0 + 16w, h0 + 16w + 16) over the whole K = I.
// y[r, h] = sum_i hid[r, i] Wd[h, i] in fp32 for every row r of the expert;
// hid (fp16) times the exactly decoded fp16 weights, block scale in fp32.
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32)
k_down_gemv(const uint16_t* __restrict__ hid, int H, int I,
            const int32_t* __restrict__ expert_off, const int32_t* __restrict__ active,
            const uint8_t* __restrict__ dcodes, const float* __restrict__ dscales,
            float* __restrict__ y) {
  const int a = blockIdx.y;
  if (a >= active[0]) return;
  const int e = active[1 + a];
  const int r0 = expert_off[e];
  const int ne = expert_off[e + 1] - r0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int h0 = blockIdx.x * 128 + warp * 16;
  if (h0 >= H) return;
  const int nch = I / 64;
  const int nIb = cdiv(I, kScaleBlock);
  const uint8_t* dp = dcodes + ((size_t)e * H + h0 + g) * I + 16 * c;
  const size_t r8 = (size_t)8 * I;
  const float* ds = dscales + ((size_t)e * cdiv(H, kScaleBlock) + h0 / kScaleBlock) * nIb;

  for (int n0 = 0; n0 < ne; n0 += NT * 8) {
    bool valid[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) valid[nt] = n0 + nt * 8 + g < ne;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
#pragma unroll 2
    for (int ch = 0; ch < nch; ++ch) {
      const int k0 = ch * 64;
      const uint4 w_lo = ldg_stream16(dp + k0), w_hi = ldg_stream16(dp + r8 + k0);
      uint4 xa[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (valid[nt]) {
          const uint16_t* hp = hid + (size_t)(r0 + n0 + nt * 8 + g) * I + k0 + 16 * c;
          xa[nt][0] = ldg16(hp);
          xa[nt][1] = ldg16(hp + 8);
        } else {
          xa[nt][0] = xa[nt][1] = make_uint4(0, 0, 0, 0);
        }
      }
      const float sd = ds[k0 / kScaleBlock];
      float p[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) p[nt][q] = 0.f;
      chunk_mma<NT, true>(w_lo, w_hi, xa, p);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = fmaf(p[nt][q], sd, acc[nt][q]);
    }
    // C fragment: q=0,1 -> row g, tokens 2c, 2c+1; q=2,3 -> row g+8.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = n0 + nt * 8 + 2 * c + (q & 1);
        const int row = g + 8 * (q >> 1);
        if (n < ne) y[(size_t)(r0 + n) * H + h0 + row] = acc[nt][q];
      }
  }
}

cudaError_t launch_expert_gemv(const uint16_t* x, const int32_t* expert_off,
                               const int32_t* row_token, const int32_t* active, int max_active,
                               const moe_fp8_ffn& w, int H, int I, int max_rows_per_expert,
                               uint16_t* hid, float* y, int32_t* status, cudaStream_t s) {
  if (max_active <= 0) return cudaSuccess;
  const dim3 block(kGemvWarps * 32);
  const dim3 g1(I / 16, max_active), g2(cdiv(H, 128), max_active);
  if (max_rows_per_expert <= 8) {
    k_gateup_gemv<1><<<g1, block, 0, s>>>(x, H, I, expert_off, row_token, active, w.gate.codes,
                                          w.gate.scales, w.up.codes, w.up.scales, hid, status);
    k_down_gemv<1><<<g2, block, 0, s>>>(hid, H, I, expert_off, active, w.down.codes,
                                        w.down.scales, y);
  } else {
    k_gateup_gemv<2><<<g1, block, 0, s>>>(x, H, I, expert_off, row_token, active, w.gate.codes,
                                          w.gate.scales, w.up.codes, w.up.scales, hid, status);
    k_down_gemv<2><<<g2, block, 0, s>>>(hid, H, I, expert_off, active, w.down.codes,
                                        w.down.scales, y);
  }
  return cudaGetLastError();
}

}  // namespace moe
