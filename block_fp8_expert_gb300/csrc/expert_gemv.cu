// Routed-expert FFN for few tokens per expert (decode): a grouped GEMV that
// streams only the selected experts' E4M3 bytes (colizig README, "Features":
// block-FP8 weights, fused decode+FMA dot products; "MoE per-expert
// evaluation").
//
// Streaming: every thread issues all of its weight copies for a work item up
// front as 16-byte cp.async into shared-memory slots that only it reads back
// (slot j of thread t at index j*256 + t: conflict-free, no barrier needed),
// then loads the matching activations straight into registers, waits once and
// computes.  Registers stay low, so several CTAs share an SM and up to
// ~200 KB of weights per SM are in flight, which is what HBM3e needs.
//
// Compute: the codes are decoded in registers and fed to warp-level
// tensor-core MMAs (m16n8k16) whose N side is the expert's tokens, 8 per MMA;
// the tensor core is only a cheap multiply-accumulate here.
//
// K permutation: an MMA's 16 logical K positions are fed from physical
// columns so that a thread owns 16 consecutive bytes of a weight row: for
// thread (g = lane/4, c = lane%4) and MMA step s of a 64-column chunk, the
// logical pairs (2c, 2c+1) and (2c+8, 2c+9) are physical columns
// 16c + 4s + {0,1} and 16c + 4s + {2,3}.  The activations use the same map,
// so every product pairs the right weight with the right activation.
//
// Block scale and range: each 64-column chunk lies inside one 128x128 scale
// block, so the chunk's MMA sum is multiplied by its scale in fp32 and added
// to an fp32 accumulator.  The activations arrive in fp16 scaled per
// (token, chunk) by a power of two (xn = x 2^(14 - e), written once per call
// by the router or launch_x_norm: the largest of the token's 64 values lands
// in [2^14, 2^15), exact because bf16 has fewer mantissa bits than fp16) and
// 2^(e - 14) rejoins the scale in fp32.  The SwiGLU output hid is stored as
// fp16 with one exponent per 16
// features of a row, the down kernel aligns a chunk's four exponents and
// again moves the power of two into the fp32 scale.  So the expert FFN has no
// range limit beyond fp32's: block scales, activations and weights of any
// magnitude keep fp16's relative precision (2^-11) at every rounding.
#include "moe_internal.h"

namespace moe {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// gate/up + SwiGLU.  grid (I/16, max active experts).  A CTA owns 16 rows of
// the expert's gate and up matrices; its 8 warps split K = H into 64-column
// chunks (warp w: chunks w, w+8, ...), kGuChunks per warp per K-group.
// hid[r, i] = silu(g) * u for every row r of the expert, stored as fp16 hid''
// with hid = hid'' 2^(hexp - 14), one exponent per row and 16 features (the
// CTA's 16): hexp[r, i0 / 16].
// ---------------------------------------------------------------------------
constexpr int kGuChunks = 4;  // chunks per warp per K-group: H <= 2048 in one group
constexpr size_t kGuSmem = sizeof(uint4) * kGuChunks * 4 * kThreads;  // 64 KB

template <int NT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 3 : 2)
k_gateup_stream(const uint16_t* __restrict__ xn, const int8_t* __restrict__ xe, int H, int I,
                const int32_t* __restrict__ expert_off, const int32_t* __restrict__ row_token,
                const int32_t* __restrict__ active,
                const uint8_t* __restrict__ gcodes, const float* __restrict__ gscales,
                const uint8_t* __restrict__ ucodes, const float* __restrict__ uscales,
                uint16_t* __restrict__ hid, int8_t* __restrict__ hexp,
                int32_t* __restrict__ status, const SharedExpert sx) {
  extern __shared__ uint4 wbuf[];  // [kGuChunks * 4][kThreads]
  __shared__ float red[8][NT][2][4][32];
  __shared__ int tok[NT * 8];
  griddep_wait();
  griddep_trigger();
  // the last CTA column is the shared expert when there is one
  const bool shared = sx.gc != nullptr && blockIdx.y == gridDim.y - 1;
  int e = 0;
  if (!shared) {
    const int a = blockIdx.y;
    if (a >= active[0]) return;
    e = active[1 + a];
  }
  const int i0 = blockIdx.x * 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int nch = H / 64;
  const int nHb = cdiv(H, kScaleBlock);
  const size_t wrow = ((size_t)e * I + i0 + g) * H;
  const uint8_t* gp = (shared ? sx.gc : gcodes) + wrow + 16 * c;
  const uint8_t* up = (shared ? sx.uc : ucodes) + wrow + 16 * c;
  const size_t r8 = (size_t)8 * H;
  const size_t srow = ((size_t)e * cdiv(I, kScaleBlock) + i0 / kScaleBlock) * nHb;
  const float* gs = (shared ? sx.gs : gscales) + srow;
  const float* us = (shared ? sx.us : uscales) + srow;
  bool bad = false;  // an infinite or NaN input or result
  // All weight copies of one K-group (2048 columns of H).
  auto issue = [&](int kg) {
#pragma unroll
    for (int j = 0; j < kGuChunks; ++j) {
      const int ch = kg + warp + 8 * j;
      if (ch < nch) {
        const int k0 = ch * 64;
        cp_async16_stream(&wbuf[(j * 4 + 0) * kThreads + tid], gp + k0);
        cp_async16_stream(&wbuf[(j * 4 + 1) * kThreads + tid], gp + r8 + k0);
        cp_async16_stream(&wbuf[(j * 4 + 2) * kThreads + tid], up + k0);
        cp_async16_stream(&wbuf[(j * 4 + 3) * kThreads + tid], up + r8 + k0);
      }
      cp_async_commit();  // one group per chunk: chunk j is computed while later ones land
    }
  };
  // The first K-group's weights depend only on the expert: start them before
  // the expert's rows and tokens are read.
  issue(0);
  const int r0 = shared ? sx.row0 : expert_off[e];
  const int ne = shared ? sx.T : expert_off[e + 1] - r0;
  bool issued = true;

  for (int n0 = 0; n0 < ne; n0 += NT * 8) {
    if (tid < NT * 8)
      tok[tid] = (n0 + tid < ne) ? (shared ? n0 + tid : row_token[r0 + n0 + tid]) : -1;
    __syncthreads();
    int trow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) trow[nt] = tok[nt * 8 + g];
    float accg[NT][4], accu[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) accg[nt][q] = accu[nt][q] = 0.f;

    for (int kg = 0; kg < nch; kg += 8 * kGuChunks) {
      // 1. all weight copies of this K-group (unless already in flight)
      if (!issued) issue(kg);
      issued = false;
      // 2. block scales and activations (fp16 and their exponents), straight
      // into registers
      float sg[kGuChunks], su[kGuChunks];
      uint4 xa[kGuChunks][NT][2];
      int xx[kGuChunks][NT];
#pragma unroll
      for (int j = 0; j < kGuChunks; ++j) {
        const int ch = kg + warp + 8 * j;
        sg[j] = ch < nch ? gs[ch * 64 / kScaleBlock] : 0.f;
        su[j] = ch < nch ? us[ch * 64 / kScaleBlock] : 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (ch < nch && trow[nt] >= 0) {
            const uint16_t* xp = xn + (size_t)trow[nt] * H + ch * 64 + 16 * c;
            xa[j][nt][0] = ldg16(xp);
            xa[j][nt][1] = ldg16(xp + 8);
            xx[j][nt] = xe[(size_t)trow[nt] * nch + ch];
          } else {
            xa[j][nt][0] = xa[j][nt][1] = make_uint4(0, 0, 0, 0);
            xx[j][nt] = kExpFloor;
          }
        }
      }
      // 3. per chunk as its copies land: decode + MMA, then block scale and
      // the activations' power of two in fp32
#pragma unroll
      for (int j = 0; j < kGuChunks; ++j) {
        const int ch = kg + warp + 8 * j;  // warp-uniform
        cp_async_wait_n(kGuChunks - 1 - j);
        if (ch < nch) {
          if (!(fabsf(sg[j]) <= FLT_MAX) || !(fabsf(su[j]) <= FLT_MAX)) bad = true;
          // factors of the accumulator columns (tokens 2c, 2c + 1 of 8)
          float fg[NT][2], fu[NT][2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int e0 = __shfl_sync(0xffffffffu, xx[j][nt], 8 * c) - kGroupTop;
            const int e1 = __shfl_sync(0xffffffffu, xx[j][nt], 8 * c + 4) - kGroupTop;
            fg[nt][0] = sg[j] * pow2f(e0);
            fg[nt][1] = sg[j] * pow2f(e1);
            fu[nt][0] = su[j] * pow2f(e0);
            fu[nt][1] = su[j] * pow2f(e1);
          }
          float pg[NT][4], pu[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) pg[nt][q] = pu[nt][q] = 0.f;
          chunk_mma<NT, true>(wbuf[(j * 4 + 0) * kThreads + tid],
                              wbuf[(j * 4 + 1) * kThreads + tid], xa[j], pg);
          chunk_mma<NT, true>(wbuf[(j * 4 + 2) * kThreads + tid],
                              wbuf[(j * 4 + 3) * kThreads + tid], xa[j], pu);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              accg[nt][q] = fmaf(pg[nt][q], fg[nt][q & 1], accg[nt][q]);
              accu[nt][q] = fmaf(pu[nt][q], fu[nt][q & 1], accu[nt][q]);
            }
        }
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
    // One output per thread: half-warp h = tid / 16 is token n0 + h, lane f
    // of it feature i0 + f (accumulator element: row f = (L >> 2) + 8 (q >> 1),
    // token 2 (L & 3) + (q & 1) of group nt).
    if (tid < NT * 128) {
      const int nl = tid >> 4, f = tid & 15;
      const int nt = nl >> 3, nn = nl & 7;
      const int q = ((f >> 3) << 1) | (nn & 1), L = ((f & 7) << 2) | (nn >> 1);
      float gv = 0.f, uv = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        gv += red[w][nt][0][q][L];
        uv += red[w][nt][1][q][L];
      }
      const int n = n0 + nl;
      const float hv = gv / (1.f + expf(-gv)) * uv;
      // the token's 16 features: largest magnitude over the half-warp
      uint32_t m = __float_as_uint(hv) & 0x7fffffffu;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int E = min(exp_of_bits(m), 127);
      if (n < ne) {
        if (m >= 0x7f800000u) bad = true;
        hid[(size_t)(r0 + n) * I + i0 + f] = f32_to_f16_bits(hv * pow2f(kGroupTop - E));
        if (f == 0) hexp[(size_t)(r0 + n) * (I / 16) + i0 / 16] = (int8_t)E;
      }
    }
    __syncthreads();
  }
  if (bad) raise_status(status, MOE_DEV_NONFINITE);
}

// ---------------------------------------------------------------------------
// down projection.  grid (H/32, max active experts).  A CTA owns 32 output
// rows (two 16-row MMA tiles); warp w works on tile w & 1 and K-part w >> 1 of
// 4 (chunks kp, kp+4, ...), kDnChunks per warp per K-group.
// y[r, h] = sum_i hid[r, i] Wd[h, i], summed in fp32, for every row r of the
// expert; stored in fp32, or (YH) as fp16 y'' with y = y'' 2^s and one
// exponent s per row and 32 columns (the CTA's 32): yexp[h / 32][r], the
// table being [H / 32][y_rows].
// FUSE (cmb.ticket set; YH only; T <= 64, k <= 8): the last CTA of each 32-row
// slice of h — one ticket per slice, counted up to the number of active
// experts — also combines that slice for every token, with the combine
// kernel's arithmetic (fp32 fmaf over the slots in order j, rounded once to
// bf16), so no combine launch follows.  A thread per (token, 8 columns)
// loads its token's slot rows and weights before the ticket, leaving one
// round trip (the y rows) after it.
// ---------------------------------------------------------------------------
constexpr int kDnChunks = 3;  // I <= 768 in one K-group
constexpr size_t kDnSmem = sizeof(uint4) * kDnChunks * 2 * kThreads;  // 24 KB

template <int NT, bool YH, bool FUSE = false>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 4 : 3)
k_down_stream(const uint16_t* __restrict__ hid, const int8_t* __restrict__ hexp, int H, int I,
              const int32_t* __restrict__ expert_off, const int32_t* __restrict__ active,
              const uint8_t* __restrict__ dcodes, const float* __restrict__ dscales,
              void* __restrict__ y, int16_t* __restrict__ yexp, int y_rows,
              int32_t* __restrict__ status, const FusedCombine cmb, const SharedExpert sx) {
  extern __shared__ uint4 wbuf[];  // [kDnChunks * 2][kThreads]
  __shared__ float red[4][2][NT][4][32];
  __shared__ int is_last;
  // The active list and the offsets come from the permutation, which had
  // completed before the previous kernel (gate/up) passed its own
  // griddep_wait; they and the weights are read before this kernel waits for
  // gate/up, so the first K-group's weights stream while gate/up finishes.
  // Everything gate/up writes (hid and its exponents) is read after the wait.
  // the last CTA column is the shared expert when there is one
  const bool shared = sx.gc != nullptr && blockIdx.y == gridDim.y - 1;
  int e = 0;
  if (!shared) {
    const int a = blockIdx.y;
    if (a >= active[0]) return;
    e = active[1 + a];
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int mt = warp & 1, kp = warp >> 1;
  const int h0 = blockIdx.x * 32 + mt * 16;
  const int nch = I / 64;
  const int nIb = cdiv(I, kScaleBlock);
  const uint8_t* dp = (shared ? sx.dc : dcodes) + ((size_t)e * H + h0 + g) * I + 16 * c;
  const size_t r8 = (size_t)8 * I;
  const float* ds = (shared ? sx.ds : dscales) +
                    ((size_t)e * cdiv(H, kScaleBlock) + h0 / kScaleBlock) * nIb;
  bool bad = false;
  // All weight copies of one K-group (768 columns of I).
  auto issue = [&](int kg) {
#pragma unroll
    for (int j = 0; j < kDnChunks; ++j) {
      const int ch = kg + kp + 4 * j;
      if (ch < nch) {
        cp_async16_stream(&wbuf[(j * 2 + 0) * kThreads + tid], dp + ch * 64);
        cp_async16_stream(&wbuf[(j * 2 + 1) * kThreads + tid], dp + r8 + ch * 64);
      }
      cp_async_commit();  // one group per chunk
    }
  };
  // The first K-group's weights depend only on the expert: start them before
  // the expert's rows are read.
  issue(0);
  griddep_wait();
  griddep_trigger();
  const int r0 = shared ? sx.row0 : expert_off[e];
  const int ne = shared ? sx.T : expert_off[e + 1] - r0;
  bool issued = true;

  for (int n0 = 0; n0 < ne; n0 += NT * 8) {
    bool valid[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) valid[nt] = n0 + nt * 8 + g < ne;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
    for (int kg = 0; kg < nch; kg += 4 * kDnChunks) {
      if (!issued) issue(kg);
      issued = false;
      float sd[kDnChunks];
      uint4 xa[kDnChunks][NT][2];
      int hx[kDnChunks][NT];
#pragma unroll
      for (int j = 0; j < kDnChunks; ++j) {
        const int ch = kg + kp + 4 * j;
        sd[j] = ch < nch ? ds[ch * 64 / kScaleBlock] : 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (ch < nch && valid[nt]) {
            // this thread's 16 features are exactly one exponent group
            const size_t row = (size_t)(r0 + n0 + nt * 8 + g);
            const uint16_t* hp = hid + row * I + ch * 64 + 16 * c;
            xa[j][nt][0] = ldg16(hp);
            xa[j][nt][1] = ldg16(hp + 8);
            hx[j][nt] = hexp[row * (I / 16) + ch * 4 + c];
          } else {
            xa[j][nt][0] = xa[j][nt][1] = make_uint4(0, 0, 0, 0);
            hx[j][nt] = kExpFloor;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kDnChunks; ++j) {
        const int ch = kg + kp + 4 * j;  // warp-uniform
        cp_async_wait_n(kDnChunks - 1 - j);
        if (ch < nch) {
          if (!(fabsf(sd[j]) <= FLT_MAX)) bad = true;
          float fd[NT][2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int m = f16x16_align(xa[j][nt], hx[j][nt]);
            fd[nt][0] = sd[j] * pow2f(__shfl_sync(0xffffffffu, m, 8 * c) - kGroupTop);
            fd[nt][1] = sd[j] * pow2f(__shfl_sync(0xffffffffu, m, 8 * c + 4) - kGroupTop);
          }
          float p[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) p[nt][q] = 0.f;
          chunk_mma<NT, true>(wbuf[(j * 2 + 0) * kThreads + tid],
                              wbuf[(j * 2 + 1) * kThreads + tid], xa[j], p);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[nt][q] = fmaf(p[nt][q], fd[nt][q & 1], acc[nt][q]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) red[kp][mt][nt][q][lane] = acc[nt][q];
    __syncthreads();
    // outputs: warp (o / 32) is token n0 + o / 32, lane f of it column
    // 32 blockIdx.x + f (accumulator element: tile f / 16, row (L >> 2) +
    // 8 (q >> 1) = f % 16, token 2 (L & 3) + (q & 1) of group nt)
    for (int o = tid; o < NT * 256; o += kThreads) {
      const int nl = o >> 5, f = o & 31;
      const int t2 = f >> 4, row = f & 15, nt = nl >> 3, nn = nl & 7;
      const int q = ((row >> 3) << 1) | (nn & 1), L = ((row & 7) << 2) | (nn >> 1);
      float v = 0.f;
#pragma unroll
      for (int p = 0; p < 4; ++p) v += red[p][t2][nt][q][L];
      const int n = n0 + nl;
      if (n < ne) {  // warp-uniform
        const size_t at = (size_t)(r0 + n) * H + blockIdx.x * 32 + f;
        if (YH) {
          const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu);
          if (m >= 0x7f800000u) bad = true;
          const int E = min(exp_of_bits(m), 127);
          static_cast<uint16_t*>(y)[at] = f32_to_f16_bits(v * pow2f(kGroupTop - E));
          if (f == 0) yexp[(size_t)blockIdx.x * y_rows + r0 + n] = (int16_t)(E - kGroupTop);
        } else {
          static_cast<float*>(y)[at] = v;
        }
      }
    }
    __syncthreads();
  }
  if (bad) raise_status(status, MOE_DEV_NONFINITE);
  if constexpr (YH && FUSE) {
    {
      const int t = tid >> 2, h = blockIdx.x * 32 + (tid & 3) * 8;
      const bool mine = t < cmb.T;
      int row[8];
      float wt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool ok = mine && j < cmb.k;
        row[j] = ok ? cmb.tok_slot_row[t * cmb.k + j] : -1;
        wt[j] = ok ? cmb.topk_w[t * cmb.k + j] : 0.f;
      }
      // the CTA's y stores (ordered by the barrier) are released device-wide
      // before its ticket counts; the last ticket acquires everyone's
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const int ctas = active[0] + (sx.gc ? 1 : 0);  // the slice's CTAs of this launch
        is_last = atomicAdd(&cmb.ticket[blockIdx.x], 1) == ctas - 1;
        __threadfence();
      }
      __syncthreads();
      if (is_last && mine) {
        // the slot rows stay packed (8 fp16 in 16 bytes) until they are used
        uint4 yr[8];
        int ys[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (row[j] >= 0) {
            yr[j] = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) +
                                                          (size_t)row[j] * H + h));
            ys[j] = __ldcg(yexp + (size_t)blockIdx.x * y_rows + row[j]);
          } else {
            yr[j] = make_uint4(0, 0, 0, 0);
            ys[j] = 0;
          }
        }
        float r[8], acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = acc[i] = 0.f;
        if (sx.gc) {
          // the shared expert's row (weight 1, exact), first
          const size_t srow = (size_t)sx.row0 + t;
          const uint4 sr = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) +
                                                                 srow * H + h));
          float f = ldexp2f(1.f, __ldcg(yexp + (size_t)blockIdx.x * y_rows + srow));
          if (cmb.sgate) f *= cmb.sgate[t];  // gated shared expert
          unpack_f16x8(sr, acc);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] *= f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (row[j] < 0) continue;
          // w 2^s is exact, so fmaf(w 2^s, y'', r) rounds w y + r once
          const float wf = ldexp2f(wt[j], ys[j]);
          float yv[8];
          unpack_f16x8(yr[j], yv);
#pragma unroll
          for (int i = 0; i < 8; ++i) r[i] = fmaf(wf, yv[i], r[i]);
        }
        uint32_t o4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o4[i] = pack_bf16x2(acc[2 * i] + r[2 * i], acc[2 * i + 1] + r[2 * i + 1]);
        *reinterpret_cast<uint4*>(cmb.out + (size_t)t * H + h) =
            make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  }
}

bool fused_combine_ok(int T, int k, int H, int max_active) {
  // a thread per (token, 8 columns of the slice), at most 8 slots, and the
  // down grid in one wave (a fenced ticket per CTA costs a round trip that
  // later waves would queue behind)
  const long long ctas = (long long)(H / 32) * max_active;
  return T >= 1 && T * 4 <= kThreads && k >= 1 && k <= 8 && H % 32 == 0 &&
         ctas <= (long long)num_sms() * 4;
}

// xn = x 2^(14 - e), xe = e per (token, 64 columns): thread 16 values,
// the quad of lanes 4g .. 4g + 3 one chunk (T H / 16 threads, launched as
// whole warps: threads past the end take part in the shuffles with zeros).
__global__ void __launch_bounds__(256)
k_x_norm(const uint16_t* __restrict__ x, long long n16, int H, uint16_t* __restrict__ xn,
         int8_t* __restrict__ xe) {
  griddep_wait();
  griddep_trigger();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool in = i < n16;
  uint4 v[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  if (in) {
    v[0] = ldg16(x + 16 * i);
    v[1] = ldg16(x + 16 * i + 8);
  }
  bool bad = false;  // a non-finite x shows in the expert kernels' results
  const int e = bf16x16_to_f16_norm(v, bad);
  if (!in) return;
  uint4* dst = reinterpret_cast<uint4*>(xn + 16 * i);
  dst[0] = v[0];
  dst[1] = v[1];
  if ((i & 3) == 0) xe[i >> 2] = (int8_t)min(e, 127);  // chunk (16 i) / 64 of the row-major array
}

cudaError_t launch_x_norm(const uint16_t* x, int T, int H, uint16_t* xn, int8_t* xe,
                          cudaStream_t s, bool pdl) {
  const long long n16 = (long long)T * H / 16;
  if (n16 == 0) return cudaSuccess;
  return launch_k(k_x_norm, dim3((unsigned)((n16 + 255) / 256)), dim3(256), 0, s, pdl, x, n16, H,
                  xn, xe);
}

cudaError_t launch_expert_gemv(const uint16_t* xn, const int8_t* xe, const int32_t* expert_off,
                               const int32_t* row_token, const int32_t* active, int max_active,
                               const moe_fp8_ffn& w, int H, int I, int tokens_per_expert_hint,
                               uint16_t* hid, int8_t* hexp, void* y, int16_t* yexp, int y_rows,
                               int32_t* status, cudaStream_t s, bool pdl,
                               const FusedCombine& cmb, const SharedExpert& sx) {
  const int cols = max_active + (sx.gc ? 1 : 0);  // CTA columns: experts (+ the shared one)
  if (cols <= 0) return cudaSuccess;
  if (cmb.ticket && (!yexp || !fused_combine_ok(cmb.T, cmb.k, H, cols)))
    return cudaErrorInvalidValue;
  cudaError_t e;
  const bool nt1 = tokens_per_expert_hint <= 8;
  const dim3 block(kThreads);
  const dim3 g1(I / 16, cols), g2(H / 32, cols);
  auto down = [&](auto kern) -> cudaError_t {
    cudaError_t err = ensure_smem((const void*)kern, kDnSmem);
    if (err != cudaSuccess) return err;
    return launch_k(kern, g2, block, kDnSmem, s, pdl, (const uint16_t*)hid, (const int8_t*)hexp,
                    H, I, expert_off, active, w.down.codes, w.down.scales, y, yexp, y_rows,
                    status, cmb, sx);
  };
  if (nt1) {
    if ((e = ensure_smem((const void*)k_gateup_stream<1>, kGuSmem)) != cudaSuccess) return e;
    e = launch_k(k_gateup_stream<1>, g1, block, kGuSmem, s, pdl, xn, xe, H, I, expert_off,
                 row_token, active, w.gate.codes, w.gate.scales, w.up.codes, w.up.scales, hid,
                 hexp, status, sx);
    if (e != cudaSuccess) return e;
    if (cmb.ticket) return down(k_down_stream<1, true, true>);
    return yexp ? down(k_down_stream<1, true>) : down(k_down_stream<1, false>);
  }
  if ((e = ensure_smem((const void*)k_gateup_stream<2>, kGuSmem)) != cudaSuccess) return e;
  e = launch_k(k_gateup_stream<2>, g1, block, kGuSmem, s, pdl, xn, xe, H, I, expert_off,
               row_token, active, w.gate.codes, w.gate.scales, w.up.codes, w.up.scales, hid, hexp,
               status, sx);
  if (e != cudaSuccess) return e;
  if (cmb.ticket) return down(k_down_stream<2, true, true>);
  return yexp ? down(k_down_stream<2, true>) : down(k_down_stream<2, false>);
}

}  // namespace moe
