// Router logits on the 5th-generation tensor cores, for 128 tokens or more
// (colizig README, model table: experts with top-k routing; the logits are
// l = x Wr^T before the bias).
//
// The fp32 router weights are split once per call into three bf16 planes
// (w = hi + mid + lo to within 2^-24 |w|); bf16 activations are exact, so
// three bf16 MMAs accumulating in fp32 give fp32-accurate logits.  A CTA owns
// 128 experts (the MMA's M, A = the three weight planes) x 128 tokens (N,
// B = x) x one of KS slices of K = H, with operands staged by TMA in a
// three-deep ring:
//   warp 0      TMA: the step's x tile and its three weight tiles;
//   warp 1      one elected thread issues tcgen05.mma (lo, mid, hi per
//               16-wide K step) into one TMEM accumulator [128 x 128] fp32;
//   warps 2-5   when xn is set (CTAs of the first expert tile): turn the
//               step's x tile into the streamed expert kernels' activations
//               (xn = fp16(x 2^(14 - e)), one e = xe per token and 64
//               columns); then write the slice's partial logits
//               part[ks][t][e].
// The top-k kernel adds the KS slices in a fixed order (deterministic).
#include <cuda.h>

#include <algorithm>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {
constexpr int RT = 128;   // tokens per CTA (MMA N)
constexpr int RE = 128;   // experts per CTA (MMA M)
constexpr int RBK = 64;   // K per step
constexpr int RNS = 3;    // ring depth
constexpr int R_TILE = RT * RBK * 2;        // 16 KB: x tile or one weight tile
constexpr int R_STAGE = 4 * R_TILE;         // x + three weight planes
constexpr int R_SMEM = RNS * R_STAGE + 1024;  // + alignment slack
constexpr int kRWarps = 6;

struct RouterShared {
  uint64_t full[RNS], empty[RNS], done;
  uint32_t tmem_base;
  int abort_flag;
};

// Warp-uniform bounded wait (see the grouped GEMM): gives up together once
// the budget is spent or another role has given up, recording
// MOE_DEV_WAIT_TIMEOUT.
__device__ __forceinline__ bool rwait(RouterShared& sh, uint64_t* bar, uint32_t parity,
                                      int32_t* status) {
  constexpr unsigned kAll = 0xffffffffu;
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(kAll, done)) return true;
  const WaitBudget b = wait_budget();
  for (uint32_t n = 1;; ++n) {
    if (__any_sync(kAll, done)) {
      for (int r = 0; !done && r < (1 << 16); ++r) done = mbar_try_wait(bar, parity);
      if (__all_sync(kAll, done)) return true;
      break;
    }
    if ((n & 31) == 0) {
      const bool give_up = *reinterpret_cast<volatile int*>(&sh.abort_flag) != 0 || budget_spent(b);
      if (__any_sync(kAll, give_up)) break;
    }
    done = mbar_try_wait(bar, parity);
  }
  if ((threadIdx.x & 31) == 0 && !sh.abort_flag) {
    sh.abort_flag = 1;
    raise_status(status, MOE_DEV_WAIT_TIMEOUT);
  }
  __syncwarp();
  return false;
}

// Instruction descriptor, kind::f16 with bf16 A and B (K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
}  // namespace

// Wr [E, H] fp32 -> planes [3][E][H] bf16 (hi, mid, lo).  The first kernel of
// a routed call on this path: it also clears the status words.
__global__ void __launch_bounds__(256)
k_router_split(const float* __restrict__ Wr, long long n, uint16_t* __restrict__ planes,
               int32_t* __restrict__ status) {
  griddep_wait();
  griddep_trigger();
  if (status && blockIdx.x == 0 && threadIdx.x < kStatusWords) status[threadIdx.x] = 0;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    uint32_t hi, mid, lo;
    split3_bf16(__ldg(Wr + i), hi, mid, lo);
    planes[i] = (uint16_t)hi;
    planes[n + i] = (uint16_t)mid;
    planes[2 * n + i] = (uint16_t)lo;
  }
}

__global__ void __launch_bounds__(kRWarps * 32, 1)
k_router_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
            int T, int H, int E, int kslice, float* __restrict__ part,
            uint16_t* __restrict__ xn, int8_t* __restrict__ xe, int32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ RouterShared sh;
  griddep_wait();
  griddep_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * RT, ks = blockIdx.y, e0 = blockIdx.z * RE;
  const int k0 = ks * kslice, nsteps = kslice / RBK;
  const bool convert = xn != nullptr && blockIdx.z == 0;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t smem_base = smem_u32(smem);
  if (tid == 0) {
    for (int s = 0; s < RNS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], convert ? 5 : 1);  // the MMA's commit (+ 4 converter warps)
    }
    mbar_init(&sh.done, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&sh.tmem_base, RT);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA
    int s = 0;
    for (; s < nsteps; ++s) {
      const int st = s % RNS;
      if (s >= RNS && !rwait(sh, &sh.empty[st], (uint32_t)(((s / RNS) - 1) & 1), status)) break;
      // the converters' reads of this slot (generic proxy) are ordered
      // before the copies that overwrite it (async proxy)
      tc::fence_proxy_async();
      if (tc::elect_one()) {
        uint8_t* dst = smem + st * R_STAGE;
        const int kx = k0 + s * RBK;
        mbar_arrive_expect_tx(&sh.full[st], R_STAGE);
        tc::tma_load_2d(dst, &xmap, kx, t0, &sh.full[st]);
#pragma unroll
        for (int p = 0; p < 3; ++p)
          tc::tma_load_2d(dst + (1 + p) * R_TILE, &wmap, kx, p * E + e0, &sh.full[st]);
      }
      __syncwarp();
    }
    // drain: the copies of the last steps issued must have landed
    if (lane == 0)
      for (int i = max(0, s - RNS); i < s; ++i) mbar_wait(&sh.full[i % RNS], (uint32_t)((i / RNS) & 1));
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA
    const uint32_t idesc = idesc_bf16_f32(RE, RT);
    int s = 0;
    for (; s < nsteps; ++s) {
      const int st = s % RNS;
      if (!rwait(sh, &sh.full[st], (uint32_t)((s / RNS) & 1), status)) break;
      tc::fence_after_sync();
      if (tc::elect_one()) {
        const uint32_t xs = smem_base + st * R_STAGE;
#pragma unroll
        for (int kk = 0; kk < RBK / 16; ++kk) {
          const uint64_t bdesc = tc::sw128_desc(xs + kk * 32);
#pragma unroll
          for (int p = 2; p >= 0; --p) {  // lo, mid, hi: smallest part first
            const uint64_t adesc = tc::sw128_desc(xs + (1 + p) * R_TILE + kk * 32);
            tc::mma_f16(tmem, adesc, bdesc, idesc, (s > 0 || kk > 0 || p < 2) ? 1u : 0u);
          }
        }
        tc::commit(&sh.empty[st]);
        if (s == nsteps - 1) tc::commit(&sh.done);
      }
      __syncwarp();
    }
    // drain: every MMA issued has completed once the newest commit has
    if (lane == 0 && s > 0) mbar_wait(&sh.empty[(s - 1) % RNS], (uint32_t)(((s - 1) / RNS) & 1));
    __syncwarp();
  } else {
    // ------------------------------------------------ activations, then logits
    const int q = warp & 3;  // TMEM lane quarter: experts e0 + 32 q + lane
    bool ok = true;
    if (convert) {
      // row r = 32 (warp - 2) + lane of each x tile: its 64 bf16 values
      const int r = 32 * (warp - 2) + lane;
      for (int s = 0; s < nsteps; ++s) {
        const int st = s % RNS;
        if (!rwait(sh, &sh.full[st], (uint32_t)((s / RNS) & 1), status)) {
          ok = false;
          break;
        }
        if (t0 + r < T) {
          const uint8_t* row = smem + st * R_STAGE + r * 128;
          uint4 v[8];
          uint32_t m = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[j] = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) m = max(m, max(w[u] & 0x7FFFu, (w[u] >> 16) & 0x7FFFu));
          }
          // a non-finite x shows in the expert kernels' results
          const int ex = min(exp_of_bits(m << 16), 127);
          const float f = pow2f(kGroupTop - ex);
          uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)(t0 + r) * H + k0 + s * RBK);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            dst[j] = make_uint4(pack_f16x2(bf16_lo(w[0]) * f, bf16_hi(w[0]) * f),
                                pack_f16x2(bf16_lo(w[1]) * f, bf16_hi(w[1]) * f),
                                pack_f16x2(bf16_lo(w[2]) * f, bf16_hi(w[2]) * f),
                                pack_f16x2(bf16_lo(w[3]) * f, bf16_hi(w[3]) * f));
          }
          xe[(size_t)(t0 + r) * (H / 64) + (k0 + s * RBK) / 64] = (int8_t)ex;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[st]);
      }
    }
    if (ok && rwait(sh, &sh.done, 0, status)) {
      tc::fence_after_sync();
      const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16);
      const int e = e0 + 32 * q + lane;
      float* out = part + ((size_t)ks * T + t0) * E + e;
#pragma unroll 1
      for (int c = 0; c < RT / 32; ++c) {
        uint32_t v[32];
        tc::ld_32x32b_x32(t_lane + 32 * c, v);
        tc::wait_ld();
        const int nv = min(32, T - t0 - 32 * c);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nv && e < E) out[(size_t)(32 * c + j) * E] = __uint_as_float(v[j]);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, RT);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool router_tc_ok(int T, int H, int E) {
  return T >= RT && E % RE == 0 && E <= kMaxExperts && H % RBK == 0;
}

cudaError_t launch_router_logits_tc(const uint16_t* x, const float* Wr, int T, int H, int E,
                                    int KS, float* part, uint16_t* planes, uint16_t* xn,
                                    int8_t* xe, int32_t* status, cudaStream_t s, bool pdl) {
  cudaError_t err = ensure_smem((const void*)k_router_tc, R_SMEM);
  if (err != cudaSuccess) return err;
  CUtensorMap xmap, wmap;
  // x [T, H] and the planes [3E, H], bf16: 64 columns x 128 rows per box,
  // 128-byte swizzled (the K-major operand layout of the MMA)
  if ((err = make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, T, H, RBK, RT,
                                128)) != cudaSuccess)
    return err;
  if ((err = make_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, planes, 3LL * E, H,
                                RBK, RE, 128)) != cudaSuccess)
    return err;
  const long long n = (long long)E * H;
  const long long nblk = std::min<long long>(4LL * num_sms(), (n + 255) / 256);
  err = launch_k(k_router_split, dim3((unsigned)nblk), dim3(256), 0, s, pdl, Wr, n, planes,
                 status);
  if (err != cudaSuccess) return err;
  return launch_k(k_router_tc, dim3(cdiv(T, RT), KS, E / RE), dim3(kRWarps * 32), (size_t)R_SMEM,
                  s, pdl, xmap, wmap, T, H, E, H / KS, part, xn, xe, status);
}

}  // namespace moe
