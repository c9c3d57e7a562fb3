// Device helpers shared by the kernels of the block-FP8 MoE layer (sm_103a).
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_fp8.h"

namespace moe {

constexpr int kScaleBlock = 128;  // edge of one block-FP8 scale block

// 2^112 as a float: the register decode below yields dec(code) * 2^-112, and
// the block scale applied after the MMA carries the 2^112 back.
constexpr float kPow2_112 = 5.192296858534828e33f;

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// bf16 helpers (bf16 = top half of an IEEE binary32)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two floats -> bf16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// E4M3 decode in registers
// ---------------------------------------------------------------------------
// Two E4M3 codes (bits 0..7 = element 0, bits 8..15 = element 1) -> f16x2.
// Every E4M3 value, subnormals included, is an f16 normal or zero, so this is
// exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const unsigned short v = static_cast<unsigned short>(two_codes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// f16x2 holding E4M3-derived values -> bf16x2 holding the same values times
// 2^-112, exactly.  Such an f16 has only its top 3 mantissa bits set, so
// moving exponent and mantissa down by 3 bits re-reads the f16 exponent field
// (bias 15) as a bf16 exponent field (bias 127); the sign stays in place and
// zero stays zero.  Two integer instructions, no float conversion.
__device__ __forceinline__ uint32_t f16x2_e4m3_to_bf16x2_scaled(uint32_t h) {
  return ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
}

// 16 E4M3 codes (one 16-byte load) -> 8 bf16x2 registers holding
// dec(code) * 2^-112; out[m] holds elements 2m (low half) and 2m+1.
__device__ __forceinline__ void decode16_scaled(const uint4& c, uint32_t (&out)[8]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    out[2 * q + 0] = f16x2_e4m3_to_bf16x2_scaled(e4m3x2_to_f16x2(w[q] & 0xFFFFu));
    out[2 * q + 1] = f16x2_e4m3_to_bf16x2_scaled(e4m3x2_to_f16x2(w[q] >> 16));
  }
}

// 16 E4M3 codes -> 8 f16x2 registers holding dec(code) exactly.
__device__ __forceinline__ void decode16_f16(const uint4& c, uint32_t (&out)[8]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    out[2 * q + 0] = e4m3x2_to_f16x2(w[q] & 0xFFFFu);
    out[2 * q + 1] = e4m3x2_to_f16x2(w[q] >> 16);
  }
}

// float -> fp16 bits, round to nearest even (saturates to inf beyond 65504).
__device__ __forceinline__ uint16_t f32_to_f16_bits(float v) {
  unsigned short r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

constexpr float kF16Max = 65504.f;

// Two floats -> f16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// Power-of-two range normalisation of the fp16 intermediates
// ---------------------------------------------------------------------------
// A group of values v is stored as fp16 v'' with v = v'' 2^(E - kGroupTop),
// E = floor(log2) of the group's largest magnitude: that magnitude lands in
// [2^14, 2^15), so every member within 2^-28 of it keeps fp16's full 11-bit
// precision whatever the group's own magnitude.  Multiplying by a power of
// two is exact, so only the one fp16 rounding remains.
constexpr int kGroupTop = 14;
// E is clamped below at kExpFloor (a group whose largest magnitude is under
// 2^-100 is scaled as if it were 2^-100; its members stay representable).
constexpr int kExpFloor = -100;

// 2^n as a float for n in [-126, 127].
__device__ __forceinline__ float pow2f(int n) { return __int_as_float((n + 127) << 23); }

// v 2^n for any int n, in two exact power-of-two steps (each within fp32's
// normal exponents): the result rounds only where it leaves fp32's normal
// range, where it becomes subnormal, zero or infinite as v 2^n would.
__device__ __forceinline__ float ldexp2f(float v, int n) {
  n = min(max(n, -252), 252);
  const int h = n / 2;
  return v * pow2f(h) * pow2f(n - h);
}

// floor(log2 |v|) from the magnitude bits of a float, clamped to
// [kExpFloor, 128] (128: infinity or NaN).
__device__ __forceinline__ int exp_of_bits(uint32_t absbits) {
  return max((int)(absbits >> 23) - 127, kExpFloor);
}

// fp16 bits of 2^d for d <= 0: subnormal below 2^-14, zero below 2^-24.
__device__ __forceinline__ uint32_t f16_pow2_bits(int d) {
  if (d >= -14) return (uint32_t)(d + 15) << 10;
  if (d >= -24) return 1u << (d + 24);
  return 0u;
}

// floor(log2) of the largest magnitude among the warp's values (magnitude
// bits, one per lane), clamped to [-126, 126]; 0 when every value is zero or
// fp32-subnormal.  Sets `bad` when one is infinite or NaN.  Warp-uniform; all
// 32 lanes must call it.
__device__ __forceinline__ int warp_max_exp(uint32_t absbits, bool& bad) {
  const uint32_t m = __reduce_max_sync(0xffffffffu, absbits);
  if (m >= 0x7f800000u) bad = true;
  if (m < 0x00800000u) return 0;
  return min(max((int)(m >> 23) - 127, -126), 126);
}

// Largest magnitude bits among n floats at p, this lane's share (lane i
// reads p[i], p[i + 32], ...), four independent loads per round so that one
// memory round trip covers up to 128 floats.
__device__ __forceinline__ uint32_t lane_max_bits(const float* __restrict__ p, int n, int lane) {
  uint32_t m = 0;
  for (int i = lane; i < n; i += 128) {
    uint32_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = i + 32 * u < n ? __float_as_uint(__ldg(p + i + 32 * u)) & 0x7fffffffu : 0u;
    m = max(m, max(max(v[0], v[1]), max(v[2], v[3])));
  }
  return m;
}

// warp_max_exp over n floats at p.
__device__ __forceinline__ int warp_max_exp_of(const float* __restrict__ p, int n, int lane,
                                               bool& bad) {
  return warp_max_exp(lane_max_bits(p, n, lane), bad);
}

// Column exponents of a 32 x 32 tile held one row per lane (v[i] = column
// i of this lane's row): on return every lane's ex[k] holds, in byte j, the
// largest biased fp32 exponent of column 4k + j over the 32 rows (255: an
// infinite or NaN value).  The exponent of a column's largest magnitude is
// the largest of its exponents, so this is exact.  Eight words of four
// bytes, five butterfly rounds of shuffles and byte-wise maxima.
__device__ __forceinline__ void column_max_exponents(const uint32_t (&v)[32], uint32_t (&ex)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    // the biased exponent is byte 3 of (bits << 1)
    const uint32_t ab = __byte_perm(v[4 * k] << 1, v[4 * k + 1] << 1, 0x0073);
    const uint32_t cd = __byte_perm(v[4 * k + 2] << 1, v[4 * k + 3] << 1, 0x0073);
    ex[k] = __byte_perm(ab, cd, 0x5410);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < 8; ++k) ex[k] = __vmaxu4(ex[k], __shfl_xor_sync(0xffffffffu, ex[k], o));
}

// 16 bf16 activations of one token (two 16-byte registers, 8 bf16x2) turned
// in place into f16x2 holding x 2^(kGroupTop - E), E = floor(log2) of the
// largest magnitude over the quad of lanes 4g .. 4g + 3 that holds the
// token's 64 columns of a chunk (the MMA's B fragment).  Returns E (the same
// in the four lanes); sets `bad` when a value is infinite or NaN.
__device__ __forceinline__ int bf16x16_to_f16_norm(uint4 (&v)[2], bool& bad) {
  uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  if (m >= 0x7F80u) bad = true;
  const int E = exp_of_bits(m << 16);
  const float f = pow2f(kGroupTop - min(E, 127));
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack_f16x2(bf16_lo(w[i]) * f, bf16_hi(w[i]) * f);
  v[0] = make_uint4(w[0], w[1], w[2], w[3]);
  v[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return E;
}

// 16 fp16 values of one token (two 16-byte registers) stored as v'' with
// v = v'' 2^(e - kGroupTop), aligned to the quad's largest e (returned):
// lanes with a smaller e scale their values by 2^(e - max) in place (exact
// down to fp16's subnormal range; values under 2^-24 of the quad's scale
// vanish).
__device__ __forceinline__ int f16x16_align(uint4 (&v)[2], int e) {
  int m = max(e, __shfl_xor_sync(0xffffffffu, e, 1));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  if (e != m) {
    const uint32_t f = f16_pow2_bits(e - m) * 0x10001u;
    uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(w[i]), "r"(f));
    v[0] = make_uint4(w[0], w[1], w[2], w[3]);
    v[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  return m;
}

// ---------------------------------------------------------------------------
// Warp-level bf16 tensor-core MMA: D(16x8 f32) += A(16x16 bf16) B(16x8 bf16)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], const uint32_t (&a)[4],
                                                 const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Same shape with fp16 operands.
__device__ __forceinline__ void mma_f16_16x8x16(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------
// Streamed once: do not keep in L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Asynchronous 16-byte global -> shared copy, cached in L2 only.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
// Same, for a stream read once in 64-byte pieces: L2 fetches whole 256-byte
// lines from HBM, so neighbouring pieces requested moments later hit L2.
__device__ __forceinline__ void cp_async16_stream(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;\n" ::"r"(s), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// cp_async_wait with a count known only after unrolling (0..7).
__device__ __forceinline__ void cp_async_wait_n(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}

// fp32 -> (hi, mid, lo) bf16 with w == hi + mid + lo to within 2^-24 |w|:
// each part is the bf16 rounding of what the previous parts left.
__device__ __forceinline__ void split3_bf16(float w, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const float h = __uint_as_float(pack_bf16x2(w, 0.f) << 16);
  const float r = w - h;
  const float m = __uint_as_float(pack_bf16x2(r, 0.f) << 16);
  hi = __float_as_uint(h) >> 16;
  mid = __float_as_uint(m) >> 16;
  lo = pack_bf16x2(r - m, 0.f) & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of a layer call starts with
// griddep_wait(): when it was launched with the programmatic-serialisation
// attribute it may be scheduled before its predecessor finishes, and this
// wait returns once the predecessor grid has completed and its writes are
// visible (without the attribute it returns at once).  griddep_trigger()
// then lets the next kernel's launch begin early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void griddep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + TMA bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking probe of the same phase (the thread is never suspended).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait budget: a wait gives up only when both the SM cycle counter (monotonic
// on this SM) and the global nanosecond timer (which the driver may step)
// say the budget is spent, so a timer step cannot end a wait early and the
// wait stays bounded either way.
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s
constexpr long long kCyclesPerNs = 2;                  // about 2 GHz
struct WaitBudget {
  uint64_t t0, ns;
  long long c0;
};
// A budget of limit_ns nanoseconds (0: the default kWaitLimitNs).
__device__ __forceinline__ WaitBudget wait_budget(uint64_t limit_ns = 0) {
  WaitBudget b;
  b.t0 = global_ns();
  b.c0 = clock64();
  b.ns = limit_ns ? limit_ns : kWaitLimitNs;
  return b;
}
__device__ __forceinline__ bool budget_spent(const WaitBudget& b) {
  return clock64() - b.c0 > (long long)b.ns * kCyclesPerNs && global_ns() - b.t0 > b.ns;
}
// Bounded wait for the phase with the given parity by a single thread (the
// rest of its warp may be elsewhere): it polls with the non-suspending probe
// and returns false once the budget is spent (the caller records
// MOE_DEV_WAIT_TIMEOUT).  Warps that wait together use a warp-uniform loop
// over the suspending form instead.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  const WaitBudget b = wait_budget();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (budget_spent(b)) return false;
  }
}
// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16);
// completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Hint: bring `bytes` (a multiple of 16) at `src` into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
// Barrier among the first `nthreads` threads of the CTA (named barrier `id`).
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Grouped-GEMV building block (decode kernels).  K permutation: an MMA's 16
// logical K positions are fed from physical columns so that a thread owns 16
// consecutive bytes of a weight row: for thread (g = lane/4, c = lane%4) and
// MMA step s of a 64-column chunk, the logical pairs (2c, 2c+1) and
// (2c+8, 2c+9) are physical columns 16c + 4s + {0,1} and 16c + 4s + {2,3}.
// The activations use the same map, so every product pairs the right weight
// with the right activation.
// ---------------------------------------------------------------------------
// One 64-column chunk: 16 weight rows (g, g+8) x NT*8 tokens.
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
// Device status word
// ---------------------------------------------------------------------------
// Word 0 holds the MOE_DEV_* bits; words 1-5 record the first bounded wait
// of a call that ran out (warp, barrier, step, parity, CTA) and words 6-15
// how far each role of that CTA had got (kernel-specific).  The first kernel
// of each call clears all of them.
constexpr int kStatusWords = 16;


// ---------------------------------------------------------------------------
// Combine of output columns h..h+V-1 of token t (V = 4 for fp32 expert
// rows, 8 for fp16; h a multiple of V):
// out[t, h..] = sum_j w[t,j] y_perm[tok_slot_row[t*k+j], h..] (+ shared_y),
// the routed terms summed in fp32 in slot order j (in groups of 8 slots,
// loads first), then added to the shared expert's row, rounded once to bf16.
// ---------------------------------------------------------------------------
// V consecutive expert outputs as fp32: V = 4 fp32 or V = 8 fp16 (16 bytes).
__device__ __forceinline__ void load_v(const float* p, float (&v)[4]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load_v(const uint16_t* p, float (&v)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
// 8 fp16 (one 16-byte register group) -> 8 floats.
__device__ __forceinline__ void unpack_f16x8(const uint4& a, float (&v)[8]) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
// L2-coherent load (ld.global.cg) of 8 fp16, for rows that other CTAs of the
// running kernel wrote.
__device__ __forceinline__ void load_v_cg(const uint16_t* p, float (&v)[8]) {
  const uint4 a = __ldcg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
// out[t, h .. h + V) = sum_j w[t, j] y_perm[tok_slot_row[t k + j], ...]
// (+ shared_y[t, ...]), summed in fp32 in slot order j, rounded once to bf16.
template <typename YT, int V>
__device__ __forceinline__ void combine_v(const YT* __restrict__ y_perm,
                                          const int32_t* __restrict__ tok_slot_row,
                                          const float* __restrict__ topk_w,
                                          const YT* __restrict__ shared_y, int t, int h, int H,
                                          int k, uint16_t* __restrict__ out) {
  float acc[V], r[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = r[i] = 0.f;
  if (shared_y) load_v(shared_y + (size_t)t * H + h, acc);
  for (int j0 = 0; j0 < k; j0 += 8) {
    int row[8];
    float w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      row[u] = j < k ? tok_slot_row[(size_t)t * k + j] : -1;
      w[u] = j < k ? topk_w[(size_t)t * k + j] : 0.f;
    }
    float y[8][V];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[u] >= 0) {
        load_v(y_perm + (size_t)row[u] * H + h, y[u]);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) y[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[u] < 0) continue;
#pragma unroll
      for (int i = 0; i < V; ++i) r[i] = fmaf(w[u], y[u][i], r[i]);
    }
  }
  uint32_t o[V / 2];
#pragma unroll
  for (int i = 0; i < V / 2; ++i) o[i] = pack_bf16x2(acc[2 * i] + r[2 * i], acc[2 * i + 1] + r[2 * i + 1]);
  if (V == 8)
    *reinterpret_cast<uint4*>(out + (size_t)t * H + h) = make_uint4(o[0], o[1], o[2], o[3]);
  else
    *reinterpret_cast<uint2*>(out + (size_t)t * H + h) = make_uint2(o[0], o[1]);
}

__device__ __forceinline__ void raise_status(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace moe
