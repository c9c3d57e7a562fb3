// The C ABI (include/moe_fp8.h): argument checks, workspace layout, launches.
// Nothing here allocates device memory or synchronises the host, except
// moe_read_device_status, whose job is to read a device word back.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include "moe_internal.h"

namespace moe {
namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE_PTR(p)                                                                    \
  do {                                                                                    \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);               \
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

#define REQUIRE_OPT_PTR(p)                                                   \
  do {                                                                       \
    if ((p) != nullptr && !aligned16(p))                                     \
      return fail(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p);    \
  } while (0)

#define CUDA_CHECK(expr, where)                           \
  do {                                                    \
    cudaError_t e_ = (expr);                              \
    if (e_ != cudaSuccess) return cuda_fail(e_, where);   \
  } while (0)

moe_status check_dims(const moe_dims& d) {
  if (d.T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d < 0", d.T);
  auto dim_ok = [](int v) { return v >= 64 && v <= 16384 && v % 64 == 0; };
  if (!dim_ok(d.H))
    return fail(MOE_ERR_UNSUPPORTED, "H = %d: need a multiple of 64 in [64, 16384]", d.H);
  if (!dim_ok(d.I))
    return fail(MOE_ERR_UNSUPPORTED, "I = %d: need a multiple of 64 in [64, 16384]", d.I);
  if (d.I_shared != 0 && !dim_ok(d.I_shared))
    return fail(MOE_ERR_UNSUPPORTED, "I_shared = %d: need 0 or a multiple of 64 in [64, 16384]",
                d.I_shared);
  if (d.E < 1 || d.E > kMaxExperts)
    return fail(MOE_ERR_UNSUPPORTED, "E = %d outside [1, %d]", d.E, kMaxExperts);
  if (d.k < 1 || d.k > 32 || d.k > d.E)
    return fail(MOE_ERR_UNSUPPORTED, "k = %d outside [1, min(E, 32)]", d.k);
  if ((long long)d.T * d.k >= (1LL << 31)) return fail(MOE_ERR_UNSUPPORTED, "T*k too large");
  return MOE_OK;
}

moe_status check_mat(const moe_fp8_mat& m, const char* name) {
  if (!m.codes || !m.scales) return fail(MOE_ERR_INVALID_ARG, "%s: NULL codes or scales", name);
  if (!aligned16(m.codes) || !aligned16(m.scales))
    return fail(MOE_ERR_INVALID_ARG, "%s: codes/scales not 16-byte aligned", name);
  return MOE_OK;
}

moe_status check_ffn(const moe_fp8_ffn& w, const char* name) {
  std::string n(name);
  moe_status s;
  if ((s = check_mat(w.gate, (n + ".gate").c_str())) != MOE_OK) return s;
  if ((s = check_mat(w.up, (n + ".up").c_str())) != MOE_OK) return s;
  return check_mat(w.down, (n + ".down").c_str());
}

moe_status check_ws(const moe_dims& d, const void* ws, size_t ws_bytes) {
  REQUIRE_PTR(ws);
  const size_t need = ws_layout(d).total;
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", ws_bytes, need);
  return MOE_OK;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

// Average rows per expert from which the tensor-core GEMM replaces the
// streamed GEMV.  Routed experts: from 1 (measured crossover: at 1 row per
// expert the two paths take the same time (Qwen3 T=16), from 2 the GEMM is
// faster (T=32: 131 vs 134 us), and it pulls ahead as soon as a few experts
// are hot, since the GEMV re-streams an expert's weights for every group of 8
// or 16 rows).  One dense expert (the shared one) has only I / 128 weight
// tiles per 128 rows to spread over the SMs: from 32 rows.  Small experts
// (H * I < 2^20 codes per matrix) stream so few bytes that the GEMM path's
// fixed costs (two more launches, the tile machinery) dominate: they keep the
// GEMV up to 32 rows per expert (the 16-expert H 256 layer: GEMV 20 / 26 us
// at 32 / 100 tokens, GEMM 30 / 32 us).
constexpr int kGemmMinRowsPerRoutedExpert = 1;
// Tokens from which the layer call gathers the GEMM's rows token-major
// (about one wave of its 8-token CTAs).
constexpr int kTokenGatherMin = 1024;
constexpr int kGemmMinRowsPerSmallExpert = 32;
constexpr int kGemmMinRowsDense = 32;
constexpr long long kSmallExpertCodes = 1ll << 20;

bool use_expert_gemm(int rows, int experts, int H, int I) {
  if (!expert_gemm_tc_ok(H, I)) return false;
  const char* f = getenv("MOE_FP8_EXPERT_PATH");
  if (f && strcmp(f, "gemm") == 0) return true;
  if (f && strcmp(f, "gemv") == 0) return false;
  if (experts == 1) return rows >= kGemmMinRowsDense;
  const int per = (long long)H * I >= kSmallExpertCodes ? kGemmMinRowsPerRoutedExpert
                                                        : kGemmMinRowsPerSmallExpert;
  return (long long)rows >= (long long)per * experts;
}

cudaError_t ensure_smem(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, func})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({dev, func});
  return e;
}

std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

WsLayout ws_layout(const moe_dims& d) {
  const size_t T = d.T, E = d.E, P = (size_t)d.T * d.k, H = d.H, I = d.I, Is = d.I_shared;
  const size_t nb = (P + 255) / 256;
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes ? bytes : 1);
    return at;
  };
  L.status = take(256);
  L.logits = take(8 * T * E * 4);  // up to 8 K-slices of partial router logits
  L.rank = take(P * 4);
  L.block_cnt = take(nb * E * 4);
  L.block_base = take(nb * E * 4);
  L.active = take((1 + E) * 4);
  L.idx = take(P * 4);
  L.w = take(P * 4);
  L.off = take((E + 1) * 4);
  L.row_token = take(P * 4);
  L.tok_slot_row = take(P * 4);
  L.row_pair = take(P * 4);
  // the streamed expert kernels' activations: fp16, exponent per 64 columns
  L.xn = take(T * H * 2);
  L.xe = take(T * (H / 64));
  // hid and y rows in fp16 with power-of-two exponents: hid per 16 features
  // (streamed GEMV), y per 32 columns, the exponent tables [H / 32][rows]
  // (P + T rows with a shared expert: the streamed GEMV may run it as one
  // more expert of the same launches, rows P .. P + T - 1)
  const size_t R = P + (Is ? T : 0);
  L.hid = take(R * I * 2);
  L.hexp = take(R * (I / 16));
  L.y_perm = take(R * H * 2);
  L.yexp = take((H / 32) * R * 2);
  L.sh_hid = take(Is ? T * Is * 2 : 0);
  L.sh_hexp = take(Is ? T * (Is / 16) : 0);
  L.sh_y = take(Is ? T * H * 2 : 0);
  L.sh_yexp = take(Is ? (H / 32) * T * 2 : 0);
  L.sgate = take(Is ? T * 4 : 0);  // gated shared expert: sigmoid(x . g) per token
  L.sh_off = take(2 * 4);
  L.sh_rows = take(Is ? T * 4 : 0);
  L.sh_active = take(2 * 4);
  L.tile_off = take((E + 1) * 4);
  L.sh_tile_off = take(2 * 4);
  // the tensor-core GEMM's normalised activation rows in expert order
  const bool gemm_ok = expert_gemm_tc_ok(d.H, d.I);
  const bool sh_gemm_ok = Is && expert_gemm_tc_ok(d.H, d.I_shared);
  L.x_perm = take(gemm_ok ? P * H * 2 : 0);
  L.xexp = take(gemm_ok ? P * 4 : 0);
  L.sh_x = take(sh_gemm_ok ? T * H * 2 : 0);
  L.sh_xexp = take(sh_gemm_ok ? T * 4 : 0);
  L.wr_planes = take(router_tc_ok(d.T, d.H, d.E) ? 3 * E * H * 2 : 0);
  L.slot_done = take(expert_gemm_slots(P, E) * 4);
  L.ticket = take(((size_t)d.H / 32) * 4);  // fused combine: one per 32 columns of H
  L.sh_slot_done = take(Is ? ((T + 127) / 128 + 1) * 4 : 0);
  L.total = o;
  return L;
}

__global__ void k_identity_perm(int T, int32_t* off, int32_t* rows, int32_t* active) {
  griddep_wait();
  griddep_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < T) rows[i] = i;
  if (i == 0) {
    off[0] = 0;
    off[1] = T;
    active[0] = T > 0 ? 1 : 0;
    active[1] = 0;
  }
}

cudaError_t launch_identity_perm(int T, int32_t* off, int32_t* rows, int32_t* active,
                                 cudaStream_t s, bool pdl) {
  return launch_k(k_identity_perm, dim3(cdiv(T > 0 ? T : 1, 256)), dim3(256), 0, s, pdl, T, off,
                  rows, active);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_STATUS: return "device reported bad input";
    case MOE_ERR_TIMEOUT: return "bounded device wait timed out";
    case MOE_ERR_NOT_IMPLEMENTED: return "not implemented";
    default: return "unknown status";
  }
}

const char* moe_last_error_message(void) { return g_last_error.c_str(); }

const char* moe_version(void) { return "moe_fp8 0.1 sm_103a"; }

unsigned long long moe_kernel_launches(void) { return moe::g_launches.load(); }

int moe_expert_uses_gemm(moe_dims d) {
  if (check_dims(d) != MOE_OK) return -1;
  return use_expert_gemm(d.T * d.k, d.E, d.H, d.I) ? 1 : 0;
}

moe_status moe_workspace_bytes(moe_dims d, size_t* bytes) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = ws_layout(d).total;
  return MOE_OK;
}

moe_status moe_route(const uint16_t* x, const float* Wr, const float* bias, moe_dims d,
                     int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                     void* stream) {
  moe_status s;
  if ((s = check_dims(d)) != MOE_OK) return s;
  if (d.T == 0) return MOE_OK;  // no token: nothing is read or written
  REQUIRE_PTR(x);
  REQUIRE_PTR(Wr);
  REQUIRE_OPT_PTR(bias);
  REQUIRE_PTR(topk_idx);
  REQUIRE_PTR(topk_w);
  if ((s = check_ws(d, ws, ws_bytes)) != MOE_OK) return s;
  const WsLayout L = ws_layout(d);
  CUDA_CHECK(launch_route(x, Wr, bias, d.T, d.H, d.E, d.k, at<float>(ws, L.logits),
                          at<uint16_t>(ws, L.wr_planes), topk_idx, topk_w, nullptr, nullptr,
                          at<int32_t>(ws, L.status), (cudaStream_t)stream, true),
             "moe_route");
  return MOE_OK;
}

moe_status moe_permute(const int32_t* topk_idx, moe_dims d, int32_t* expert_off,
                       int32_t* row_token, int32_t* tok_slot_row, void* ws, size_t ws_bytes,
                       void* stream) {
  moe_status s;
  if ((s = check_dims(d)) != MOE_OK) return s;
  REQUIRE_PTR(expert_off);
  if (d.T > 0) {  // with no token only the offsets (all zero) are written
    REQUIRE_PTR(topk_idx);
    REQUIRE_PTR(row_token);
    REQUIRE_PTR(tok_slot_row);
  }
  if ((s = check_ws(d, ws, ws_bytes)) != MOE_OK) return s;
  const WsLayout L = ws_layout(d);
  cudaStream_t st = (cudaStream_t)stream;
  CUDA_CHECK(cudaMemsetAsync(at<int32_t>(ws, L.status), 0, sizeof(int32_t) * kStatusWords, st),
             "moe_permute");
  CUDA_CHECK(launch_permute(topk_idx, d.T, d.E, d.k, at<int32_t>(ws, L.rank),
                            at<int32_t>(ws, L.block_cnt), at<int32_t>(ws, L.block_base),
                            expert_off, row_token, tok_slot_row, nullptr,
                            at<int32_t>(ws, L.active), at<int32_t>(ws, L.status), st, false),
             "moe_permute");
  return MOE_OK;
}

moe_status moe_expert_ffn_fp8(const uint16_t* x, const int32_t* expert_off,
                              const int32_t* row_token, moe_fp8_ffn w, moe_dims d,
                              float* y_perm, void* ws, size_t ws_bytes, void* stream) {
  moe_status s;
  if ((s = check_dims(d)) != MOE_OK) return s;
  if (d.T == 0) return MOE_OK;  // no token: nothing is read or written
  REQUIRE_PTR(x);
  REQUIRE_PTR(expert_off);
  REQUIRE_PTR(row_token);
  REQUIRE_PTR(y_perm);
  if ((s = check_ffn(w, "w")) != MOE_OK) return s;
  if ((s = check_ws(d, ws, ws_bytes)) != MOE_OK) return s;
  const WsLayout L = ws_layout(d);
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* active = at<int32_t>(ws, L.active);
  int32_t* status = at<int32_t>(ws, L.status);
  CUDA_CHECK(launch_active_from_offsets(expert_off, d.E, active, status, st, true),
             "moe_expert_ffn_fp8");
  const int P = d.T * d.k;
  const bool gemm = use_expert_gemm(P, d.E, d.H, d.I);
  if (!gemm)
    CUDA_CHECK(launch_x_norm(x, d.T, d.H, at<uint16_t>(ws, L.xn), at<int8_t>(ws, L.xe), st, true),
               "moe_expert_ffn_fp8");
  if (gemm)
    CUDA_CHECK(launch_expert_gemm_tc(x, d.T, expert_off, row_token, at<uint16_t>(ws, L.x_perm),
                                     at<int32_t>(ws, L.xexp), d.E, P, w, d.H, d.I,
                                     at<int32_t>(ws, L.tile_off), at<int32_t>(ws, L.slot_done),
                                     at<uint16_t>(ws, L.hid), y_perm, nullptr, 0, status, st,
                                     true),
               "moe_expert_ffn_fp8");
  else
    CUDA_CHECK(launch_expert_gemv(at<uint16_t>(ws, L.xn), at<int8_t>(ws, L.xe), expert_off,
                                  row_token, active, d.E < P ? d.E : P, w, d.H, d.I,
                                  cdiv(P, d.E), at<uint16_t>(ws, L.hid), at<int8_t>(ws, L.hexp),
                                  y_perm, nullptr, 0, status, st, true),
               "moe_expert_ffn_fp8");
  return MOE_OK;
}

moe_status moe_combine(const float* y_perm, const int32_t* tok_slot_row, const float* topk_w,
                       const float* shared_y, moe_dims d, uint16_t* out, void* stream) {
  moe_status s;
  if ((s = check_dims(d)) != MOE_OK) return s;
  if (d.T == 0) return MOE_OK;  // no token: nothing is read or written
  REQUIRE_PTR(y_perm);
  REQUIRE_PTR(tok_slot_row);
  REQUIRE_PTR(topk_w);
  REQUIRE_OPT_PTR(shared_y);
  REQUIRE_PTR(out);
  CUDA_CHECK(launch_combine(y_perm, tok_slot_row, topk_w, shared_y, d.T, d.H, d.k, out,
                            (cudaStream_t)stream, true),
             "moe_combine");
  return MOE_OK;
}

}  // extern "C"

namespace moe {
namespace {
// The layer call, with an optional gate vector for the shared expert; act8:
// the routed experts on E4M3 activations (routed experts only).
moe_status layer_forward(const uint16_t* x, const float* Wr, const float* bias,
                         moe_fp8_ffn routed, const moe_fp8_ffn* shared,
                         const float* shared_gate, moe_dims d, uint16_t* out,
                         int32_t* topk_idx_out, float* topk_w_out, void* ws, size_t ws_bytes,
                         void* stream, bool act8 = false) {
  moe_status s;
  if ((s = check_dims(d)) != MOE_OK) return s;
  if (act8) {
    if (d.I_shared > 0 || shared)
      return fail(MOE_ERR_UNSUPPORTED, "E4M3 activations: layers with a shared expert are not supported");
    if (!expert_gemm_tc_ok(d.H, d.I) || d.H > 2048 || d.I > 2048)
      return fail(MOE_ERR_UNSUPPORTED, "E4M3 activations need H % 256 == 0, I % 128 == 0 "
                                       "and H, I <= 2048");
  }
  if (d.T == 0) return MOE_OK;  // no token: nothing is read or written
  REQUIRE_PTR(x);
  REQUIRE_PTR(Wr);
  REQUIRE_OPT_PTR(bias);
  REQUIRE_PTR(out);
  REQUIRE_OPT_PTR(topk_idx_out);
  REQUIRE_OPT_PTR(topk_w_out);
  if ((s = check_ffn(routed, "routed")) != MOE_OK) return s;
  if (d.I_shared > 0) {
    if (!shared) return fail(MOE_ERR_INVALID_ARG, "I_shared > 0 but shared is NULL");
    if ((s = check_ffn(*shared, "shared")) != MOE_OK) return s;
  } else if (shared) {
    return fail(MOE_ERR_INVALID_ARG, "shared given but I_shared == 0");
  }
  REQUIRE_OPT_PTR(shared_gate);
  if ((s = check_ws(d, ws, ws_bytes)) != MOE_OK) return s;
  const WsLayout L = ws_layout(d);
  cudaStream_t st = (cudaStream_t)stream;
  const int P = d.T * d.k;
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.idx);
  float* w = topk_w_out ? topk_w_out : at<float>(ws, L.w);
  int32_t* off = at<int32_t>(ws, L.off);
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  int32_t* tok_slot_row = at<int32_t>(ws, L.tok_slot_row);
  int32_t* active = at<int32_t>(ws, L.active);
  // expert outputs inside the layer call: fp16 rows, exponent per 32 columns
  uint16_t* y_perm = at<uint16_t>(ws, L.y_perm);
  int16_t* yexp = at<int16_t>(ws, L.yexp);

  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* soff = at<int32_t>(ws, L.sh_off);
  int32_t* srows = at<int32_t>(ws, L.sh_rows);
  int32_t* sact = at<int32_t>(ws, L.sh_active);
  const bool has_shared = d.I_shared > 0;
  const bool gemm = act8 || use_expert_gemm(P, d.E, d.H, d.I);
  const bool small = small_route_permute_ok(d.T, d.E, d.k);
  // streamed GEMV, one-CTA permutation, no shared expert: the down kernel
  // also combines (its tickets cleared by the permutation)
  const bool shared_gemm = has_shared && use_expert_gemm(d.T, 1, d.H, d.I_shared);
  // The shared expert as one more expert of the routed GEMV launches (rows
  // P .. P + T - 1), when both run on the GEMV and their I match.
  const bool fused_shared = has_shared && !gemm && !shared_gemm && d.I_shared == d.I;
  const bool sep_shared = has_shared && !fused_shared;  // its own launches
  const int y_rows = P + (has_shared ? d.T : 0);  // rows of y_perm / yexp
  const int max_active = d.E < P ? d.E : P;
  const bool fuse_combine = !gemm && small && (!has_shared || fused_shared) &&
                            fused_combine_ok(d.T, d.k, d.H, max_active + (fused_shared ? 1 : 0));
  // the router writes the streamed kernels' activations when one runs
  const bool need_xn = !gemm || (has_shared && !shared_gemm);
  uint16_t* xn = need_xn ? at<uint16_t>(ws, L.xn) : nullptr;
  int8_t* xe = need_xn ? at<int8_t>(ws, L.xe) : nullptr;
  float* sgate = shared_gate ? at<float>(ws, L.sgate) : nullptr;
  if (small) {
    // router logits, then top-k + permutation (+ the shared expert's identity
    // permutation) in one CTA
    CUDA_CHECK(launch_route_permute_small(
                   x, Wr, bias, d.T, d.H, d.E, d.k, at<float>(ws, L.logits),
                   at<uint16_t>(ws, L.wr_planes), idx, w, off,
                   row_token, tok_slot_row, at<int32_t>(ws, L.row_pair), active,
                   sep_shared ? soff : nullptr, sep_shared ? srows : nullptr,
                   sep_shared ? sact : nullptr, xn, xe,
                   gemm ? at<int32_t>(ws, L.tile_off) : nullptr,
                   gemm ? at<int32_t>(ws, L.slot_done)
                        : (fuse_combine ? at<int32_t>(ws, L.ticket) : nullptr),
                   gemm ? expert_gemm_slots(P, d.E) : d.H / 32,
                   status, st, true, shared_gate, sgate),
               "moe_layer_forward: route+permute");
  } else {
    CUDA_CHECK(launch_route(x, Wr, bias, d.T, d.H, d.E, d.k, at<float>(ws, L.logits),
                            at<uint16_t>(ws, L.wr_planes), idx, w, xn, xe, status, st, true,
                            shared_gate, sgate),
               "moe_layer_forward: route");
    // (with the tensor-core GEMM: also its token-tile prefix and zeroed
    // completion counters, so that no tile-offset launch follows)
    CUDA_CHECK(launch_permute(idx, d.T, d.E, d.k, at<int32_t>(ws, L.rank),
                              at<int32_t>(ws, L.block_cnt), at<int32_t>(ws, L.block_base), off,
                              row_token, tok_slot_row, at<int32_t>(ws, L.row_pair), active,
                              status, st, true, gemm ? at<int32_t>(ws, L.tile_off) : nullptr,
                              gemm ? at<int32_t>(ws, L.slot_done) : nullptr,
                              gemm ? expert_gemm_slots(P, d.E) : 0),
               "moe_layer_forward: permute");
    if (sep_shared)
      CUDA_CHECK(launch_identity_perm(d.T, soff, srows, sact, st, true),
                 "moe_layer_forward: shared");
  }
  // From kTokenGatherMin tokens one warp per token normalises its row once
  // and writes its k routed rows (and its shared-expert row when that expert
  // also runs on the GEMM); below, one warp per routed row keeps more CTAs
  // in flight (8 tokens per CTA would leave most SMs idle).
  const bool token_gather = gemm && d.T >= kTokenGatherMin;
  if (act8) {
    // E4M3 activations: x and hid codes with their group scales in the
    // activation-row and hid scratch (codes first, then the scales)
    uint8_t* x8 = at<uint8_t>(ws, L.x_perm);
    float* xs = reinterpret_cast<float*>(x8 + (size_t)P * d.H);
    uint8_t* hid8 = at<uint8_t>(ws, L.hid);
    float* hs = reinterpret_cast<float*>(hid8 + (size_t)P * d.I);
    CUDA_CHECK(launch_expert_gemm_f8(x, d.T, off, tok_slot_row, d.k, d.E, P, routed, d.H, d.I,
                                     at<int32_t>(ws, L.tile_off), at<int32_t>(ws, L.slot_done),
                                     x8, xs, hid8, hs, y_perm, yexp, y_rows, status, st, true),
               "moe_layer_forward_act8: experts");
  } else if (gemm) {
    GemmGather gth;
    if (token_gather) {
      gth.tok_slot_row = tok_slot_row;
      gth.k = d.k;
      if (shared_gemm) {
        gth.shared_rows = at<uint16_t>(ws, L.sh_x);
        gth.shared_xexp = at<int32_t>(ws, L.sh_xexp);
      }
    }
    CUDA_CHECK(launch_expert_gemm_tc(x, d.T, off, row_token, at<uint16_t>(ws, L.x_perm),
                                     at<int32_t>(ws, L.xexp), d.E, P, routed, d.H, d.I,
                                     at<int32_t>(ws, L.tile_off), at<int32_t>(ws, L.slot_done),
                                     at<uint16_t>(ws, L.hid), y_perm, yexp, y_rows, status, st,
                                     true, /*tile_off_ready=*/true, gth),
               "moe_layer_forward: experts");
  } else {
    FusedCombine cmb;
    if (fuse_combine) {
      cmb.ticket = at<int32_t>(ws, L.ticket);
      cmb.tok_slot_row = tok_slot_row;
      cmb.topk_w = w;
      cmb.T = d.T;
      cmb.k = d.k;
      cmb.out = out;
      cmb.sgate = sgate;
    }
    SharedExpert sx;
    if (fused_shared) {
      sx.gc = shared->gate.codes;
      sx.gs = shared->gate.scales;
      sx.uc = shared->up.codes;
      sx.us = shared->up.scales;
      sx.dc = shared->down.codes;
      sx.ds = shared->down.scales;
      sx.T = d.T;
      sx.row0 = P;
    }
    CUDA_CHECK(launch_expert_gemv(xn, xe, off, row_token, active, max_active, routed, d.H, d.I,
                                  cdiv(P, d.E), at<uint16_t>(ws, L.hid), at<int8_t>(ws, L.hexp),
                                  y_perm, yexp, y_rows, status, st, true, cmb, sx),
               "moe_layer_forward: experts");
  }
  uint16_t* shared_y = nullptr;
  int16_t* shared_yexp = nullptr;
  int shared_stride = d.T;
  if (fused_shared) {
    shared_y = y_perm + (size_t)P * d.H;
    shared_yexp = yexp + P;
    shared_stride = y_rows;
  } else if (has_shared) {
    shared_y = at<uint16_t>(ws, L.sh_y);
    shared_yexp = at<int16_t>(ws, L.sh_yexp);
    if (shared_gemm) {
      GemmGather gth;
      gth.rows_ready = token_gather;  // the routed gather wrote the shared rows
      CUDA_CHECK(launch_expert_gemm_tc(x, d.T, soff, srows, at<uint16_t>(ws, L.sh_x),
                                       at<int32_t>(ws, L.sh_xexp), 1, d.T, *shared, d.H,
                                       d.I_shared, at<int32_t>(ws, L.sh_tile_off),
                                       at<int32_t>(ws, L.sh_slot_done), at<uint16_t>(ws, L.sh_hid),
                                       shared_y, shared_yexp, d.T, status, st, true, false, gth),
                 "moe_layer_forward: shared expert");
    }
    else
      CUDA_CHECK(launch_expert_gemv(xn, xe, soff, srows, sact, 1, *shared, d.H, d.I_shared, d.T,
                                    at<uint16_t>(ws, L.sh_hid), at<int8_t>(ws, L.sh_hexp),
                                    shared_y, shared_yexp, d.T, status, st, true),
                 "moe_layer_forward: shared expert");
  }
  if (!fuse_combine)
    CUDA_CHECK(launch_combine_layer(y_perm, yexp, y_rows, tok_slot_row, w, shared_y,
                                    shared_yexp, shared_stride, sgate, d.T, d.H, d.k, out, st),
               "moe_layer_forward: combine");
  return MOE_OK;
}
}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_layer_forward(const uint16_t* x, const float* Wr, const float* bias,
                             moe_fp8_ffn routed, const moe_fp8_ffn* shared, moe_dims d,
                             uint16_t* out, int32_t* topk_idx_out, float* topk_w_out, void* ws,
                             size_t ws_bytes, void* stream) {
  return layer_forward(x, Wr, bias, routed, shared, nullptr, d, out, topk_idx_out, topk_w_out,
                       ws, ws_bytes, stream);
}

moe_status moe_layer_forward_gated(const uint16_t* x, const float* Wr, const float* bias,
                                   moe_fp8_ffn routed, const moe_fp8_ffn* shared,
                                   const float* shared_gate, moe_dims d, uint16_t* out,
                                   int32_t* topk_idx_out, float* topk_w_out, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (check_dims(d) != MOE_OK) return check_dims(d);
  if (d.I_shared == 0 || !shared)
    return fail(MOE_ERR_INVALID_ARG, "the gated layer needs a shared expert (I_shared > 0)");
  if (!shared_gate) return fail(MOE_ERR_INVALID_ARG, "shared_gate is NULL");
  return layer_forward(x, Wr, bias, routed, shared, shared_gate, d, out, topk_idx_out,
                       topk_w_out, ws, ws_bytes, stream);
}

moe_status moe_layer_forward_act8(const uint16_t* x, const float* Wr, const float* bias,
                                  moe_fp8_ffn routed, moe_dims d, uint16_t* out,
                                  int32_t* topk_idx_out, float* topk_w_out, void* ws,
                                  size_t ws_bytes, void* stream) {
  return layer_forward(x, Wr, bias, routed, nullptr, nullptr, d, out, topk_idx_out, topk_w_out, ws,
                       ws_bytes, stream, true);
}

moe_status moe_verify_workspace_bytes(moe_dims d, int n_tokens, size_t* bytes) {
  moe_status s = check_dims(d);
  if (s != MOE_OK) return s;
  if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
  if (n_tokens < 1 || n_tokens > verify_max_tokens())
    return fail(MOE_ERR_UNSUPPORTED, "n_tokens = %d outside [1, %d]", n_tokens,
                verify_max_tokens());
  *bytes = verify_workspace(d, n_tokens);
  return MOE_OK;
}

moe_status moe_verify_layer(const uint16_t* x, moe_fp8_ffn routed, const moe_fp8_ffn* shared,
                            const float* shared_gate, moe_dims d, const uint16_t* out,
                            const int32_t* topk_idx, const float* topk_w, const int32_t* tokens,
                            int n_tokens, float* result, void* ws, size_t ws_bytes,
                            void* stream) {
  moe_status s;
  if ((s = check_dims(d)) != MOE_OK) return s;
  if (d.T < 1) return fail(MOE_ERR_INVALID_ARG, "no token to verify (T = 0)");
  if (n_tokens < 1 || n_tokens > verify_max_tokens())
    return fail(MOE_ERR_UNSUPPORTED, "n_tokens = %d outside [1, %d]", n_tokens,
                verify_max_tokens());
  REQUIRE_PTR(x);
  REQUIRE_PTR(out);
  REQUIRE_PTR(topk_idx);
  REQUIRE_PTR(topk_w);
  REQUIRE_PTR(tokens);
  REQUIRE_PTR(result);
  REQUIRE_OPT_PTR(shared_gate);
  if ((s = check_ffn(routed, "routed")) != MOE_OK) return s;
  if (d.I_shared > 0) {
    if (!shared) return fail(MOE_ERR_INVALID_ARG, "I_shared > 0 but shared is NULL");
    if ((s = check_ffn(*shared, "shared")) != MOE_OK) return s;
  } else if (shared || shared_gate) {
    return fail(MOE_ERR_INVALID_ARG, "shared expert given but I_shared == 0");
  }
  REQUIRE_PTR(ws);
  if (ws_bytes < verify_workspace(d, n_tokens))
    return fail(MOE_ERR_WORKSPACE, "verify workspace of %zu bytes, need %zu", ws_bytes,
                verify_workspace(d, n_tokens));
  CUDA_CHECK(launch_verify(x, routed, shared, shared_gate, d, out, topk_idx, topk_w, tokens,
                           n_tokens, result, ws, (cudaStream_t)stream),
             "moe_verify_layer");
  return MOE_OK;
}

moe_status moe_read_device_status(const void* ws, int32_t* status, void* stream) {
  REQUIRE_OPT_PTR(ws);
  if (!status) return fail(MOE_ERR_INVALID_ARG, "status is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  const void* word = ws;
  if (!word) {
    // no workspace: the fixed array of moe_permute_static_scratch
    int32_t* p = nullptr;
    CUDA_CHECK(static_scratch_status(&p), "moe_read_device_status");
    word = p;
  }
  int32_t v = 0;
  CUDA_CHECK(cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, st),
             "moe_read_device_status");
  CUDA_CHECK(cudaStreamSynchronize(st), "moe_read_device_status");
  *status = v;
  if (v != 0) return fail(MOE_ERR_DEVICE_STATUS, "device status word 0x%x", v);
  return MOE_OK;
}

}  // extern "C"
