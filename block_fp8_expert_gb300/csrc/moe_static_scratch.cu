// moe_permute_static_scratch: the expert permutation for callers that cannot
// allocate device memory.
//
// moe_permute needs a caller-allocated workspace for its scratch (per-pair
// ranks, per-block expert counts and prefixes, the active-expert list and the
// status word).  Some callers have no way to provide one: a plugin whose host
// framework hands it only the input and output buffers of each call, or a
// serving loop whose memory is fixed at start-up and may not grow later.  For
// them this entry point keeps that scratch in one fixed array compiled into
// the library, sized for at most kStaticMaxPairs (token, slot) pairs and
// kStaticMaxExperts experts.  It runs the same three permutation kernels as
// moe_permute, on pointers into that array.
//
// Costs and rules that come with a fixed array:
//  - every GPU that loads the library holds the array (about 1.3 MB) until
//    the process exits;
//  - all calls on one device share it: two calls whose work overlaps on the
//    GPU (different streams, no ordering between them) race and both results
//    are undefined; order such calls on one stream or with events;
//  - the array keeps the previous call's contents; the kernels overwrite every
//    value they read except the status word, which each call clears first
//    and moe_read_device_status reads back when it is given no workspace.
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kStaticMaxPairs = 65536;  // T * k
constexpr int kStaticMaxExperts = 512;  // E
constexpr int kStaticBlocks = kStaticMaxPairs / kPermPairsPerBlock;

constexpr size_t round256(size_t v) { return (v + 255) & ~size_t(255); }
constexpr size_t kOffStatus = 0;
constexpr size_t kOffRank = 256;
constexpr size_t kOffCnt = kOffRank + round256(sizeof(int32_t) * kStaticMaxPairs);
constexpr size_t kOffBase =
    kOffCnt + round256(sizeof(int32_t) * kStaticBlocks * kStaticMaxExperts);
constexpr size_t kOffActive =
    kOffBase + round256(sizeof(int32_t) * kStaticBlocks * kStaticMaxExperts);
constexpr size_t kStaticBytes = kOffActive + round256(sizeof(int32_t) * (1 + kStaticMaxExperts));

// The scratch itself.  In host code this name is only a host-side stand-in
// for the symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_permute_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// The fixed array's status word on the current device (read by
// moe_read_device_status when it is given no workspace).
cudaError_t static_scratch_status(int32_t** out) {
  void* base = nullptr;
  const cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return e;
  *out = reinterpret_cast<int32_t*>(static_cast<char*>(base) + kOffStatus);
  return cudaSuccess;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_static_scratch(const int32_t* topk_idx, moe_dims d,
                                                 int32_t* expert_off, int32_t* row_token,
                                                 int32_t* tok_slot_row, void* stream) {
  if (d.T < 0) {
    set_last_error("moe_permute_static_scratch: T < 0");
    return MOE_ERR_INVALID_ARG;
  }
  if (d.E < 1 || d.E > kStaticMaxExperts || d.k < 1 || d.k > 32 || d.k > d.E) {
    set_last_error("moe_permute_static_scratch: need 1 <= E <= 512 and 1 <= k <= min(E, 32)");
    return MOE_ERR_UNSUPPORTED;
  }
  if ((long long)d.T * d.k > kStaticMaxPairs) {
    set_last_error("moe_permute_static_scratch: T*k exceeds the fixed scratch limit of 65536 "
                   "pairs; use moe_permute with a workspace");
    return MOE_ERR_UNSUPPORTED;
  }
  if (!expert_off || !aligned16(expert_off) ||
      (d.T > 0 && (!topk_idx || !row_token || !tok_slot_row || !aligned16(topk_idx) ||
                   !aligned16(row_token) || !aligned16(tok_slot_row)))) {
    set_last_error("moe_permute_static_scratch: NULL or misaligned array");
    return MOE_ERR_INVALID_ARG;
  }
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  char* b = static_cast<char*>(base);
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* status = reinterpret_cast<int32_t*>(b + kOffStatus);
  e = cudaMemsetAsync(status, 0, sizeof(int32_t) * kStatusWords, st);
  if (e == cudaSuccess)
    e = launch_permute(topk_idx, d.T, d.E, d.k, reinterpret_cast<int32_t*>(b + kOffRank),
                       reinterpret_cast<int32_t*>(b + kOffCnt),
                       reinterpret_cast<int32_t*>(b + kOffBase), expert_off, row_token,
                       tok_slot_row, nullptr, reinterpret_cast<int32_t*>(b + kOffActive), status,
                       st, false);
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
