// Internal declarations shared by the kernel translation units and the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_fp8.h"

namespace moe {

// Pairs handled by one CTA of the permutation's count and scatter kernels;
// the per-block scratch arrays are sized by it.
constexpr int kPermPairsPerBlock = 256;

// Sets the text returned by moe_last_error_message() on this host thread.
void set_last_error(const char* msg);

// Workspace layout for one set of dims (byte offsets, each 256-aligned).
struct WsLayout {
  size_t status, logits, rank, block_cnt, block_base, active, idx, w, off, row_token,
      tok_slot_row, hid, y_perm, sh_hid, sh_y, sh_off, sh_rows, sh_active, total;
};
WsLayout ws_layout(const moe_dims& d);

cudaError_t launch_route(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                         int E, int k, float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* status, cudaStream_t s);

cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, int32_t* rank,
                           int32_t* block_cnt, int32_t* block_base, int32_t* expert_off,
                           int32_t* row_token, int32_t* tok_slot_row, int32_t* active,
                           int32_t* status, cudaStream_t s);

cudaError_t launch_active_from_offsets(const int32_t* expert_off, int E, int32_t* active,
                                       int32_t* status, cudaStream_t s);

// Grouped GEMV over the experts listed in `active` (count, then ids).
// max_active bounds the list length; max_rows_per_expert bounds any segment.
cudaError_t launch_expert_gemv(const uint16_t* x, const int32_t* expert_off,
                               const int32_t* row_token, const int32_t* active, int max_active,
                               const moe_fp8_ffn& w, int H, int I, int max_rows_per_expert,
                               uint16_t* hid, float* y, int32_t* status, cudaStream_t s);

cudaError_t launch_combine(const float* y_perm, const int32_t* tok_slot_row, const float* topk_w,
                           const float* shared_y, int T, int H, int k, uint16_t* out,
                           cudaStream_t s);

// Identity permutation of T tokens onto one expert (the shared expert):
// off = {0, T}, rows = 0..T-1, active = {1, 0}.
cudaError_t launch_identity_perm(int T, int32_t* off, int32_t* rows, int32_t* active,
                                 cudaStream_t s);

}  // namespace moe
