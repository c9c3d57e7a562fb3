// Internal declarations shared by the kernel translation units and the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_fp8.h"

namespace moe {

// Pairs handled by one CTA of the permutation's count and scatter kernels;
// the per-block scratch arrays are sized by it.
constexpr int kPermPairsPerBlock = 256;

// Sets the text returned by moe_last_error_message() on this host thread.
void set_last_error(const char* msg);

// Kernel launch on `s`, optionally with programmatic stream serialisation
// (the kernel must begin with griddep_wait()).
// Adds one to the process-wide launch counter (moe_kernel_launches).
void count_launch();

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, bool pdl, Args&&... args) {
  count_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises `func`'s dynamic shared-memory limit to `bytes`, once per device
// (host-side attribute; the first call on a device should precede capture).
cudaError_t ensure_smem(const void* func, int bytes);

// 2-D TMA map over a row-major matrix [rows, cols] of esize-byte elements:
// box = box_cols x box_rows, swizzle 0, 64 or 128 bytes, L2 256-byte
// promotion, out-of-range elements read as zero.
cudaError_t make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, int esize,
                               const void* base, long long rows, int cols, int box_cols,
                               int box_rows, int swizzle_bytes);

// Largest expert count the library accepts.
constexpr int kMaxExperts = 1024;

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Workspace layout for one set of dims (byte offsets, each 256-aligned).
struct WsLayout {
  size_t status, logits, rank, block_cnt, block_base, active, idx, w, off, row_token,
      tok_slot_row, row_pair, xn, xe, hid, hexp, y_perm, yexp, sh_hid, sh_hexp, sh_y, sh_yexp,
      sgate, sh_off,
      sh_rows, sh_active, tile_off, sh_tile_off, x_perm, xexp, sh_x, sh_xexp, wr_planes,
      slot_done, sh_slot_done, ticket, total;
};
WsLayout ws_layout(const moe_dims& d);

// All launchers enqueue on `s`; with pdl the kernels are launched with
// programmatic stream serialisation (each begins with griddep_wait()).

// Router logits and top-k.  `part` holds up to 8 K-slices of partial
// logits, [8][T][E] floats; `planes` is scratch for the bf16 split of Wr,
// [3][E][H] (used from 128 tokens, router_tc_ok).  xn / xe (may be NULL):
// the streamed expert kernels' activations, written on the way
// (xn [T, H] fp16 = x 2^(14 - e), xe [T, H / 64] int8 = e per 64 columns).
cudaError_t launch_route(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                         int E, int k, float* part, uint16_t* planes, int32_t* topk_idx,
                         float* topk_w, uint16_t* xn, int8_t* xe, int32_t* status,
                         cudaStream_t s, bool pdl, const float* shared_gate = nullptr,
                         float* sgate = nullptr);

// Router logits on the tensor cores (route_tc.cu): T >= 128, E % 128 == 0,
// H % 64 == 0.  Writes KS slices of partial logits (KS from route_kslices).
bool router_tc_ok(int T, int H, int E);
cudaError_t launch_router_logits_tc(const uint16_t* x, const float* Wr, int T, int H, int E,
                                    int KS, float* part, uint16_t* planes, uint16_t* xn,
                                    int8_t* xe, int32_t* status, cudaStream_t s, bool pdl);

// Token rows per tile of the tensor-core GEMM (its MMA N, at most).
constexpr int kGemmTokenTile = 128;

// Both route launchers: with sgate set, the top-k warps also write
// sgate[t] = sigmoid(x[t] . shared_gate) (the gated shared expert's factor).

// Router logits, then top-k and the full permutation in one CTA, for
// T*k <= 4096 (small_route_permute_ok).  sh_* may be NULL (no shared expert).
// tile_off (E + 1 ints) may be NULL; else the permutation also writes the
// GEMM's token-tile prefix there.  counters[0, n_counters) (may be NULL) are
// zeroed: the GEMM's completion counters or the fused combine's tickets.
bool small_route_permute_ok(int T, int E, int k);
cudaError_t launch_route_permute_small(const uint16_t* x, const float* Wr, const float* bias,
                                       int T, int H, int E, int k, float* part,
                                       uint16_t* planes, int32_t* topk_idx, float* topk_w, int32_t* expert_off,
                                       int32_t* row_token, int32_t* tok_slot_row,
                                       int32_t* row_pair, int32_t* active, int32_t* sh_off,
                                       int32_t* sh_rows, int32_t* sh_active, uint16_t* xn,
                                       int8_t* xe, int32_t* tile_off, int32_t* counters,
                                       int n_counters,
                                       int32_t* status, cudaStream_t s, bool pdl,
                                       const float* shared_gate = nullptr,
                                       float* sgate = nullptr);

// The multi-kernel permutation (T*k > 4096).  tile_off (E + 1 ints, may be
// NULL): also the tensor-core GEMM's token-tile prefix; counters[0,
// n_counters) (may be NULL) are zeroed (the GEMM's completion counters).
cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, int32_t* rank,
                           int32_t* block_cnt, int32_t* block_base, int32_t* expert_off,
                           int32_t* row_token, int32_t* tok_slot_row, int32_t* row_pair,
                           int32_t* active, int32_t* status, cudaStream_t s, bool pdl,
                           int32_t* tile_off = nullptr, int32_t* counters = nullptr,
                           int n_counters = 0);

cudaError_t launch_active_from_offsets(const int32_t* expert_off, int E, int32_t* active,
                                       int32_t* status, cudaStream_t s, bool pdl);

// The streamed expert kernels' activations from bf16 x [T, H] (n = T H):
// xn [T, H] fp16 = x 2^(14 - e), xe [T, H / 64] int8 = e per 64 columns.
cudaError_t launch_x_norm(const uint16_t* x, int T, int H, uint16_t* xn, int8_t* xe,
                          cudaStream_t s, bool pdl);

// Grouped GEMV over the experts listed in `active` (count, then ids), on the
// normalised activations xn / xe (launch_x_norm or the router).  hid: [P, I]
// fp16 scratch with hexp [P, I/16]
// int8 exponents.  y: [P, H] fp32 when yexp is NULL, else fp16 with yexp
// [H/32][y_rows] int16 exponents (y = y'' 2^s).  max_active bounds the list
// length; tokens_per_expert_hint (the expected rows per expert) picks the
// MMA's N width; any segment length is handled.
// The combine folded into the streamed down projection (fp16 y only): the
// last down CTA of each 32-row slice of H writes out[t, slice] for every
// token.  ticket: H / 32 ints that are zero when the down kernel starts (the
// one-CTA permutation clears them); NULL = no fused combine.  Only for
// shapes fused_combine_ok accepts (T <= 64, k <= 8, the down grid of
// H / 32 x max_active CTAs in one wave).
bool fused_combine_ok(int T, int k, int H, int max_active);
struct FusedCombine {
  int32_t* ticket = nullptr;
  const int32_t* tok_slot_row = nullptr;
  const float* topk_w = nullptr;
  const float* sgate = nullptr;  // the shared expert's per-token factor, or NULL
  int T = 0, k = 0;
  uint16_t* out = nullptr;
};
// The shared expert as one more, always-selected expert of the same GEMV
// launches (the last CTA column of each grid): rows row0 .. row0 + T - 1 of
// hid and y hold tokens 0 .. T - 1, and its weights are these (one expert
// with the routed experts' I).  gc == NULL: no shared expert.
struct SharedExpert {
  const uint8_t *gc = nullptr, *uc = nullptr, *dc = nullptr;
  const float *gs = nullptr, *us = nullptr, *ds = nullptr;
  int T = 0, row0 = 0;
};
cudaError_t launch_expert_gemv(const uint16_t* xn, const int8_t* xe, const int32_t* expert_off,
                               const int32_t* row_token, const int32_t* active, int max_active,
                               const moe_fp8_ffn& w, int H, int I, int tokens_per_expert_hint,
                               uint16_t* hid, int8_t* hexp, void* y, int16_t* yexp, int y_rows,
                               int32_t* status, cudaStream_t s, bool pdl,
                               const FusedCombine& cmb = FusedCombine{},
                               const SharedExpert& sx = SharedExpert{});

// Grouped GEMM on the tensor cores (tcgen05) for many tokens per expert:
// gate/up + SwiGLU -> hid, then down -> y.  Needs H % 256 == 0 and
// I % 128 == 0, H, I <= 4096 (expert_gemm_tc_ok).  tile_off: E + 1 ints of scratch;
// slot_done: cdiv(P, 128) + min(E, P) ints of scratch (the down GEMM then
// starts each token tile as soon as its hid rows are stored), or NULL.
// tile_off_ready: the permutation already wrote tile_off and zeroed slot_done
// (launch_route_permute_small), so the tile-offset kernel is skipped.
bool expert_gemm_tc_ok(int H, int I);
// How the GEMM's activation rows are gathered.  Default: one warp per row
// from row_token.  tok_slot_row set (the layer call): one warp per token,
// written to the token's k rows and, when shared_rows is set, also to row t
// of shared_rows / shared_xexp (the shared expert's rows, which a later GEMM
// call then uses with rows_ready).  rows_ready: x_perm / xexp already hold
// the rows; no gather is launched.
struct GemmGather {
  const int32_t* tok_slot_row = nullptr;
  int k = 0;
  uint16_t* shared_rows = nullptr;
  int32_t* shared_xexp = nullptr;
  bool rows_ready = false;
};
// x: [T, H] bf16.  x_perm: [P, H] fp16 and xexp: [P] int32 scratch that
// receive the activation rows in expert order, normalised by a power of two
// (x[row_token[p]] = x_perm[p] 2^xexp[p]).  hid: [P, I] fp16 scratch.  y:
// [P, H] fp32 when yexp is NULL, else fp16 with yexp [H/32][yexp_rows] int16
// exponents (y = y'' 2^s).
cudaError_t launch_expert_gemm_tc(const uint16_t* x, int T, const int32_t* expert_off,
                                  const int32_t* row_token, uint16_t* x_perm, int32_t* xexp,
                                  int E, int P, const moe_fp8_ffn& w, int H, int I,
                                  int32_t* tile_off, int32_t* slot_done, uint16_t* hid, void* y,
                                  int16_t* yexp, int yexp_rows, int32_t* status, cudaStream_t s,
                                  bool pdl, bool tile_off_ready = false,
                                  const GemmGather& gather = GemmGather{});
// The same GEMMs on E4M3 activations (tcgen05.mma kind::f8f6f4): x is
// quantised per row and 128-column group while it is gathered (the layer
// call's token -> row map), hid per row and 128 features by the gate/up
// epilogue.  tile_off and zeroed slot_done come from the permutation.
// x8 [P][H] / hid8 [P][I] codes, xs [P][act8_scale_ld(H)] / hs
// [P][act8_scale_ld(I)] float scales (scratch); y [P][H] fp16 with yexp
// [H/32][yexp_rows].  Needs expert_gemm_tc_ok(H, I).
int act8_scale_ld(int K);
cudaError_t launch_expert_gemm_f8(const uint16_t* x, int T, const int32_t* expert_off,
                                  const int32_t* tok_slot_row, int k, int E, int P,
                                  const moe_fp8_ffn& w, int H, int I, const int32_t* tile_off,
                                  int32_t* slot_done, uint8_t* x8, float* xs, uint8_t* hid8,
                                  float* hs, uint16_t* y, int16_t* yexp, int yexp_rows,
                                  int32_t* status, cudaStream_t s, bool pdl);
// slot_done entries the GEMM uses for P routed rows over E experts.
inline int expert_gemm_slots(int P, int E) { return (P + 127) / 128 + (E < P ? E : P); }

// Regime: true -> tensor-core grouped GEMM, false -> streamed grouped GEMV.
// Decided on the host from shapes only; MOE_FP8_EXPERT_PATH=gemm|gemv in the
// environment overrides it (when the GEMM supports the shapes).
bool use_expert_gemm(int rows, int experts, int H, int I);

// fp32 y_perm and shared_y (may be NULL), the C ABI's moe_combine.
cudaError_t launch_combine(const float* y_perm, const int32_t* tok_slot_row, const float* topk_w,
                           const float* shared_y, int T, int H, int k, uint16_t* out,
                           cudaStream_t s, bool pdl);
// The same inside moe_layer_forward (programmatic dependent launch) on fp16
// rows with power-of-two exponents: y [P, H] with yexp [H/32][P], the shared
// rows sy [T, H] with syexp [H/32][T] (both NULL without a shared expert).
// The slot rows and weights, which the routing wrote before any expert
// kernel ran, are loaded before the kernel waits for the expert outputs.
// yexp's row stride is P, syexp's sstride; sgate (may be NULL) scales the
// shared row per token.
cudaError_t launch_combine_layer(const uint16_t* y, const int16_t* yexp, int P,
                                 const int32_t* tok_slot_row, const float* topk_w,
                                 const uint16_t* sy, const int16_t* syexp, int sstride,
                                 const float* sgate, int T, int H, int k, uint16_t* out,
                                 cudaStream_t s);

// Device address of the status word of moe_permute_static_scratch's fixed
// array on the current device.
cudaError_t static_scratch_status(int32_t** out);

// Runtime cross-check (verify.cu): scratch bytes for n sampled tokens, the
// largest n, and the launch (result: device float[3]).
size_t verify_workspace(const moe_dims& d, int n);
int verify_max_tokens();
cudaError_t launch_verify(const uint16_t* x, const moe_fp8_ffn& routed, const moe_fp8_ffn* shared,
                          const float* shared_gate, const moe_dims& d, const uint16_t* out,
                          const int32_t* topk_idx, const float* topk_w, const int32_t* tokens,
                          int n, float* result, void* ws, cudaStream_t s);

// Identity permutation of T tokens onto one expert (the shared expert):
// off = {0, T}, rows = 0..T-1, active = {1, 0}.
cudaError_t launch_identity_perm(int T, int32_t* off, int32_t* rows, int32_t* active,
                                 cudaStream_t s, bool pdl);

}  // namespace moe
