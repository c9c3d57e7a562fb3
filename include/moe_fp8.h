/*
 * moe_fp8.h - C ABI of a block-FP8 (E4M3) Mixture-of-Experts FFN layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer, as the colizig README states its parts (model table under "What
 * this project is trying to prove": experts, top-k routing, an optional shared
 * expert; "Features": block-FP8 E4M3 expert weights evaluated with a fused
 * decode+FMA dot product, MoE per-expert evaluation):
 *
 *   l[t,e]  = sum_h x[t,h] Wr[e,h] (+ b[e])                       router GEMM
 *   p[t,:]  = softmax(l[t,:]) over the E experts
 *   idx,w   = the k largest p[t,e] (descending, ties to the lower e),
 *             w_j = p_j / sum_{selected} p                        top-k, renorm
 *   rows    = the (t,j) pairs sorted by expert, ascending t inside an expert
 *   W[r,c]  = dec(C[r,c]) * S[r/128, c/128]                       block-FP8
 *   hid     = silu(x Wg^T) * (x Wu^T),  silu(z) = z/(1+exp(-z))   SwiGLU
 *   y       = hid Wd^T                                            down proj.
 *   out[t]  = sum_j w[t,j] y[row(t,j)] (+ shared(x[t]))           combine
 *
 * Conventions shared by every call:
 *  - Every pointer is a DEVICE pointer the caller owns (allocated, for
 *    example, by PyTorch); the library allocates no memory.  Every array must
 *    start on a 16-byte boundary.
 *  - bf16 arrays are passed as uint16_t bit patterns (IEEE binary32 top half).
 *  - `stream` is a cudaStream_t passed as void*; every call only enqueues
 *    work on it and returns without synchronising the host, so a sequence of
 *    calls can be captured into a CUDA graph.  Host-side argument errors are
 *    returned before anything is enqueued.
 *  - `ws` is a caller-owned device workspace of at least the size returned
 *    by moe_workspace_bytes() for the same dims; its contents on entry do not
 *    matter.  Calls that overlap on the GPU must not share one workspace.
 *  - T = 0 is valid: the call checks its dims and returns MOE_OK without
 *    touching any array (moe_permute still writes the E+1 zero offsets), so
 *    token-sized pointers may then be NULL.
 *  - Supported shapes: H, I and I_shared (when non-zero) multiples of 64 and
 *    at most 16384; 1 <= E <= 1024; 1 <= k <= min(E, 32); 0 <= T and
 *    T*k < 2^31.  Other shapes return MOE_ERR_UNSUPPORTED.
 *  - Errors are never silent.  A call returns MOE_OK only after every check
 *    it can make on the host; errors the kernels detect (for example an
 *    expert index out of range given to moe_permute) set a status word in the
 *    workspace that moe_read_device_status() returns.  There is no CPU
 *    fallback: without a usable GPU every call fails with MOE_ERR_CUDA.
 */
#ifndef MOE_FP8_H
#define MOE_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1     /* null or misaligned pointer, bad value  */
#define MOE_ERR_UNSUPPORTED 2     /* shape outside the supported set        */
#define MOE_ERR_WORKSPACE 3       /* workspace smaller than required        */
#define MOE_ERR_CUDA 4            /* a CUDA launch or runtime call failed   */
#define MOE_ERR_DEVICE_STATUS 5   /* a kernel flagged bad input on device   */
#define MOE_ERR_TIMEOUT 6         /* a bounded device wait gave up          */
#define MOE_ERR_NOT_IMPLEMENTED 7

/* Device status bits (moe_read_device_status). */
#define MOE_DEV_BAD_EXPERT_INDEX 1 /* moe_permute saw idx < 0 or idx >= E   */
#define MOE_DEV_WAIT_TIMEOUT 2     /* a kernel's bounded wait ran out       */
#define MOE_DEV_FP16_RANGE 4       /* an fp16 intermediate left its range   */
#define MOE_DEV_NONFINITE 8        /* an input (x, a block scale) or an
                                      intermediate was infinite or NaN      */

/* Layer dimensions. T tokens, hidden size H, routed-expert intermediate I,
 * E routed experts, top-k, shared-expert intermediate I_shared (0 = none). */
typedef struct {
  int32_t T, H, I, E, k, I_shared;
} moe_dims;

/* One block-FP8 weight stack: codes are E4M3 bytes, scales one float per
 * 128x128 block.  For a stack of n matrices of shape [rows, cols] (rows =
 * output features, cols = input features, cols contiguous):
 *   codes  uint8 [n, rows, cols]
 *   scales float [n, ceil(rows/128), ceil(cols/128)]                       */
typedef struct {
  const uint8_t* codes;
  const float* scales;
} moe_fp8_mat;

/* The three projections of n experts: gate and up [n, I, H], down [n, H, I]. */
typedef struct {
  moe_fp8_mat gate, up, down;
} moe_fp8_ffn;

/* Short text for a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Text of the most recent failure on the calling host thread ("" if none). */
const char* moe_last_error_message(void);

/* Library version string, e.g. "moe_fp8 0.1 sm_103a". */
const char* moe_version(void);

/* Diagnostic: kernel launches this library has issued in this process (all
 * host threads; a launch recorded into a CUDA graph counts once, at capture).
 * No counterpart in the pages: it lets a caller count the kernels of one
 * call, e.g. around the capture of one moe_layer_forward. */
unsigned long long moe_kernel_launches(void);

/* Diagnostic: 1 if the routed experts of a layer call with dimensions d run
 * on the tensor-core grouped GEMM, 0 if on the streamed GEMV (the regime rule
 * documented at moe_layer_forward, including the MOE_FP8_EXPERT_PATH
 * override); -1 if d is invalid.  No GPU work, no counterpart in the pages. */
int moe_expert_uses_gemm(moe_dims d);

/* Workspace size in bytes that every call below needs for dims d. */
moe_status moe_workspace_bytes(moe_dims d, size_t* bytes);

/*
 * Router: logits, softmax over experts, top-k with renormalisation (colizig
 * README, model table under "What this project is trying to prove": 128
 * experts top-8, or 512 experts top-10, per MoE layer).
 *   x        bf16  [T, H]
 *   Wr       float [E, H]
 *   bias     float [E] or NULL
 *   topk_idx int32 [T, k]  out: experts in descending probability, ties to
 *                          the lower expert index
 *   topk_w   float [T, k]  out: p_j / sum of the k selected p
 * Logits are accumulated in fp32.  The renormalised weights equal the softmax
 * over the k selected logits, which is how they are computed.  Clears the
 * workspace's device status word.
 */
moe_status moe_route(const uint16_t* x, const float* Wr, const float* bias,
                     moe_dims d, int32_t* topk_idx, float* topk_w, void* ws,
                     size_t ws_bytes, void* stream);

/*
 * Permutation of the T*k (token, slot) pairs into expert-contiguous rows, so
 * that each selected expert is evaluated once over all of its tokens
 * (colizig README, "Features": MoE per-expert evaluation).
 *   topk_idx     int32 [T, k]   in
 *   expert_off   int32 [E + 1]  out: segment e is rows [off[e], off[e+1]),
 *                               off[0] = 0, off[E] = T*k
 *   row_token    int32 [T*k]    out: token of each permuted row; inside one
 *                               segment tokens ascend
 *   tok_slot_row int32 [T*k]    out: row of pair (t, j) at index t*k + j
 * The result is unique and deterministic (no atomics decide an order).  An
 * index outside [0, E) sets MOE_DEV_BAD_EXPERT_INDEX; its pair gets no row
 * (tok_slot_row = -1) and off[E] counts only valid pairs.
 */
moe_status moe_permute(const int32_t* topk_idx, moe_dims d,
                       int32_t* expert_off, int32_t* row_token,
                       int32_t* tok_slot_row, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * Routed experts: for every permuted row r of expert e,
 *   y_perm[r] = (silu(x[row_token[r]] Wg_e^T) * (x[row_token[r]] Wu_e^T)) Wd_e^T
 * with W = dec(codes) * block scale (colizig README, "Features": block-FP8
 * E4M3 weights dequantised inside a fused decode+FMA dot product, MoE
 * per-expert evaluation).
 *   x          bf16  [T, H]
 *   expert_off int32 [E + 1], row_token int32 [T*k]  (from moe_permute)
 *   w          the E routed experts
 *   y_perm     float [T*k, H] out (rows past off[E] are left untouched)
 * d.T and d.k size the row space; d.I_shared is ignored.
 * Precision and range: the products run on fp16 operands with fp32
 * accumulation.  Every fp16 operand and intermediate (activations, scaled
 * weights, the SwiGLU output hid) is normalised by an exact power of two
 * that the fp32 side undoes, so block scales and activations of any
 * magnitude keep fp16's relative precision; the remaining roundings are
 * one fp16 rounding of each scaled weight (tensor-core GEMM) and of hid.
 * Flags: MOE_DEV_NONFINITE for an infinite or NaN activation, block scale
 * or result; on the tensor-core GEMM (many rows per expert), whose hid uses
 * a fixed power of two per expert, MOE_DEV_FP16_RANGE when a hid value
 * exceeds fp16's range or a token's values of 32 features all fall below
 * 2^-12 of the normalised scale (weights whose codes are far smaller or
 * larger than their block scale suggests).  Clears the device status word
 * first.
 */
moe_status moe_expert_ffn_fp8(const uint16_t* x, const int32_t* expert_off,
                              const int32_t* row_token, moe_fp8_ffn w,
                              moe_dims d, float* y_perm, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * Combine of the expert outputs back to token order, weighted by the
 * renormalised routing weights (colizig README, model table: top-k routed
 * experts plus, for the 512-expert family, one shared expert):
 * out[t] = sum_j topk_w[t,j] y_perm[tok_slot_row[t*k+j]]
 *                   (+ shared_y[t] when shared_y is not NULL),
 * summed in fp32 in slot order and rounded once to bf16 (nearest-even).
 * Pairs with tok_slot_row < 0 contribute nothing.
 *   y_perm float [T*k, H], tok_slot_row int32 [T*k], topk_w float [T, k],
 *   shared_y float [T, H] or NULL, out bf16 [T, H].
 */
moe_status moe_combine(const float* y_perm, const int32_t* tok_slot_row,
                       const float* topk_w, const float* shared_y, moe_dims d,
                       uint16_t* out, void* stream);

/*
 * The whole layer (colizig README, model table under "What this project is
 * trying to prove" and "Status": MoE (+shared expert) with block-FP8
 * weights): route, permute, routed experts, the shared expert when
 * d.I_shared > 0 (applied to every token with weight 1), combine.  The
 * expert outputs stay in the workspace as fp16 with one power-of-two
 * exponent per row and 32 columns, so they too have no range limit; the
 * precision and flags are those of moe_expert_ffn_fp8.
 *   shared       NULL when d.I_shared == 0, else one expert (n = 1) with
 *                gate/up [I_shared, H] and down [H, I_shared]
 *   out          bf16 [T, H]
 *   topk_idx_out int32 [T, k] or NULL: the routing, for inspection
 *   topk_w_out   float [T, k] or NULL
 * The regime (few tokens per expert: streamed grouped GEMV; many tokens per
 * expert: tensor-core grouped GEMM) is chosen on the host from T*k/E only:
 * the GEMM (tcgen05, needs H % 256 == 0, I % 128 == 0, H, I <= 4096) from 1
 * row per routed expert on average (T*k >= E) when H*I >= 2^20, else from
 * 32 rows per expert; the shared expert: from 32 tokens.  The
 * environment variable MOE_FP8_EXPERT_PATH=gemm or =gemv overrides the choice
 * (diagnostics and tests; read on every call).  The GEMM runs its gate/up
 * and down tiles in one launch when gate/up tiles alone fill the SMs and
 * there are at most 16 tiles per SM (bounded from the shapes), else in two;
 * MOE_FP8_GEMM_LAUNCHES=1 or =2 forces either.  Two more diagnostic
 * variables, read on every call of the tensor-core GEMM, exist to test the
 * failure path: MOE_FP8_WAIT_LIMIT_US shortens its bounded device waits
 * (default 2 s), and MOE_FP8_TEST_STALL=down makes its down projection wait
 * for one more finished gate/up tile than exists, so that the wait runs out
 * and MOE_DEV_WAIT_TIMEOUT is set (the output is then not valid).
 */
moe_status moe_layer_forward(const uint16_t* x, const float* Wr,
                             const float* bias, moe_fp8_ffn routed,
                             const moe_fp8_ffn* shared, moe_dims d,
                             uint16_t* out, int32_t* topk_idx_out,
                             float* topk_w_out, void* ws, size_t ws_bytes,
                             void* stream);

/*
 * The layer with a gated shared expert: as moe_layer_forward, except that
 * the shared expert's output for token t is scaled by
 * sigmoid(sum_h x[t,h] shared_gate[h]) before it is added.  This variant is
 * not on the colizig README (its 512-expert family lists "top-10 + 1 shared"
 * without a gate); it is the sigmoid-gated form of that shared expert.
 *   shared_gate float [H]; the layer must have a shared expert
 *               (d.I_shared > 0, shared not NULL).
 * The gate is computed by the routing kernels in fp32 and applied in the
 * combine.
 */
moe_status moe_layer_forward_gated(const uint16_t* x, const float* Wr,
                                   const float* bias, moe_fp8_ffn routed,
                                   const moe_fp8_ffn* shared,
                                   const float* shared_gate, moe_dims d,
                                   uint16_t* out, int32_t* topk_idx_out,
                                   float* topk_w_out, void* ws, size_t ws_bytes,
                                   void* stream);

/*
 * The layer with E4M3 activations in the routed experts.  The pages' block-FP8
 * format covers the weights only; this variant also feeds the experts' inputs
 * to the tensor cores as E4M3 (tcgen05.mma kind::f8f6f4), so the weight
 * codes are multiplied without a decode.  Routing and combine are those of
 * moe_layer_forward.  The inputs of each projection (x, then the SwiGLU
 * output hid in fp32) are quantised per row and group of 128 input features
 * (the weights' scale-block width): with a the group's largest magnitude,
 * code = E4M3(v * fp32(448 / a)) rounded to nearest even and saturated to
 * +-448, scale = fp32(a / 448); a = 0 gives zero codes and scale.  Each
 * 128-wide K block's E4M3 product sums are scaled by the weight and
 * activation scales in fp32 and accumulated in fp32.
 * Accuracy: the quantisation of x and hid costs about 4.5% of the output's
 * rms against the bf16-activation layer (measured on the synthetic
 * workloads; largest elements up to about 20%), so the layer is checked
 * against its own definition, not against moe_layer_forward's tolerance.
 * Shapes: H % 256 == 0, I % 128 == 0, H, I <= 2048, any T; other shapes
 * and layers with a shared expert (d.I_shared > 0) return
 * MOE_ERR_UNSUPPORTED.  Arguments as moe_layer_forward without `shared`.
 */
moe_status moe_layer_forward_act8(const uint16_t* x, const float* Wr,
                                  const float* bias, moe_fp8_ffn routed,
                                  moe_dims d, uint16_t* out,
                                  int32_t* topk_idx_out, float* topk_w_out,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * moe_permute without a workspace, for callers that cannot allocate device
 * memory: for example a plugin whose host framework passes it only the input
 * and output buffers of each call, or a serving loop whose device memory is
 * fixed at start-up.  The paper has no counterpart to this call.
 *
 * Same arguments, results and determinism as moe_permute, minus ws/ws_bytes.
 * Its scratch is one array compiled into the library (about 1.3 MB, held on
 * every GPU that loads the library until the process exits), sized for
 * T*k <= 65536 and E <= 512; larger sizes return MOE_ERR_UNSUPPORTED before
 * anything is enqueued.  It calls no allocator.
 *  - The first call on a device looks up the array's device address with
 *    that device current (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture on the device.
 *  - All calls on a device share the array, and it keeps the last call's
 *    contents: calls that overlap on the GPU race and give undefined
 *    results; order them on one stream (or with events).  Each call clears
 *    the status word it uses before its kernels run; every other scratch
 *    value is written before it is read.
 *  - An expert index outside [0, E) gives its pair tok_slot_row = -1 and no
 *    row, as in moe_permute, and sets MOE_DEV_BAD_EXPERT_INDEX in the fixed
 *    array's status word: moe_read_device_status(NULL, ...) reads it.
 */
moe_status moe_permute_static_scratch(const int32_t* topk_idx, moe_dims d,
                                      int32_t* expert_off, int32_t* row_token,
                                      int32_t* tok_slot_row, void* stream);

/*
 * Runtime cross-check of a layer call on sampled tokens, the GPU counterpart
 * of the colizig README's --cuda-verify (CLI reference), which checks the
 * CUDA path against the CPU path.  It recomputes the layer output of each
 * listed token on an arithmetic path independent of the layer kernels
 * (plain fp32 dot products, the E4M3 codes decoded from their bit fields
 * times their block scale, no tensor cores, no power-of-two normalisation),
 * from the routing the layer call produced, and compares it with `out`.
 *   x, routed, shared, shared_gate, d   as given to the layer call
 *                  (shared_gate NULL for moe_layer_forward)
 *   out            bf16 [T, H], the layer call's output
 *   topk_idx, topk_w  the layer call's routing ([T, k]; pass topk_idx_out /
 *                  topk_w_out of the layer call)
 *   tokens         int32 [n_tokens], token indices in [0, T); 1 <= n_tokens
 *                  <= 64
 *   result         float [3] out (device): worst |out - ref| / (1e-2 (|ref| +
 *                  rms(ref))) over the sampled outputs (<= 1: within the
 *                  layer tolerance; infinite for a NaN or an expert index
 *                  outside [0, E)), worst |out - ref|, rms(ref)
 *   ws, ws_bytes   scratch of at least moe_verify_workspace_bytes(d, n_tokens)
 * Enqueued on `stream` like every call; read `result` after synchronising.
 */
moe_status moe_verify_workspace_bytes(moe_dims d, int n_tokens, size_t* bytes);
moe_status moe_verify_layer(const uint16_t* x, moe_fp8_ffn routed,
                            const moe_fp8_ffn* shared, const float* shared_gate,
                            moe_dims d, const uint16_t* out,
                            const int32_t* topk_idx, const float* topk_w,
                            const int32_t* tokens, int n_tokens, float* result,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Copy the workspace's device status word to *status (MOE_DEV_* bits) after
 * synchronising `stream`.  Returns MOE_ERR_DEVICE_STATUS when any bit is set.
 * The word is cleared at the start of moe_route, moe_permute,
 * moe_expert_ffn_fp8 and moe_layer_forward.  With ws == NULL it reads the
 * status word of moe_permute_static_scratch's fixed array on the current
 * device instead (this does no allocation; on a device where that call has
 * not run yet it looks up the array's address first).  An unfinished or
 * invalid result is reported here rather than returned as a plausible
 * number (colizig README, "What this project is trying to prove" and
 * "Status": an incomplete subsystem returns an error, not a wrong number).
 */
moe_status moe_read_device_status(const void* ws, int32_t* status,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP8_H */
