/*
 * moe.h - C ABI of the grouped-expert MoE FFN library for GB300 (sm_103a).
 *
 * The layer: per token, top-k softmax routing over E experts; every routed expert and the
 * always-on shared expert apply a W8A8 SwiGLU FFN (int8 gate/up GEMM, SiLU(gate)*up,
 * requantisation, int8 down GEMM); the expert outputs are combined with the routing weights
 * (shared expert weight 1). All routed experts are computed as ONE grouped computation
 * instead of one launch per expert: the remedy the page "Qwen3.6-35B-A3B Linux v1.0.4:
 * ~2.7s fixed per-request TTFT = ~4,900 serialized per-expert NPU execs ..." proposes in
 * section "The fix (concatenated-expert dispatch)" (one run per operator per layer-block,
 * N = TOP_K x 2 x IM_EXP). Batched decode and small batches (T <= 64 rows) deduplicate
 * experts across rows and stream each unique expert's int8 weights once with an int8 dot,
 * as the page "[job] Strix Halo: multi-session serving ... #145", section "Status", item
 * "Next" asks. The expert weights may instead be NVFP4 (moe_pack_weights_nvfp4), the format
 * the same page keeps for the routed experts; the activations stay int8.
 *
 * Conventions (every entry point):
 *  - Data pointers are DEVICE pointers unless a comment says host. Tensors are row-major
 *    and contiguous; every data pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls that
 *    take a stream are asynchronous on it and never synchronise the host, except where
 *    stated.
 *  - Errors: argument and shape errors are detected on the host and returned before any
 *    work is queued. Device-side failures (a bounded wait that ran out, an index out of
 *    range) set a sticky error word in the plan, read by moe_get_error. No entry point
 *    aborts, throws, or falls back to a CPU path.
 *  - Numerics: integer results (routing indices, permutation, int32 accumulators) are
 *    exact; floating point is fp32 (NVFP4 weights: see moe_pack_weights_nvfp4).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, T out of range        */
  MOE_ERR_UNSUPPORTED = 2,  /* shape the kernels do not support (see moe_plan)          */
  MOE_ERR_OOM = 3,          /* device allocation failed                                 */
  MOE_ERR_CAPACITY = 4,     /* T larger than the plan's max_tokens                      */
  MOE_ERR_CUDA = 5,         /* a CUDA runtime call failed                               */
  MOE_ERR_TIMEOUT = 6,      /* a device-side bounded wait ran out (sticky)              */
  MOE_ERR_DEVICE = 7,       /* a device-side range check failed (sticky)                */
  MOE_ERR_NO_DEVICE = 8     /* no CUDA device, or not an sm_103 GPU                     */
} moe_status;

typedef struct moe_plan_s* moe_plan_t;      /* shapes + workspace, one per layer shape   */
typedef struct moe_packed_s* moe_packed_t;  /* one layer's weights, repacked for the GPU */

/* One layer's quantised weights (device pointers, caller-owned).
 * Routed experts: w_gate, w_up int8 [E, I, H]; w_down int8 [E, H, I];
 *                 s_gate, s_up fp32 [E, I]; s_down fp32 [E, H] (per output channel).
 * Shared expert (only when the plan has I_shared > 0, else all NULL):
 *                 sh_gate, sh_up int8 [I_shared, H]; sh_down int8 [H, I_shared];
 *                 sh_s_gate, sh_s_up fp32 [I_shared]; sh_s_down fp32 [H].
 * Dequantised weight = int8 value * scale of its output channel. */
typedef struct {
  const int8_t* w_gate;
  const int8_t* w_up;
  const int8_t* w_down;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
  const int8_t* sh_gate;
  const int8_t* sh_up;
  const int8_t* sh_down;
  const float* sh_s_gate;
  const float* sh_s_up;
  const float* sh_s_down;
} moe_weights;

/* One layer's NVFP4 expert weights (device pointers, caller-owned): the format the page
 * "[job] Strix Halo: multi-session serving (parallel or sequential) and long context,
 * Flash-Next and the 27B #145" keeps for the routed experts (its comment of Oct 19, which
 * compares the FP4 formats). Every weight row (reduction dimension contiguous) is stored as
 * 4-bit E2M1 codes (OCP Microscaling Formats v1.0, FP4: sign, 2 exponent bits with bias 1, 1
 * mantissa bit), two per byte with element 2j in the low nibble, plus one E4M3 block scale
 * byte (finite, non-negative) per 16 consecutive elements, plus one fp32 scale per matrix:
 *   dequantised weight = e2m1(code) * e4m3(block scale) * matrix scale.
 * Routed experts: w_gate, w_up uint8 [E, I, H/2]; w_down uint8 [E, H, I/2];
 *                 b_gate, b_up uint8 [E, I, H/16]; b_down uint8 [E, H, I/16];
 *                 g_gate, g_up, g_down fp32 [E].
 * Shared expert (only when the plan has I_shared > 0, else all NULL): sh_gate, sh_up
 *                 [I_shared, H/2]; sh_down [H, I_shared/2]; sh_b_gate, sh_b_up
 *                 [I_shared, H/16]; sh_b_down [H, I_shared/16]; sh_g fp32 [3] (gate, up,
 *                 down matrix scales).
 * The activations stay int8 per token, as in the int8 layer. */
typedef struct {
  const uint8_t* w_gate;
  const uint8_t* w_up;
  const uint8_t* w_down;
  const uint8_t* b_gate;
  const uint8_t* b_up;
  const uint8_t* b_down;
  const float* g_gate;
  const float* g_up;
  const float* g_down;
  const uint8_t* sh_gate;
  const uint8_t* sh_up;
  const uint8_t* sh_down;
  const uint8_t* sh_b_gate;
  const uint8_t* sh_b_up;
  const uint8_t* sh_b_down;
  const float* sh_g;
} moe_weights_nvfp4;

/* Create a plan for one layer shape and allocate its workspace for up to max_tokens
 * tokens per call (the only allocation on the forward path's behalf). The plan is the
 * persistent per-layer-shape state that the page "Qwen3.6-35B-A3B Linux v1.0.4: ~2.7s fixed
 * per-request TTFT ..." (section "Evidence", item 1, and "Request" (b)) finds missing: no
 * buffer is created or destroyed per call.
 *   E: routed experts (1..256); top_k: 1..min(E, 8); H: hidden size; I: routed expert
 *   intermediate size; I_shared: shared expert intermediate size, 0 = no shared expert.
 * Supported shapes: H a multiple of 128, I (and I_shared when > 0) multiples of 64; H <= 8192;
 *   I, I_shared <= 4096. Otherwise MOE_ERR_UNSUPPORTED.
 * Uses the current CUDA device. *out receives the handle; release with moe_plan_destroy. */
MOE_API moe_status moe_plan(int E, int top_k, int H, int I, int I_shared, int max_tokens,
                    moe_plan_t* out);

/* Free the plan and its workspace. Work queued on it must have completed. */
MOE_API moe_status moe_plan_destroy(moe_plan_t plan);

/* Register one layer's weights with the plan's shapes. Allocates and fills (on `stream`)
 * the device copy the tensor-core path reads: the int8 gate and up rows interleaved in
 * channel pairs (row 2i = gate channel i, row 2i+1 = up channel i, per expert; the shared
 * expert likewise), still int8, plus the maxima over weight rows of the sum of squared codes
 * that the GEMMs' exactness test uses. The down GEMM and the decode path read the caller's
 * int8 arrays and scales directly, so they must stay alive and unchanged while the packed
 * handle is in use. Release with moe_packed_destroy. */
MOE_API moe_status moe_pack_weights(moe_plan_t plan, const moe_weights* w, void* stream,
                            moe_packed_t* out);
MOE_API moe_status moe_packed_destroy(moe_packed_t packed);

/* Register one layer's NVFP4 expert weights (moe_weights_nvfp4). Allocates and fills (on
 * `stream`) the tensor-core copy: every (128-row, 128-K) weight tile's codes and block scales
 * in one contiguous 9216-byte block, gate and up rows interleaved in channel pairs, plus the
 * matrix scales as per-row scales. The decode path reads the caller's arrays in place, so
 * they must stay alive and unchanged while the handle is in use. Also queues a check of every
 * block scale byte; a negative or NaN one sets the plan's sticky error word to
 * MOE_ERR_DEVICE (read by moe_get_error). With the returned handle, moe_forward and
 * moe_route_forward compute the same layer with these weights:
 *   per weight row, acc = sum over elements of q * e2m1(code) * e4m3(block scale)
 *   (q = the int8 activation or h code); then g = (float(acc) * s_x) * g_gate, u likewise,
 *   h = SiLU(g) * u requantised per row as in the int8 layer, and
 *   d = (float(acc_d) * s_h) * g_down, combined as in the int8 layer.
 * The dispatch is the int8 layer's: T <= the plan's decode threshold runs the deduplicated
 * weight-streaming kernels, which form acc exactly (int64) and round it once to fp32; larger
 * T runs the grouped tensor-core GEMMs, which decode each weight exactly to fp16 and
 * accumulate the products in fp32 (rounded as the tensor core adds them). Pointers must be
 * 16-byte aligned. */
MOE_API moe_status moe_pack_weights_nvfp4(moe_plan_t plan, const moe_weights_nvfp4* w, void* stream,
                                  moe_packed_t* out);

/* Top-k softmax routing (warp per token): the "top-8" selection of routed experts per token
 * that the page "Qwen3.6-35B-A3B Linux v1.0.4 ..." (section "The fix (concatenated-expert
 * dispatch)") dispatches, with the softmax weights of the selected experts.
 *   logits fp32 [T, E] -> idx int32 [T, top_k], w fp32 [T, top_k].
 * Selection compares the fp32 logits; ties go to the lowest expert id; slots are ordered by
 * logit descending, then id ascending. w is a softmax over the selected logits, so each
 * row sums to 1 (within 1e-6). Logits must be finite. 1 <= T <= max_tokens. */
MOE_API moe_status moe_route(moe_plan_t plan, const float* logits, int T, int32_t* idx, float* w,
                     void* stream);

/* The MoE layer: y fp32 [T, H] = sum_j w[t,j] * expert_{idx[t,j]}(x[t]) + shared(x[t]),
 * computed as one grouped (concatenated-expert) computation per operator, as the page
 * "Qwen3.6-35B-A3B Linux v1.0.4 ..." proposes in section "The fix (concatenated-expert
 * dispatch)": gate and up concatenated (N = top_k x 2 x I per token), one GLU region over
 * all experts, then the down projection and the weighted combine.
 *   x bf16 [T, H] (raw bf16 bits); idx, w as produced by moe_route (any valid top-k
 *   routing: idx[t,*] distinct, in [0, E)); y is overwritten. 1 <= T <= max_tokens: an
 *   empty batch (T = 0) is MOE_ERR_INVALID_ARG, a larger one MOE_ERR_CAPACITY, both
 *   returned before any work is queued.
 * T <= the plan's decode threshold (moe_plan_set_decode_rows; default 24) runs the
 * deduplicated weight-streaming decode kernels; larger T runs the grouped tensor-core GEMMs.
 * Both give identical integer accumulators. Allocates nothing, never
 * synchronises, and may be captured in a CUDA graph. The workspace is per plan: calls on
 * one plan must not overlap in time (use one plan per concurrent stream). */
MOE_API moe_status moe_forward(moe_plan_t plan, moe_packed_t packed, const uint16_t* x, int T,
                       const int32_t* idx, const float* w, float* y, void* stream);

/* moe_route followed by moe_forward, with the routing done inside the forward's first kernel
 * (the step before the layer fused into it; page "Qwen3.6-35B-A3B Linux v1.0.4 ...",
 * section "The fix (concatenated-expert dispatch)": fewer dispatches per layer). logits fp32
 * [T, E] in; idx int32 [T, k] and w fp32 [T, k] are written exactly as moe_route writes them
 * (the same selection and softmax code) and y as moe_forward computes it from them. Same
 * arguments, errors and conditions as moe_forward; logits must be 16-byte aligned. Uses a
 * per-plan counter (calls on one plan must not overlap in time; moe_clear_error resets it
 * after a call that failed). */
MOE_API moe_status moe_route_forward(moe_plan_t plan, moe_packed_t packed, const uint16_t* x,
                                     int T, const float* logits, int32_t* idx, float* w, float* y,
                                     void* stream);

/* Dispatch threshold of moe_forward on this plan: T <= rows runs the weight-streaming decode
 * kernels (each unique expert's weights read once, rows applied 8 at a time), larger T the
 * grouped GEMMs. 0 <= rows <= 64 (else MOE_ERR_INVALID_ARG); 0 sends every call to the
 * grouped GEMMs. Default 24: measured on GB300 for a 35B-A3B-shaped layer with the routing
 * inside the forward, streaming is the faster path up to T=24 and the grouped GEMMs from
 * T=32. The crossover between the two paths is a measured property of the GPU and
 * the layer shape (the page "[job] Strix Halo ... #145", "Done / measured", on the grouped
 * threshold), so it is a setting rather than a constant. Host-only; takes effect on the next
 * moe_forward. */
MOE_API moe_status moe_plan_set_decode_rows(moe_plan_t plan, int rows);

/* Sticky device-side error word of the plan (synchronises the device). MOE_OK if none. */
MOE_API moe_status moe_get_error(moe_plan_t plan);
/* Clear the sticky error word (synchronises the device). */
MOE_API moe_status moe_clear_error(moe_plan_t plan);
/* Self-test of device-side failure detection: queues on `stream` one kernel whose single
 * thread waits, with the library's bounded wait, on a barrier that nothing completes. After
 * the wait's time limit (2 s) it gives up and sets the plan's sticky error word to
 * MOE_ERR_TIMEOUT; the context stays usable (moe_clear_error, then any other call). Returns
 * MOE_ERR_INVALID_ARG for a NULL plan, MOE_ERR_CUDA if the launch fails. Asynchronous. */
MOE_API moe_status moe_selftest_wait_timeout(moe_plan_t plan, void* stream);

/* Short static description of a status code. */
MOE_API const char* moe_status_string(moe_status s);

/* ---- test taps: copies of intermediate results of the last moe_forward ----------------
 * moe_debug_enable(plan, 1) allocates tap buffers and makes later forwards also write the
 * accumulators: the int32 taps after a forward with int8 weights, the fp64 taps after one
 * with NVFP4 weights (the other kind then holds no valid data) (it is the one call besides moe_plan/moe_pack_weights that allocates).
 * Rows are in the plan's row order: rows [0, T) are the shared expert's (row t = token t),
 * when I_shared > 0; then the routed assignments, grouped by expert id and, inside an
 * expert, by (token, slot) ascending. moe_debug_tap copies one tap to HOST memory
 * `dst_host` (synchronises the device); `bytes` must equal the tap's size for the last
 * forward's T, as given by moe_debug_tap_bytes. */
typedef enum {
  MOE_TAP_COUNTS = 0,   /* int32 [E]              tokens per routed expert               */
  MOE_TAP_OFFSETS = 1,  /* int32 [E + 1]          exclusive prefix of COUNTS             */
  MOE_TAP_PERM = 2,     /* int32 [T*top_k]        flat slot t*top_k+j of each routed row */
  MOE_TAP_QX = 3,       /* int8  [T, H]           quantised activations                  */
  MOE_TAP_SX = 4,       /* fp32  [T]              activation scales                      */
  MOE_TAP_ACC_GU = 5,   /* int32 [R, 2*Imax]      gate accumulators, then up accumulators */
  MOE_TAP_HQ = 6,       /* int8  [R, Imax]        requantised SiLU(gate)*up               */
  MOE_TAP_SH = 7,       /* fp32  [R]              scales of HQ                            */
  MOE_TAP_ACC_D = 8,    /* int32 [R, H]           down accumulators                       */
  MOE_TAP_ACC_GU_F64 = 9,  /* fp64 [R, 2*Imax]    NVFP4 weights: gate, then up accumulators */
  MOE_TAP_ACC_D_F64 = 10   /* fp64 [R, H]         NVFP4 weights: down accumulators          */
} moe_tap;              /* R = T*top_k + (I_shared > 0 ? T : 0); Imax = max(I, I_shared)   */

MOE_API moe_status moe_debug_enable(moe_plan_t plan, int on);
MOE_API size_t moe_debug_tap_bytes(moe_plan_t plan, int which);
MOE_API moe_status moe_debug_tap(moe_plan_t plan, int which, void* dst_host, size_t bytes);

/* ---- per-stage device timing (benchmark instrument) ----------------------------------
 * When enabled, every moe_forward also records CUDA events around its kernels on the call's
 * stream (no extra synchronisation). moe_profile_read synchronises on those events and
 * writes, for the chosen path (0 = prefill, 1 = decode), the summed device milliseconds of
 * each stage over all forwards since the previous read into ms_out[4] and their number into
 * *calls, then starts a new accumulation. Stages: prefill {permute+quant, gate/up GEMM,
 * requant, down GEMM adding into y}; decode {dedup + quant, gate/up stream +
 * requant, down stream adding into y, 0}. Not for use inside CUDA graph capture. */
MOE_API moe_status moe_profile_enable(moe_plan_t plan, int on);
MOE_API moe_status moe_profile_read(moe_plan_t plan, int path, float* ms_out, int* calls);

/* ---- the two steps around the layer in a stacked prefill -------------------------------
 * Router projection: logits fp32 [T, E] = float(x bf16 [T, H]) @ w_router fp32 [H, E],
 * fp32 accumulation. Residual: x[t,h] <- bf16_round_nearest_even(float(x[t,h]) + y[t,h]),
 * x bf16 [T, H] updated in place, y fp32 [T, H]. Neither needs a plan. */
/* Stacked-prefill layer input: when y is not NULL, first x <- bf16_rne(float(x) + y) (the
 * residual update, x updated in place); then x_in <- bf16_rne(float(x) / sqrt(mean_h(x^2) +
 * 1e-6)) per token (a parameter-free RMS pre-norm of the next layer's input). x, x_in bf16
 * [T, H]; y fp32 [T, H] or NULL. One block per token, fp32 arithmetic. */
MOE_API moe_status moe_rmsnorm_residual(uint16_t* x, const float* y, uint16_t* x_in, int T, int H,
                                        void* stream);
/* Router projection on the tensor cores. moe_router_pack splits w_router fp32 [H, E] into
 * three bf16 parts hi + mid + lo (exact to 2^-26 relative) and stores them as packed bf16
 * [3E, H] (caller-allocated, 6*H*E bytes; a one-time step per router weight): blocks of 16
 * experts, each block the hi rows, then the mid rows, then the lo rows of its experts.
 * moe_router_logits_packed computes logits fp32 [T, E] = float(x bf16 [T, H]) @ W: per
 * expert three bf16 dot products over H (exact products, fp32 accumulation), added as
 * (hi + mid) + lo. H a multiple of 64, E a multiple of 16. Encodes two TMA descriptors on the
 * host per call; MOE_ERR_INVALID_ARG on a bad size or an unaligned pointer. */
MOE_API moe_status moe_router_pack(const float* w_router, int H, int E, uint16_t* packed,
                                   void* stream);
MOE_API moe_status moe_router_logits_packed(const uint16_t* x, const uint16_t* packed, int T,
                                            int H, int E, float* logits, void* stream);
MOE_API moe_status moe_router_logits(const uint16_t* x, const float* w_router, int T, int H, int E,
                             float* logits, void* stream);
MOE_API moe_status moe_residual_add(uint16_t* x, const float* y, int T, int H, void* stream);

/* ---- allocation-free batched decode ---------------------------------------------------
 * The source pages have no counterpart of this entry point; it exists for callers that
 * cannot allocate device memory on their call path: a plugin inside a host runtime that owns
 * every device allocation and forbids its guests from calling cudaMalloc, or a serving loop
 * that cannot afford the implicit device synchronisation of cudaMalloc/cudaFree between
 * steps. moe_plan allocates a workspace, so such callers use this instead for decode-sized
 * batches.
 *
 * Computes exactly what moe_forward computes for 1 <= T <= 8 rows (the deduplicated
 * weight-streaming decode kernels), taking the shapes directly instead of a plan:
 *   E, top_k, H, I, I_shared, w (caller-owned int8 weights and fp32 scales, as in
 *   moe_weights), x bf16 [T, H], idx int32 [T, top_k], w fp32 [T, top_k] -> y fp32 [T, H].
 *   status: optional device int32; receives the call's device-side error word (0 = ok,
 *   MOE_ERR_DEVICE for an expert id out of range or repeated within a token).
 * It allocates nothing: its scratch (at most 2 MiB: per-token codes, the unique-expert
 * list, row maps, fp32 SiLU(gate)*up rows) is a file-scope __device__ array inside the
 * library, present on every GPU that loads the library until the process exits. Limits:
 * T <= 8 (else MOE_ERR_CAPACITY), E <= 256, top_k <= 8, H <= 8192 and a multiple of 128,
 * I and I_shared <= 4096 and multiples of 64 (else MOE_ERR_UNSUPPORTED). The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress) and keeps it for
 * the life of the process; make that first call before any stream capture, and do not call
 * this entry point again on a device after cudaDeviceReset (the array may then move). Every
 * call shares the one array and keeps the previous call's contents (only the error word is
 * cleared per call): calls that overlap on the GPU - on two streams, or from two host
 * threads - race and corrupt each other's results; serialise them. */
MOE_API moe_status moe_forward_decode_static(int E, int top_k, int H, int I, int I_shared,
                                             const moe_weights* w, const uint16_t* x, int T,
                                             const int32_t* idx, const float* wts, float* y,
                                             int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
