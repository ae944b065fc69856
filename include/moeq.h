/*
 * moeq.h -- C ABI of the weight-only-quantised fused MoE library (libmoeq.so).
 *
 * The operations restate, as plain C, the interface documented on the vLLM API
 * pages "vllm.model_executor.layers.quantization.experts_int8" (W8A16) and
 * "vllm.model_executor.layers.quantization.moe_wna16" (W4A16):
 *
 *   ExpertsInt8MoEMethod.apply(layer, x, router_logits, top_k, renormalize, ...)
 *     = select_experts(...)  -> moe_topk_route
 *     + fused_experts(x, w13, w2, topk_weights, topk_ids, activation="silu",
 *                     use_int8_w8a16=True, w1_scale, w2_scale)
 *                            -> moe_align_block + moe_quant_forward
 *   quantize_in_place_and_get_scales(weight) -> moe_quantize_int8_per_channel
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer marked (device) is a CUDA device pointer on the current
 *   device; (host) pointers are ordinary host memory.  The caller owns every
 *   buffer.  No call allocates or frees device memory.
 * - All tensors are dense row-major with the shapes given; "bf16" is IEEE
 *   bfloat16 (uint16 storage), "f16" IEEE half.  Device pointers must be
 *   16-byte aligned.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *   work is enqueued on it and the call returns without waiting.
 * - Return value: an mq_status.  Argument errors are detected on the host
 *   before anything is launched, and leave every output untouched.  Errors
 *   found on the device (an expert id outside [0, E), a bounded wait that ran
 *   out) never trap: kernels set bits in a per-device status word, read with
 *   mq_device_status().
 * - mq_last_error_message() gives a human-readable reason for the most recent
 *   failing call on the calling thread.
 */
#ifndef MOEQ_H
#define MOEQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MQ_OK = 0,
  MQ_ERR_INVALID_ARG = 1,   /* bad pointer, shape, alignment or size          */
  MQ_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels cover */
  MQ_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed              */
  MQ_ERR_WORKSPACE = 4      /* workspace smaller than the query returned      */
} mq_status;

/* Bits of the device status word (see mq_device_status). */
#define MQ_DEV_BAD_EXPERT_ID  0x1u  /* a topk id outside [0, E); slot ignored   */
#define MQ_DEV_WAIT_TIMEOUT   0x2u  /* a pipeline wait gave up; output invalid  */

const char* mq_status_string(int status);
const char* mq_last_error_message(void);

/*
 * Waits for `stream`, then returns in *flags the OR of the MQ_DEV_* bits set
 * by kernels on the current device since the last call, and clears them.
 */
int mq_device_status(void* stream, uint32_t* flags);

/*
 * moe_quantize_int8_per_channel -- experts_int8 page,
 * quantize_in_place_and_get_scales (used by quantizing_weight_loader).
 *
 * For each row r of w (bf16 [rows, cols], device):
 *   scale[r] = max_c |w[r,c]| / 127           (float32, IEEE division)
 *   q[r,c]   = clamp(rint(w[r,c] / scale[r]), -127, 127)
 *              (float32 true division, round half to even)
 * A row of zeros gets scale 0 and codes 0.
 * Outputs: q int8 [rows, cols] (device), scale float32 [rows] (device).
 * For expert tensors pass rows = E * N (w13: N = 2I with the gate rows first,
 * then the up rows; w2: N = H) and cols = K.
 * Errors: MQ_ERR_INVALID_ARG for null pointers, rows/cols < 0, cols > 2^31,
 * misaligned pointers or cols % 8 != 0.
 */
int moe_quantize_int8_per_channel(const void* w, int64_t rows, int64_t cols,
                                  int8_t* q, float* scale, void* stream);

/*
 * moe_quantize_uint4_group -- produces the moe_wna16 page's W4A16 storage
 * (MoeWNA16Method.create_weights) from bf16 weights.  The page consumes
 * GPTQ/AWQ tensors already quantised; this call exists so that callers (and
 * the benchmark) can build such tensors on the device.
 *
 * Per row r and group g of `group_size` consecutive columns:
 *   lo = min(0, min w_g), hi = max(0, max w_g)
 *   s  = f16((hi - lo) / 15)      z = clamp(rint(-lo / s), 0, 15)
 *   q  = clamp(rint(w / s) + z, 0, 15)          (s == 0: z = 0, q = 0)
 * Outputs (device):
 *   qweight uint8 [rows, cols/2]   byte j = q[2j] | q[2j+1] << 4
 *   scales  f16   [rows, cols/group_size]
 *   qzeros  uint8 [rows/2, cols/group_size]  byte = z[2i] | z[2i+1] << 4
 * Errors: MQ_ERR_INVALID_ARG for odd rows, group_size not in {32,64,128,256}
 * or not dividing cols, null or misaligned pointers.
 */
int moe_quantize_uint4_group(const void* w, int64_t rows, int64_t cols, int group_size,
                             uint8_t* qweight, uint16_t* scales, uint8_t* qzeros,
                             void* stream);

/*
 * moe_topk_route -- the router of ExpertsInt8MoEMethod.apply
 * (select_experts with scoring_func="softmax", top_k, renormalize).
 *
 * logits float32 [T, E] (device).  For each token: p = softmax(logits[t]);
 * the k experts with the largest logits (ties -> lower index) fill slots
 * j = 0..k-1 in decreasing order; topk_w[t,j] = p[id_j], divided by the sum
 * of the k chosen p when renormalize != 0.
 * Outputs: topk_w float32 [T, k], topk_ids int32 [T, k] (device).
 * Limits: 1 <= k <= E <= 1024, k <= 32, T >= 0.
 */
int moe_topk_route(const float* logits, int T, int E, int k, int renormalize,
                   float* topk_w, int32_t* topk_ids, void* stream);

/*
 * Router options: the further select_experts arguments that
 * ExpertsInt8MoEMethod.apply and MoeWNA16Method.apply_monolithic pass on
 * (scoring_func, num_expert_group / topk_group of use_grouped_topk,
 * e_score_correction_bias, routed_scaling_factor).  The pages name them
 * without their arithmetic; this library reads them as follows.
 *   1. Score s_e of each expert: softmax over the token's logits
 *      (MQ_SCORING_SOFTMAX) or sigmoid(logit_e) (MQ_SCORING_SIGMOID).
 *   2. Selection key: the logit itself when e_score_correction_bias is NULL
 *      (either score rises with it); else the float32 s_e + bias[e].
 *   3. num_expert_group G > 1: experts [g*E/G, (g+1)*E/G) form group g,
 *      scored by its largest key; the topk_group best groups (ties: lower
 *      group) stay and every expert of the other groups is out.
 *   4. The k largest keys left (ties: lower index) fill slots 0..k-1.
 *   5. topk_w[t,j] = s_{id_j} (the bias steers the choice only), divided by
 *      the sum over the k chosen when renormalize != 0, times
 *      routed_scaling_factor.
 * {MQ_SCORING_SOFTMAX, r, 0, 0, NULL, 1.0f} is moe_topk_route's router.
 */
#define MQ_SCORING_SOFTMAX 0
#define MQ_SCORING_SIGMOID 1
typedef struct mq_route_opts {
  int scoring_func;                      /* MQ_SCORING_SOFTMAX or MQ_SCORING_SIGMOID */
  int renormalize;                       /* nonzero: renormalise over the k chosen */
  int num_expert_group;                  /* 0 or 1: no groups; else 2..32, divides E */
  int topk_group;                        /* groups kept, 1..num_expert_group (G > 1) */
  const float* e_score_correction_bias;  /* float32 [E] (device, 16-byte aligned) or NULL */
  float routed_scaling_factor;           /* finite; 1.0f leaves the weights as they are */
} mq_route_opts;

/*
 * moe_topk_route_ex -- moe_topk_route with router options (opts: host
 * pointer, read during the call).  Limits as moe_topk_route, and with
 * groups k <= topk_group * E / num_expert_group.  Errors:
 * MQ_ERR_INVALID_ARG for a NULL opts, an unknown scoring_func, a group
 * setting outside those limits or a non-finite scaling factor.
 */
int moe_topk_route_ex(const float* logits, int T, int E, int k, const mq_route_opts* opts,
                      float* topk_w, int32_t* topk_ids, void* stream);

/*
 * moe_align_capacity -- number of rows moe_align_block may produce:
 * round_up(T*k + min(E, T*k) * (block_m - 1), block_m).  Returns -1 for bad
 * arguments.
 */
int64_t moe_align_capacity(int T, int k, int E, int block_m);

/*
 * moe_align_block -- sorts the S = T*k token-slots (slot s = t*k + j) by
 * expert, stably, and pads every expert's segment to a multiple of block_m
 * with the sentinel S.  This is the grouping step fused_experts performs
 * before its grouped GEMMs.
 *
 * Inputs: topk_ids int32 [T, k] (device).
 * Outputs (device):
 *   sorted_slot_ids int32 [capacity]: entries [0, num_padded) hold expert 0's
 *       slots in increasing order, then padding, then expert 1's, ...;
 *       entries past num_padded are unspecified.
 *   block_expert    int32 [capacity / block_m]: expert of each block.
 *   expert_offsets  int32 [E + 1]: padded segment starts; [E] = num_padded.
 *   num_padded      int32 [1].
 * An expert with no slot gets no block.  A slot whose id is outside [0, E)
 * is left out and sets MQ_DEV_BAD_EXPERT_ID.
 * Limits: E <= 1024, 1 <= block_m <= 1024, capacity >= moe_align_capacity().
 */
int moe_align_block(const int32_t* topk_ids, int T, int k, int E, int block_m,
                    int32_t* sorted_slot_ids, int32_t* block_expert,
                    int32_t* expert_offsets, int32_t* num_padded,
                    int64_t capacity, void* stream);

/*
 * Weight formats of moe_quant_forward (bits, group_size, has_zp):
 *   W8A16 (experts_int8):  bits = 8, group_size = -1, has_zp = 0
 *     w13 int8 [E, 2I, H], w2 int8 [E, H, I],
 *     s13 float32 [E, 2I], s2 float32 [E, H]       (dequant = q * s)
 *   W4A16 (moe_wna16):     bits = 4, group_size in {32, 64, 128, 256}
 *     w13 uint8 [E, 2I, H/2], w2 uint8 [E, H, I/2]  (two codes per byte,
 *         even index in the low nibble)
 *     s13 f16 [E, 2I, H/gs], s2 f16 [E, H, I/gs]
 *     z13 uint8 [E, I, H/gs], z2 uint8 [E, H/2, I/gs] (zero points packed two
 *         output rows per byte, even row low) when has_zp = 1; with
 *         has_zp = 0 the zero point is 8 and z13/z2 must be NULL.
 *     dequant = (q - z) * s
 * In both, rows [0, I) of w13 are the gate projection (w1) and rows [I, 2I)
 * the up projection (w3), as quantizing_weight_loader lays them out.
 */

/*
 * moe_quant_forward_workspace -- bytes of device workspace moe_quant_forward
 * needs for these sizes (0 on bad arguments).
 */
size_t moe_quant_forward_workspace(int T, int H, int I, int E, int k,
                                   int bits, int group_size);

/*
 * moe_quant_forward -- fused_experts for the formats above:
 *   for every token t and slot j with e = topk_ids[t,j]:
 *     h  = dequant(w13[e]) . x[t]             (2I values)
 *     a  = silu(h[0:I]) * h[I:2I]             silu(u) = u / (1 + exp(-u))
 *     y  = dequant(w2[e]) . a                 (H values)
 *     out[t] += topk_w[t,j] * y
 * x bf16 [T, H] (device), topk_w float32 [T, k], topk_ids int32 [T, k]
 * (device, e.g. from moe_topk_route), out bf16 [T, H] (device; either x
 * itself -- fused_experts' inplace, x is read before any output is written --
 * or not overlapping x at all).  The block alignment runs inside, in the
 * workspace.
 * Accumulation is float32; the intermediate a is rounded to bf16.
 * Limits: H % 128 == 0, I % 128 == 0, E <= 1024, 1 <= k <= min(E, 32).
 * Errors: MQ_ERR_INVALID_ARG (null/misaligned pointers, bad shapes),
 * MQ_ERR_UNSUPPORTED (format or sizes outside the limits),
 * MQ_ERR_WORKSPACE (ws_bytes below the query).
 */
int moe_quant_forward(const void* x, int T, int H, int I, int E, int k,
                      int bits, int group_size, int has_zp,
                      const void* w13, const void* w2,
                      const void* s13, const void* s2,
                      const uint8_t* z13, const uint8_t* z2,
                      const float* topk_w, const int32_t* topk_ids,
                      void* workspace, size_t ws_bytes,
                      void* out, void* stream);

/*
 * Option flags of moe_quant_forward_ex (0 gives moe_quant_forward).
 *
 * MQ_FWD_W8_UINT8 (bits = 8): w13 / w2 hold uint8 codes u, the 8-bit form of
 *     "vllm.model_executor.layers.quantization.moe_wna16" (MoeWNA16Method
 *     with num_bits 8, group_size -1: qweight uint8 [E, N, K], scales
 *     [E, N, 1], optional qzeros uint8 [E, N, 1]).  dequant = (u - z) * s
 *     with z = 128, or with has_zp = 1 z13 uint8 [E, 2I] / z2 uint8 [E, H]
 *     (one zero point per output row).
 * MQ_FWD_SCALE_F16, MQ_FWD_SCALE_BF16 (bits = 8, at most one): the scales
 *     are float16 / bfloat16 (the moe_wna16 parameter dtype) instead of
 *     float32.
 * MQ_FWD_SCALE_PER_TENSOR (bits = 8): one scale per expert and weight
 *     tensor, s13 [E] and s2 [E] -- the "tensor" strategy of the
 *     compressed-tensors int8 MoE config, chosen there when the weight scale
 *     has fewer elements than experts x output rows.
 * MQ_FWD_ACT_F16: x and out are float16 instead of bfloat16 (experts_int8
 *     lists both as supported activation dtypes).
 * MQ_FWD_ROUTER_WEIGHT_ON_INPUT: fused_experts' apply_router_weight_on_input
 *     (a name only on the pages; read as): the router weight scales each
 *     expert's input, h = dequant(w13[e]) . (topk_w[t,j] * x[t]), and the
 *     expert's output is added unweighted, out[t] += y.
 */
#define MQ_FWD_W8_UINT8 0x1u
#define MQ_FWD_SCALE_F16 0x2u
#define MQ_FWD_SCALE_BF16 0x4u
#define MQ_FWD_SCALE_PER_TENSOR 0x8u
#define MQ_FWD_ACT_F16 0x10u
#define MQ_FWD_ROUTER_WEIGHT_ON_INPUT 0x20u
/*
 * Kernel selection (no counterpart on the pages; the result is the same
 * forward either way, up to float32 summation order).  The expert GEMMs
 * stream TMA-staged weight tiles through converter warps that dequantise
 * them exactly; the products run either on tcgen05 (a single issuing thread
 * per SM, accumulators in tensor memory) or, for experts holding a few
 * token-slots, on warp-level MMAs issued by the converter warps themselves.
 * By default both GEMMs run on tcgen05 (the faster choice measured on GB300
 * for every GEMM and batch size); the warp-level MMAs run when forced.
 * For 8-bit layers both GEMMs can also run in one persistent launch on
 * tcgen05 (token tiles of 16, 32, 64 or 128 rows, as in two launches): each
 * SM streams its gate/up weight tiles and then its down weight tiles without
 * a kernel boundary, and the down GEMM of a token tile starts as soon as all
 * gate/up tiles of that token tile are done.  By default that launch serves
 * 8-bit batches of 65 to 2048 tokens in layers of more than 16 experts, and
 * of one or two tokens in layers of up to 16 experts.  It relies on all of
 * its CTAs (one per SM, at most the SM count) becoming resident together,
 * as they do unless kernels of other streams hold SMs for longer than a
 * second; its waits on other CTAs give up after a second with
 * MQ_DEV_WAIT_TIMEOUT.
 * MQ_FWD_PATH_TENSOR_CORE forces tcgen05 for both GEMMs in two launches,
 * MQ_FWD_PATH_DECODE the warp-level MMAs for both (MQ_ERR_UNSUPPORTED for
 * uint4 with group_size 32 or 64), MQ_FWD_PATH_LAYER the one-launch layer
 * (MQ_ERR_UNSUPPORTED for uint4); at most one of the three.  Each fits the
 * workspace the query returns.
 */
#define MQ_FWD_PATH_TENSOR_CORE 0x40u
#define MQ_FWD_PATH_DECODE 0x80u
#define MQ_FWD_PATH_LAYER 0x100u

/*
 * moe_quant_forward_ex -- moe_quant_forward with option flags (above).
 * Arguments are those of moe_quant_forward, with x / out in the activation
 * dtype the flags select.  out may be x itself (fused_experts' inplace =
 * True: x is read only before out is written); any other overlap is
 * rejected.  has_zp = 1 with bits = 8 requires MQ_FWD_W8_UINT8.
 * Errors: as moe_quant_forward; flags that do not apply to the format (or
 * unknown bits) give MQ_ERR_UNSUPPORTED.
 */
int moe_quant_forward_ex(const void* x, int T, int H, int I, int E, int k,
                         int bits, int group_size, int has_zp,
                         const void* w13, const void* w2,
                         const void* s13, const void* s2,
                         const uint8_t* z13, const uint8_t* z2,
                         const float* topk_w, const int32_t* topk_ids,
                         void* workspace, size_t ws_bytes,
                         void* out, unsigned flags, void* stream);

/*
 * moe_quant_forward_logits -- the whole of ExpertsInt8MoEMethod.apply(layer,
 * x, router_logits, top_k, renormalize, ...) in one call: select_experts
 * (softmax, top-k, optional renormalisation; moe_topk_route's arithmetic)
 * followed by fused_experts (moe_quant_forward_ex).  router_logits float32
 * [T, E] (device); the chosen weights and ids stay in the workspace.  When
 * T * k * ceil(E / 32) <= 512 the routing runs inside the align kernel (one
 * launch fewer); either way the result is bitwise that of moe_topk_route
 * followed by moe_quant_forward_ex.  Other arguments, limits and errors as
 * moe_quant_forward_ex; the workspace size comes from
 * moe_quant_forward_logits_workspace.
 */
size_t moe_quant_forward_logits_workspace(int T, int H, int I, int E, int k,
                                          int bits, int group_size);
int moe_quant_forward_logits(const void* x, const float* router_logits,
                             int T, int H, int I, int E, int k, int renormalize,
                             int bits, int group_size, int has_zp,
                             const void* w13, const void* w2,
                             const void* s13, const void* s2,
                             const uint8_t* z13, const uint8_t* z2,
                             void* workspace, size_t ws_bytes,
                             void* out, unsigned flags, void* stream);

/*
 * moe_quant_forward_logits_ex -- moe_quant_forward_logits with router
 * options (see mq_route_opts; opts replaces renormalize), as
 * MoeWNA16Method.apply_monolithic passes them: the result is bitwise that of
 * moe_topk_route_ex followed by moe_quant_forward_ex.  Workspace from
 * moe_quant_forward_logits_workspace; other arguments, limits and errors as
 * moe_quant_forward_logits and moe_topk_route_ex.
 */
int moe_quant_forward_logits_ex(const void* x, const float* router_logits,
                                int T, int H, int I, int E, int k,
                                const mq_route_opts* opts,
                                int bits, int group_size, int has_zp,
                                const void* w13, const void* w2,
                                const void* s13, const void* s2,
                                const uint8_t* z13, const uint8_t* z2,
                                void* workspace, size_t ws_bytes,
                                void* out, unsigned flags, void* stream);

/*
 * moe_quant_forward_noalloc -- moe_quant_forward without a workspace
 * argument.  (The pages have no counterpart: their forward allocates its
 * intermediates through torch.)
 *
 * For callers that cannot allocate device memory or hand over a workspace:
 * e.g. a plugin inside a host application that owns all device memory
 * through its own allocator and passes the plugin only its input and output
 * buffers, or a path on which an allocation (a synchronising call that may
 * fail) is not allowed.  The scratch the forward needs lives in a fixed
 * 32 MiB array inside libmoeq.so, held on every GPU that loads the library
 * until the process exits.  Nothing is allocated per call.
 *
 * Arguments, layouts and results are those of moe_quant_forward.  Sizes whose
 * scratch (moe_quant_forward_workspace) exceeds 32 MiB are rejected with
 * MQ_ERR_UNSUPPORTED and a message naming both sizes; nothing is launched.
 * The first call on each device looks up that device's address of the array
 * (a CUDA runtime query, no allocation), so make that first call before any
 * stream capture.  All calls on a device share the one array, which keeps
 * the previous call's contents (nothing in it needs to start at zero): calls
 * whose GPU work overlaps -- on different streams, or from several host
 * threads -- race on it and must be serialised by the caller.
 * The array's device address is looked up once per device and cached for the
 * life of the process (as is the status word's, for every call): do not keep
 * using the library on a device after cudaDeviceReset() on it, since the
 * module's arrays may then live at other addresses.
 */
int moe_quant_forward_noalloc(const void* x, int T, int H, int I, int E, int k,
                              int bits, int group_size, int has_zp,
                              const void* w13, const void* w2,
                              const void* s13, const void* s2,
                              const uint8_t* z13, const uint8_t* z2,
                              const float* topk_w, const int32_t* topk_ids,
                              void* out, void* stream);

/*
 * Instrumentation (no counterpart on the pages; used by the benchmark).
 *
 * mq_kernel_launch_count: kernels this library has launched in this process.
 * mq_profile_enable(on): while on, every kernel launch is bracketed by a pair
 *   of CUDA events recorded on the launch's own stream (costs a few
 *   microseconds of host time per launch).
 * mq_profile_read(total_ms, launches, n_slots): waits for the recorded
 *   events, writes per slot the summed device time in milliseconds and the
 *   number of timed launches (host arrays of n_slots entries), and resets.
 *   Slots are the MQ_PROF_* values.
 */
#define MQ_PROF_QUANT   0
#define MQ_PROF_ROUTE   1
#define MQ_PROF_ALIGN   2
#define MQ_PROF_GEMM1   3
#define MQ_PROF_GEMM2   4
#define MQ_PROF_COMBINE 5
#define MQ_PROF_GATHER  6
#define MQ_PROF_ACTF16  7
#define MQ_PROF_LAYER   8  /* both expert GEMMs in one launch (MQ_FWD_PATH_LAYER) */
#define MQ_PROF_SLOTS   9

long long mq_kernel_launch_count(void);
int mq_profile_enable(int on);
int mq_profile_read(double* total_ms, long long* launches, int n_slots);

/*
 * Testing aid for the bounded waits (no counterpart on the pages).
 * mq_test_layer_wait_extra(extra): adds `extra` (>= 0) to the number of
 *   gate/up completions that each down unit of the one-launch layer
 *   (MQ_FWD_PATH_LAYER) waits for, in later launches.  With extra > 0 those
 *   waits cannot end: after their limit of about a second the kernel stops
 *   its CTAs cleanly, the forward's output is invalid and
 *   mq_device_status reports MQ_DEV_WAIT_TIMEOUT; later forwards run
 *   normally.  0 restores normal operation.  Returns MQ_OK, or
 *   MQ_ERR_INVALID_ARG for extra < 0.  Process-wide; not for concurrent
 *   forwards.
 */
int mq_test_layer_wait_extra(int extra);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ_H */
