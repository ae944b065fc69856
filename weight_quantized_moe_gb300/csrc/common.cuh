// Shared device helpers for the moeq kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/moeq.h"

#define MQ_HIDDEN __attribute__((visibility("hidden")))

namespace mq {

// Per-device status word: kernels OR MQ_DEV_* bits into it.  Each launcher
// receives its device address from the API layer.
__device__ __forceinline__ void flag(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ unsigned lane_id() {
  unsigned r;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Programmatic dependent launch.  The forward's kernels are launched so that
// each may start while its predecessor in the stream is still running.
// pdl_wait() blocks until the predecessor has completed and its writes are
// visible; pdl_trigger() lets the successor begin launching.  Without the
// launch attribute both are no-ops.
//
// Ordering the kernels rely on: the align kernel and the small kernels
// (gather, act conversion, combine) trigger only after their own wait; the
// expert GEMMs trigger early, before their wait, so that the next GEMM can
// set up and start its weight stream.  A GEMM therefore may start while the
// kernel two launches back is still running (e.g. the down GEMM while the
// gather runs), but never before the align kernel has completed: before its
// own wait a GEMM may read only the align kernel's outputs (the chunk table,
// the sorted slots, the expert counts and offsets), the router's outputs
// written before the align kernel, and the weights.  Everything else waits.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// silu(u) * v in float32; silu(u) = u / (1 + exp(-u)).
__device__ __forceinline__ float silu_mul(float u, float v) {
  return u / (1.0f + expf(-u)) * v;
}

}  // namespace mq

// Launch with the programmatic-stream-serialization attribute (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------------------
// Internal launchers (one translation unit each, not exported).
// ---------------------------------------------------------------------------
MQ_HIDDEN cudaError_t launch_quant_int8(const void* w, int64_t rows, int64_t cols, int8_t* q,
                                        float* scale, cudaStream_t st);
MQ_HIDDEN cudaError_t launch_quant_uint4(const void* w, int64_t rows, int64_t cols, int gs,
                                         uint8_t* qw, uint16_t* sc, uint8_t* qz, cudaStream_t st);
MQ_HIDDEN cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm,
                                   float* topk_w, int32_t* topk_ids, cudaStream_t st);
// Router options beyond softmax + renormalisation (moe_topk_route_ex).
struct RouteOpts {
  int scoring;        // MQ_SCORING_SOFTMAX / MQ_SCORING_SIGMOID
  int renorm;
  int groups;         // expert groups; <= 1: none
  int topk_group;     // groups kept when groups > 1
  const float* bias;  // score-correction bias [E] (device) or null
  float scale;        // routed scaling factor
};
inline bool route_opts_plain(const RouteOpts& o) {
  return o.scoring == MQ_SCORING_SOFTMAX && o.groups <= 1 && !o.bias && o.scale == 1.0f;
}
MQ_HIDDEN cudaError_t launch_route_ex(const float* logits, int T, int E, int k,
                                      const RouteOpts& o, float* topk_w, int32_t* topk_ids,
                                      cudaStream_t st);
// Router logits -> topk_w / topk_ids -> align as one kernel (the align
// kernel's 32 warps route first) when the routing work is small enough for
// one CTA: tokens x k argmax rounds over ceil(E / 32) registers per lane at
// most kFusedRouteWork (measured: Mixtral-shaped E=8, k=2 gains up to 5 us
// at T <= 64; E=128, k=8 at T=64 loses 2.4 us).  Otherwise the router kernel
// runs first.
constexpr int kFusedRouteWork = 512;
inline bool route_fused(int T, int k, int E) {
  return (int64_t)T * k * ((E + 31) / 32) <= kFusedRouteWork;
}
MQ_HIDDEN cudaError_t launch_route_align(const float* logits, int renorm, float* topk_w,
                                         int32_t* topk_ids, int T, int k, int E, int bm,
                                         int32_t* sorted, int32_t* block_expert,
                                         int32_t* offsets, int32_t* num_padded, unsigned* status,
                                         cudaStream_t st, int chunk, int32_t* chunk_expert,
                                         int32_t* chunk_start, int32_t* counts,
                                         int32_t* dep = nullptr);
// chunk > 0 also writes the chunk table of the expert GEMMs' token tiles
// (chunk_expert [cap / bm], chunk_start [E + 1]) and, with dep != null,
// zeroes each chunk's dependency counter of the fused layer kernel [cap / bm];
// counts != null the number of token-slots of each expert [E].
MQ_HIDDEN cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int bm,
                                   int32_t* sorted, int32_t* block_expert, int32_t* offsets,
                                   int32_t* num_padded, unsigned* status, cudaStream_t st,
                                   int chunk = 0, int32_t* chunk_expert = nullptr,
                                   int32_t* chunk_start = nullptr, int32_t* counts = nullptr,
                                   int32_t* dep = nullptr);

struct MoeArgs {
  const void* x;          // bf16, or f16 with MQ_FWD_ACT_F16
  unsigned flags;         // MQ_FWD_* options
  int T, H, I, E, k;
  int bits, group_size, has_zp;
  const void* w13;
  const void* w2;
  const void* s13;
  const void* s2;
  const uint8_t* z13;
  const uint8_t* z2;
  const float* topk_w;
  const int32_t* topk_ids;
  void* out;              // bf16, or f16 with MQ_FWD_ACT_F16
  unsigned* status;
  // workspace views
  int32_t* sorted;        // [cap]
  int32_t* block_expert;  // [cap / bm]
  int32_t* offsets;       // [E + 1]
  int32_t* num_padded;    // [1]
  int32_t* chunk_expert;  // [cap / bm]: expert of each token tile (chunk)
  int32_t* chunk_start;   // [E + 1]: first chunk of each expert; [E] = number of chunks
  int32_t* counts;        // [E]: token-slots of each expert
  int32_t* dep;           // [cap / bm]: fused layer, gate/up warps done per token tile
  __nv_bfloat16* act;     // [cap, I]
  float* y;               // [S, H]
  int bm;
  int64_t cap;
};

// Tensor-core path (tcgen05): tile plan and launchers.
struct TcPlan {
  int bn;      // token-slots per tile at most (MMA N <= bn); the align block is 16
  int splits;  // K splits of the down GEMM
  bool sync1;  // gate/up GEMM: warp-MMA consumers (few tokens per expert), not tcgen05
  bool sync2;  // down GEMM: the same
  bool layer;  // 8-bit, tcgen05: both GEMMs in one launch (moe_layer_tc)
  bool f16down;  // 8-bit, two launches: act to f16 in place, f16 down GEMM
};
MQ_HIDDEN TcPlan tc_plan(int T, int H, int I, int E, int k, int bits);
MQ_HIDDEN int tc_num_sms();
MQ_HIDDEN cudaError_t launch_gather_rows(const MoeArgs& a, void* xs, float* xinv, cudaStream_t st);
MQ_HIDDEN cudaError_t launch_gemm1_tc(const MoeArgs& a, const TcPlan& pl, const void* xs,
                                      const float* xinv, cudaStream_t st);
MQ_HIDDEN cudaError_t launch_act_to_f16(const MoeArgs& a, float* act_inv, cudaStream_t st);
MQ_HIDDEN cudaError_t launch_gemm2_tc(const MoeArgs& a, const TcPlan& pl, const float* act_inv,
                                      float* ypart, cudaStream_t st);
MQ_HIDDEN cudaError_t launch_combine_splits(const MoeArgs& a, const float* ypart, int splits,
                                            cudaStream_t st);
// Both expert GEMMs of an 8-bit layer in one launch (token tiles of 64 or 128
// rows): act and the down GEMM's partial sums as the two launches write them.
MQ_HIDDEN cudaError_t launch_layer_tc(const MoeArgs& a, const TcPlan& pl, const void* xs,
                                      const float* xinv, float* ypart, cudaStream_t st);
// Testing aid: extra gate/up completions the layer's down units wait for
// (their waits then run out); returns the previous value.
MQ_HIDDEN int set_layer_wait_extra(int extra);

// Warp-MMA ("decode") mode of the expert GEMMs: the formats it takes, and
// the K splits of its down GEMM.
MQ_HIDDEN bool dec_supported(int bits, int group_size, int H, int I);
MQ_HIDDEN int dec_splits(int T, int H, int I, int E, int k, int bits);

// Records `msg` as the calling thread's mq_last_error_message(); returns status.
MQ_HIDDEN int mq_set_error(int status, const char* msg);
