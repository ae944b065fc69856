// Router: softmax -> top-k -> optional renormalisation (the select_experts
// call of ExpertsInt8MoEMethod.apply with scoring_func="softmax").
//
// One warp per token.  Lane l holds logits l, l+32, l+64, ... in registers;
// k rounds of a warp-shuffle arg-max pick the experts (largest logit first,
// ties to the lower expert index).  Selection compares the float32 logits
// themselves, so the chosen ids do not depend on how exp() rounds.
#include "common.cuh"

#include <math_constants.h>

namespace {

struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

template <int PER>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int renorm, float* __restrict__ topk_w,
                                                    int32_t* __restrict__ topk_ids) {
  __shared__ float s_val[8][32];
  __shared__ int s_idx[8][32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  mq::pdl_wait();  // the logits come from the previous kernel
  mq::pdl_trigger();
  if (t >= T) return;
  const float* row = logits + (int64_t)t * E;
  float v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? row[e] : -CUDART_INF_F;
    if (x != x) x = -CUDART_INF_F;  // NaN never wins
    v[i] = x;
  }
  unsigned taken = 0;  // bit i: v[i] already selected (or out of range)
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;

  for (int j = 0; j < k; ++j) {
    float bv = -CUDART_INF_F;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (!(taken >> i & 1u) && better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      s_val[warp][j] = bv;
      s_idx[warp][j] = bi;
    }
  }
  __syncwarp();
  const float vmax = s_val[warp][0];
  float sum_all = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i < E) sum_all += expf(v[i] - vmax);
#pragma unroll
  for (int o = 16; o; o >>= 1) sum_all += __shfl_xor_sync(0xffffffffu, sum_all, o);
  const float ej = (lane < k) ? expf(s_val[warp][lane] - vmax) : 0.0f;
  float denom = sum_all;
  if (renorm) {
    float ssel = ej;
#pragma unroll
    for (int o = 16; o; o >>= 1) ssel += __shfl_xor_sync(0xffffffffu, ssel, o);
    denom = ssel;
  }
  if (lane < k) {
    topk_w[(int64_t)t * k + lane] = __fdiv_rn(ej, denom);
    topk_ids[(int64_t)t * k + lane] = s_idx[warp][lane];
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, float* topk_w,
                         int32_t* topk_ids, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((T + 7) / 8);
  const int per = (E + 31) / 32;
  cudaError_t err = cudaSuccess;
#define MQ_ROUTE(P)                                                                           \
  err = launch_pdl(route_kernel<P>, dim3(blocks), dim3(256), 0, st, logits, T, E, k, renorm, \
                   topk_w, topk_ids);                                                         \
  break;
  switch (per) {
    case 1: MQ_ROUTE(1)
    case 2: MQ_ROUTE(2)
    case 3: MQ_ROUTE(3)
    case 4: MQ_ROUTE(4)
    case 5: case 6: case 7: case 8: MQ_ROUTE(8)
    case 9: case 10: case 11: case 12: case 13: case 14: case 15: case 16: MQ_ROUTE(16)
    default: MQ_ROUTE(32)
  }
#undef MQ_ROUTE
  return err != cudaSuccess ? err : cudaGetLastError();
}
