// Router core: one warp routes one token -- softmax over the E logits, top-k
// (largest logit first, ties to the lower expert index), optional
// renormalisation over the chosen k (the select_experts call of
// ExpertsInt8MoEMethod.apply with scoring_func="softmax").
//
// Lane l holds logits l, l+32, l+64, ... in registers; k rounds of a
// warp-shuffle arg-max pick the experts.  Selection compares the float32
// logits themselves, so the chosen ids do not depend on how exp() rounds.
// Used by the router kernel and by the align kernel's fused routing.
#pragma once

#include "common.cuh"

#include <math_constants.h>

namespace mq {

__device__ __forceinline__ bool route_better(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Token row -> w_out[0..k), id_out[0..k).  s_val / s_idx: this warp's 32-entry
// shared scratch.  The whole warp calls it.
template <int PER>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int renorm,
                                            float* s_val, int* s_idx, float* __restrict__ w_out,
                                            int32_t* __restrict__ id_out) {
  const int lane = threadIdx.x & 31;
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
      if (!(taken >> i & 1u) && route_better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (route_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      s_val[j] = bv;
      s_idx[j] = bi;
    }
  }
  __syncwarp();
  const float vmax = s_val[0];
  float sum_all = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i < E) sum_all += expf(v[i] - vmax);
#pragma unroll
  for (int o = 16; o; o >>= 1) sum_all += __shfl_xor_sync(0xffffffffu, sum_all, o);
  const float ej = (lane < k) ? expf(s_val[lane] - vmax) : 0.0f;
  float denom = sum_all;
  if (renorm) {
    float ssel = ej;
#pragma unroll
    for (int o = 16; o; o >>= 1) ssel += __shfl_xor_sync(0xffffffffu, ssel, o);
    denom = ssel;
  }
  if (lane < k) {
    w_out[lane] = __fdiv_rn(ej, denom);
    id_out[lane] = s_idx[lane];
  }
  __syncwarp();
}

}  // namespace mq
