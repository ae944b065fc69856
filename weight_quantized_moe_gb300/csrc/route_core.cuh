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

// The router with the other select_experts arguments (RouteOpts):
//  1. score s_e: softmax over the E logits, or sigmoid(logit_e);
//  2. selection key: the logit (no bias; both scores rise with it), or the
//     float32 s_e + bias_e;
//  3. groups > 1: experts [gE/G, (g+1)E/G) form group g, scored by its
//     largest key; the topk_group best groups (ties: lower group) stay and
//     the other groups' experts are out;
//  4. the k largest keys left (ties: lower index) fill slots 0..k-1;
//  5. weight j = s_{id_j}, divided by the chosen experts' sum when
//     renormalising, times the scaling factor.
// Host checks: groups <= 32 and divides E, topk_group in [1, groups], and k
// at most the experts of topk_group groups.  The whole warp calls it.
template <int PER>
__device__ __forceinline__ void route_token_ex(const float* __restrict__ row, int E, int k,
                                               const RouteOpts& o, float* s_val, int* s_idx,
                                               float* __restrict__ w_out,
                                               int32_t* __restrict__ id_out) {
  const int lane = threadIdx.x & 31;
  const bool sigm = o.scoring == MQ_SCORING_SIGMOID;
  float l[PER];
  float lmax = -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? row[e] : -CUDART_INF_F;
    if (x != x) x = -CUDART_INF_F;  // NaN never wins
    l[i] = x;
    lmax = fmaxf(lmax, x);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
  float sum_all = 0.0f;  // softmax denominator
  if (!sigm) {
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane + 32 * i < E) sum_all += expf(l[i] - lmax);
#pragma unroll
    for (int off = 16; off; off >>= 1) sum_all += __shfl_xor_sync(0xffffffffu, sum_all, off);
  }
  float key[PER];
  unsigned taken = 0;  // bit i: expert lane + 32 i chosen, out of range or in a dropped group
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    if (e >= E) {
      taken |= 1u << i;
      key[i] = -CUDART_INF_F;
      continue;
    }
    float c = l[i];
    if (o.bias) {
      const float sc = sigm ? __fdiv_rn(1.0f, 1.0f + expf(-l[i])) : __fdiv_rn(expf(l[i] - lmax), sum_all);
      c = __fadd_rn(sc, o.bias[e]);
      if (c != c) c = -CUDART_INF_F;
    }
    key[i] = c;
  }
  if (o.groups > 1) {
    const int gsz = E / o.groups;
    float gscore = -CUDART_INF_F;  // lane g: score of group g
    for (int g = 0; g < o.groups; ++g) {
      float m = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        if (e < E && e / gsz == g) m = fmaxf(m, key[i]);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == g) gscore = m;
    }
    unsigned kept = 0;
    for (int r = 0; r < o.topk_group; ++r) {
      const bool cand = lane < o.groups && !(kept >> lane & 1u);
      float bv = cand ? gscore : -CUDART_INF_F;
      int bi = cand ? lane : 0x7fffffff;
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (route_better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi < 32) kept |= 1u << bi;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(kept >> (e / gsz) & 1u)) taken |= 1u << i;
    }
  }
  for (int j = 0; j < k; ++j) {
    float bv = -CUDART_INF_F;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (!(taken >> i & 1u) && route_better(key[i], e, bv, bi)) {
        bv = key[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (route_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi < E && (bi & 31) == lane) {  // the owner records the weight's numerator
      taken |= 1u << (bi >> 5);
      float lv = -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (i == (bi >> 5)) lv = l[i];
      s_val[j] = sigm ? __fdiv_rn(1.0f, 1.0f + expf(-lv)) : expf(lv - lmax);
      s_idx[j] = bi;
    } else if (bi >= E && lane == 0) {  // nothing left (excluded by the host checks)
      s_val[j] = 0.0f;
      s_idx[j] = 0;
    }
  }
  __syncwarp();
  const float num = (lane < k) ? s_val[lane] : 0.0f;
  float denom = sigm ? 1.0f : sum_all;
  if (o.renorm) {
    float ssel = num;
#pragma unroll
    for (int off = 16; off; off >>= 1) ssel += __shfl_xor_sync(0xffffffffu, ssel, off);
    denom = ssel;
  }
  if (lane < k) {
    w_out[lane] = __fmul_rn(__fdiv_rn(num, denom), o.scale);
    id_out[lane] = s_idx[lane];
  }
  __syncwarp();
}

}  // namespace mq
