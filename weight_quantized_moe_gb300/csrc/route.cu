// Router kernel: one warp per token (see route_core.cuh).
#include "common.cuh"
#include "route_core.cuh"

namespace {

template <int PER>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int renorm, float* __restrict__ topk_w,
                                                    int32_t* __restrict__ topk_ids) {
  __shared__ float s_val[8][32];
  __shared__ int s_idx[8][32];
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + warp;
  mq::pdl_wait();  // the logits come from the previous kernel
  mq::pdl_trigger();
  if (t >= T) return;
  mq::route_token<PER>(logits + (int64_t)t * E, E, k, renorm, s_val[warp], s_idx[warp],
                       topk_w + (int64_t)t * k, topk_ids + (int64_t)t * k);
}

template <int PER>
__global__ void __launch_bounds__(256) route_ex_kernel(const float* __restrict__ logits, int T,
                                                       int E, int k, RouteOpts o,
                                                       float* __restrict__ topk_w,
                                                       int32_t* __restrict__ topk_ids) {
  __shared__ float s_val[8][32];
  __shared__ int s_idx[8][32];
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + warp;
  mq::pdl_wait();
  mq::pdl_trigger();
  if (t >= T) return;
  mq::route_token_ex<PER>(logits + (int64_t)t * E, E, k, o, s_val[warp], s_idx[warp],
                          topk_w + (int64_t)t * k, topk_ids + (int64_t)t * k);
}

}  // namespace

cudaError_t launch_route_ex(const float* logits, int T, int E, int k, const RouteOpts& o,
                            float* topk_w, int32_t* topk_ids, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((T + 7) / 8);
  const int per = (E + 31) / 32;
  cudaError_t err = cudaSuccess;
#define MQ_ROUTE(P)                                                                          \
  err = launch_pdl(route_ex_kernel<P>, dim3(blocks), dim3(256), 0, st, logits, T, E, k, o, \
                   topk_w, topk_ids);                                                        \
  break;
  switch (per) {
    case 1: MQ_ROUTE(1)
    case 2: MQ_ROUTE(2)
    case 3: case 4: MQ_ROUTE(4)
    case 5: case 6: case 7: case 8: MQ_ROUTE(8)
    case 9: case 10: case 11: case 12: case 13: case 14: case 15: case 16: MQ_ROUTE(16)
    default: MQ_ROUTE(32)
  }
#undef MQ_ROUTE
  return err != cudaSuccess ? err : cudaGetLastError();
}

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
