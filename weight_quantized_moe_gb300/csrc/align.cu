// Block alignment: stable counting sort of the token-slots by expert, each
// expert's segment padded to a multiple of block_m (the grouping fused_experts
// performs before its grouped GEMMs).
//
// One CTA of 32 warps.  Warp w owns the contiguous slot range
// [w * per_warp, (w + 1) * per_warp).
//   1. per-warp histograms hist[w][e] (shared-memory atomics);
//   2. per expert: count, pad, block-wide exclusive scan -> segment starts;
//      hist[w][e] becomes the first position of warp w's slots of expert e;
//   3. each warp walks its range again in slot order and places every slot at
//      hist[w][e] + (rank among equal experts in this 32-slot step), found
//      with __match_any_sync; the rank order is lane order, i.e. slot order.
// The result is therefore deterministic and identical to a stable sort.
//
// Optionally (chunk > 0) it also cuts each expert's padded segment into
// chunks of at most `chunk` slots, the token tiles of the expert GEMMs:
// chunk_start[e] = index of expert e's first chunk (chunk_start[E] = the
// number of chunks) and chunk_expert[c] = the expert of chunk c.  With
// counts != null it also writes each expert's number of token-slots.
//
// With PER > 0 it first routes the T tokens itself (router logits in, the
// router's code, one warp per token), writing topk_w and the ids it then
// aligns: at small batches one launch instead of two.
#include "common.cuh"
#include "route_core.cuh"

namespace {

constexpr int kWarps = 32;
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 8;  // 32-slot steps whose ids a warp loads before using them

template <int PER>
__global__ void __launch_bounds__(kThreads, 1)
    align_kernel(int32_t* __restrict__ ids, int S, int E, int bm, int32_t* __restrict__ sorted,
                 int32_t* __restrict__ block_expert, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ num_padded, int chunk, int32_t* __restrict__ chunk_expert,
                 int32_t* __restrict__ chunk_start, int32_t* __restrict__ counts,
                 int32_t* __restrict__ dep, const float* __restrict__ logits, int T, int k, int renorm,
                 float* __restrict__ topk_w, unsigned* status) {
  extern __shared__ int smem[];
  int* hist = smem;                   // [kWarps][E]
  int* warp_tot = smem + kWarps * E;  // [kWarps] scan scratch
  int* warp_tot2 = warp_tot + kWarps; // [kWarps] scan scratch (chunks)
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  for (int i = tid; i < kWarps * E; i += kThreads) hist[i] = 0;
  mq::pdl_wait();  // the ids (or logits) come from the previous kernel
  mq::pdl_trigger();
  if constexpr (PER > 0) {
    float* s_val = reinterpret_cast<float*>(warp_tot2 + kWarps) + warp * 32;
    int* s_idx = warp_tot2 + kWarps + kWarps * 32 + warp * 32;
    for (int t = warp; t < T; t += kWarps)
      mq::route_token<PER>(logits + (int64_t)t * E, E, k, renorm, s_val, s_idx,
                           topk_w + (int64_t)t * k, ids + (int64_t)t * k);
  }
  __syncthreads();  // (ids written by this block are visible to all of it)

  const int per_warp = (S + kWarps - 1) / kWarps;
  const int begin = warp * per_warp;
  const int end = min(S, begin + per_warp);
  bool bad = false;
  for (int base = begin; base < end; base += 32 * kBatch) {
    int ev[kBatch];  // all loads of the batch in flight before the first use
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = base + b * 32 + lane;
      ev[b] = s < end ? ids[s] : 0;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (base + b * 32 >= end) break;  // warp-uniform
      if (base + b * 32 + lane < end) {
        if (ev[b] >= 0 && ev[b] < E) atomicAdd(&hist[warp * E + ev[b]], 1);
        else bad = true;
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) mq::flag(status, MQ_DEV_BAD_EXPERT_ID);
  __syncthreads();

  // ---- per-expert totals and exclusive scan of the padded sizes ----------
  const int e = tid;  // E <= kThreads
  int count = 0;
  if (e < E)
    for (int w = 0; w < kWarps; ++w) count += hist[w * E + e];
  const int padded = (count + bm - 1) / bm * bm;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int start = incl - padded + (warp ? warp_tot[warp - 1] : 0);
  if (e < E) {
    offsets[e] = start;
    if (counts) counts[e] = count;
    int run = start;
    for (int w = 0; w < kWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    for (int p = start + count; p < start + padded; ++p) sorted[p] = S;
    for (int b = start / bm; b < (start + padded) / bm; ++b) block_expert[b] = e;
  }
  if (tid == 0) {
    const int total = warp_tot[kWarps - 1];
    offsets[E] = total;
    num_padded[0] = total;
  }
  if (chunk > 0) {
    // exclusive scan of the chunk counts, the same way as the padded sizes
    const int nch = e < E ? (padded + chunk - 1) / chunk : 0;
    int cincl = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, cincl, o);
      if (lane >= o) cincl += n;
    }
    if (lane == 31) warp_tot2[warp] = cincl;
    __syncthreads();
    if (warp == 0) {
      int t2 = warp_tot2[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, t2, o);
        if (lane >= o) t2 += n;
      }
      warp_tot2[lane] = t2;
    }
    __syncthreads();
    const int cstart = cincl - nch + (warp ? warp_tot2[warp - 1] : 0);
    if (e < E) {
      chunk_start[e] = cstart;
      for (int c = 0; c < nch; ++c) chunk_expert[cstart + c] = e;
      if (dep)
        for (int c = 0; c < nch; ++c) dep[cstart + c] = 0;
    }
    if (tid == 0) chunk_start[E] = warp_tot2[kWarps - 1];
  }
  __syncthreads();

  // ---- stable placement (32-slot steps in slot order) ----------------------
  for (int base = begin; base < end; base += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = base + b * 32 + lane;
      ev[b] = s < end ? ids[s] : -1;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (base + b * 32 >= end) break;  // warp-uniform
      const int s = base + b * 32 + lane;
      const int ex = (s < end && ev[b] >= 0 && ev[b] < E) ? ev[b] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, ex);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (ex >= 0) sorted[hist[warp * E + ex] + rank] = s;
      __syncwarp();
      if (ex >= 0 && rank == 0) hist[warp * E + ex] += __popc(peers);
      __syncwarp();
    }
  }
}

}  // namespace

namespace {

template <int PER>
cudaError_t launch_align_impl(int32_t* ids, int T, int k, int E, int bm, int32_t* sorted,
                              int32_t* block_expert, int32_t* offsets, int32_t* num_padded,
                              unsigned* status, cudaStream_t st, int chunk, int32_t* chunk_expert,
                              int32_t* chunk_start, int32_t* counts, int32_t* dep,
                              const float* logits, int renorm, float* topk_w) {
  size_t smem = (size_t)(kWarps * E + 2 * kWarps) * sizeof(int);
  if (PER > 0) smem += (size_t)kWarps * 32 * (sizeof(float) + sizeof(int));  // routing scratch
  auto kern = align_kernel<PER>;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
  }
  const cudaError_t err =
      launch_pdl(kern, dim3(1), dim3(kThreads), smem, st, ids, T * k, E, bm, sorted,
                 block_expert, offsets, num_padded, chunk, chunk_expert, chunk_start, counts,
                 dep, logits, T, k, renorm, topk_w, status);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int bm, int32_t* sorted,
                         int32_t* block_expert, int32_t* offsets, int32_t* num_padded,
                         unsigned* status, cudaStream_t st, int chunk, int32_t* chunk_expert,
                         int32_t* chunk_start, int32_t* counts, int32_t* dep) {
  return launch_align_impl<0>(const_cast<int32_t*>(ids), T, k, E, bm, sorted, block_expert,
                              offsets, num_padded, status, st, chunk, chunk_expert, chunk_start,
                              counts, dep, nullptr, 0, nullptr);
}

cudaError_t launch_route_align(const float* logits, int renorm, float* topk_w, int32_t* topk_ids,
                               int T, int k, int E, int bm, int32_t* sorted,
                               int32_t* block_expert, int32_t* offsets, int32_t* num_padded,
                               unsigned* status, cudaStream_t st, int chunk,
                               int32_t* chunk_expert, int32_t* chunk_start, int32_t* counts,
                               int32_t* dep) {
  if (!route_fused(T, k, E)) {
    const cudaError_t err = launch_route(logits, T, E, k, renorm, topk_w, topk_ids, st);
    if (err != cudaSuccess) return err;
    return launch_align(topk_ids, T, k, E, bm, sorted, block_expert, offsets, num_padded, status,
                        st, chunk, chunk_expert, chunk_start, counts, dep);
  }
  const int per = (E + 31) / 32;
#define MQ_RA(P)                                                                               \
  return launch_align_impl<P>(topk_ids, T, k, E, bm, sorted, block_expert, offsets, num_padded, \
                              status, st, chunk, chunk_expert, chunk_start, counts, dep, logits, \
                              renorm, topk_w);
  switch (per) {
    case 1: MQ_RA(1)
    case 2: MQ_RA(2)
    case 3: MQ_RA(3)
    case 4: MQ_RA(4)
    case 5: case 6: case 7: case 8: MQ_RA(8)
    case 9: case 10: case 11: case 12: case 13: case 14: case 15: case 16: MQ_RA(16)
    default: MQ_RA(32)
  }
#undef MQ_RA
}
