// Plain CUDA-core expert GEMMs: the straightforward form of fused_experts
// (gate/up GEMM with dequant, SiLU-and-mul, down GEMM with dequant), kept
// for shapes the tensor-core kernels do not tile and as a cross-check.
//
// Both GEMMs walk the aligned blocks: block b holds kBM sorted token-slots
// that all go to expert block_expert[b].  Weights are dequantised to float32
// on the way into shared memory; accumulation is float32.
#include "common.cuh"

namespace {

constexpr int kBM = 16;   // token-slots per block (the align block size)
constexpr int kKC = 32;   // K chunk staged in shared memory
constexpr int kThreads = 256;

template <int BITS>
__device__ __forceinline__ float load_w(const void* w, const void* scales, const uint8_t* zeros,
                                        int has_zp, int gs, int64_t row, int rows_total,
                                        int K, int kk) {
  if (BITS == 8) {
    return (float)reinterpret_cast<const int8_t*>(w)[row * K + kk];
  } else {
    const uint8_t byte = reinterpret_cast<const uint8_t*>(w)[row * (K / 2) + kk / 2];
    const int q = (kk & 1) ? (byte >> 4) : (byte & 15);
    const int G = K / gs;
    int z = 8;
    if (has_zp) {
      const uint8_t zb = zeros[(row >> 1) * G + kk / gs];
      z = (row & 1) ? (zb >> 4) : (zb & 15);
    }
    const float s = __half2float(reinterpret_cast<const __half*>(scales)[row * G + kk / gs]);
    return (float)(q - z) * s;
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) gemm1_simple(MoeArgs a) {
  const int b = blockIdx.y;
  if (b * kBM >= *a.num_padded) return;
  const int e = a.block_expert[b];
  const int n0 = blockIdx.x * 64;
  const int S = a.T * a.k;
  const int H = a.H, I = a.I;
  __shared__ float xs[kBM][kKC + 1];
  __shared__ float ws[128][kKC + 1];
  __shared__ float ys[128][kBM + 1];
  __shared__ int tok[kBM];
  const int tid = threadIdx.x;
  if (tid < kBM) {
    const int s = a.sorted[b * kBM + tid];
    tok[tid] = (s < S) ? s / a.k : -1;
  }
  __syncthreads();
  const int n = tid & 127;
  const int tg = tid >> 7;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  const int64_t row_base = (int64_t)e * 2 * I;
  for (int k0 = 0; k0 < H; k0 += kKC) {
    for (int i = tid; i < kBM * kKC; i += kThreads) {
      const int r = i / kKC, c = i % kKC;
      xs[r][c] = tok[r] >= 0 ? __bfloat162float(a.x[(int64_t)tok[r] * H + k0 + c]) : 0.0f;
    }
    for (int i = tid; i < 128 * kKC; i += kThreads) {
      const int r = i / kKC, c = i % kKC;
      const int grow = r < 64 ? n0 + r : I + n0 + (r - 64);
      ws[r][c] = load_w<BITS>(a.w13, a.s13, a.z13, a.has_zp, a.group_size, row_base + grow,
                              2 * I, H, k0 + c);
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kKC; ++c) {
      const float wv = ws[n][c];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wv, xs[tg * 8 + i][c], acc[i]);
    }
    __syncthreads();
  }
  const int grow = n < 64 ? n0 + n : I + n0 + (n - 64);
  const float sc = (BITS == 8) ? reinterpret_cast<const float*>(a.s13)[row_base + grow] : 1.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ys[n][tg * 8 + i] = acc[i] * sc;
  __syncthreads();
  for (int i = tid; i < 64 * kBM; i += kThreads) {
    const int col = i % 64, r = i / 64;
    const float g = ys[col][r], u = ys[64 + col][r];
    a.act[(int64_t)(b * kBM + r) * I + n0 + col] = __float2bfloat16_rn(mq::silu_mul(g, u));
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) gemm2_simple(MoeArgs a) {
  const int b = blockIdx.y;
  if (b * kBM >= *a.num_padded) return;
  const int e = a.block_expert[b];
  const int h0 = blockIdx.x * 128;
  const int S = a.T * a.k;
  const int H = a.H, I = a.I;
  __shared__ float xs[kBM][kKC + 1];
  __shared__ float ws[128][kKC + 1];
  __shared__ int slot[kBM];
  const int tid = threadIdx.x;
  if (tid < kBM) slot[tid] = a.sorted[b * kBM + tid];
  __syncthreads();
  const int n = tid & 127;
  const int tg = tid >> 7;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  const int64_t row_base = (int64_t)e * H;
  for (int k0 = 0; k0 < I; k0 += kKC) {
    for (int i = tid; i < kBM * kKC; i += kThreads) {
      const int r = i / kKC, c = i % kKC;
      xs[r][c] = __bfloat162float(a.act[(int64_t)(b * kBM + r) * I + k0 + c]);
    }
    for (int i = tid; i < 128 * kKC; i += kThreads) {
      const int r = i / kKC, c = i % kKC;
      ws[r][c] = load_w<BITS>(a.w2, a.s2, a.z2, a.has_zp, a.group_size, row_base + h0 + r, H, I,
                              k0 + c);
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < kKC; ++c) {
      const float wv = ws[n][c];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wv, xs[tg * 8 + i][c], acc[i]);
    }
    __syncthreads();
  }
  const float sc = (BITS == 8) ? reinterpret_cast<const float*>(a.s2)[row_base + h0 + n] : 1.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int s = slot[tg * 8 + i];
    if (s < S) a.y[(int64_t)s * H + h0 + n] = acc[i] * sc * a.topk_w[s];
  }
}

// out[t, :] = sum over valid slots j of y[t*k + j, :], rounded once to bf16.
__global__ void __launch_bounds__(256) combine_kernel(MoeArgs a) {
  const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 4 columns per thread
  const int H4 = a.H / 4;
  if (i4 >= (int64_t)a.T * H4) return;
  const int t = (int)(i4 / H4);
  const int c = (int)(i4 % H4) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.k; ++j) {
    const int s = t * a.k + j;
    const int e = a.topk_ids[s];
    if (e < 0 || e >= a.E) continue;
    const float4 v = *reinterpret_cast<const float4*>(a.y + (int64_t)s * a.H + c);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 o;
  o.x = *reinterpret_cast<uint32_t*>(&lo);
  o.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a.out + (int64_t)t * a.H + c) = o;
}

}  // namespace

int simple_block_m() { return kBM; }

cudaError_t launch_gemm1_simple(const MoeArgs& a, cudaStream_t st) {
  const unsigned blocks = (unsigned)(a.cap / kBM);
  if (blocks == 0) return cudaSuccess;
  dim3 g(a.I / 64, blocks);
  if (a.bits == 8) gemm1_simple<8><<<g, kThreads, 0, st>>>(a);
  else gemm1_simple<4><<<g, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemm2_simple(const MoeArgs& a, cudaStream_t st) {
  const unsigned blocks = (unsigned)(a.cap / kBM);
  if (blocks == 0) return cudaSuccess;
  dim3 g(a.H / 128, blocks);
  if (a.bits == 8) gemm2_simple<8><<<g, kThreads, 0, st>>>(a);
  else gemm2_simple<4><<<g, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const MoeArgs& a, cudaStream_t st) {
  const int64_t n = (int64_t)a.T * (a.H / 4);
  if (n == 0) return cudaSuccess;
  combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}
