// Weight quantisers (run once, at load time).
//
// int8: experts_int8 page, quantize_in_place_and_get_scales -- one float32
//       scale per output row, scale = max|w| / 127, q = clamp(rint(w / s)).
// uint4: the moe_wna16 page's packed storage (MoeWNA16Method.create_weights),
//       asymmetric min-max per group along K.
//
// Both take every rounding decision in float32 with IEEE division and
// round-half-even, and are built without fast-math / flush-to-zero, so the
// codes are reproducible bit for bit on any IEEE float32 implementation.
#include "common.cuh"

namespace {

using mq::bf16_hi;
using mq::bf16_lo;

__device__ __forceinline__ int code_int8(float w, float s) {
  if (!(s > 0.0f)) return 0;
  float r = rintf(__fdiv_rn(w, s));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return (int)r;
}

__device__ __forceinline__ uint32_t pack4_int8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
         ((uint32_t)(d & 0xff) << 24);
}

// One warp per row; 8 bf16 per 16-byte load.
__global__ void __launch_bounds__(256) quant_int8_kernel(const uint4* __restrict__ w, int64_t rows,
                                                         int nvec, int8_t* __restrict__ q,
                                                         float* __restrict__ scale) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const unsigned lane = threadIdx.x & 31;
  const uint4* wr = w + row * nvec;
  float m = 0.0f;
  for (int i = lane; i < nvec; i += 32) {
    const uint4 v = __ldg(wr + i);
    m = fmaxf(m, fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))));
    m = fmaxf(m, fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
    m = fmaxf(m, fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))));
    m = fmaxf(m, fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w))));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s = __fdiv_rn(m, 127.0f);
  if (lane == 0) scale[row] = s;
  uint2* qr = reinterpret_cast<uint2*>(q + row * (int64_t)nvec * 8);
  for (int i = lane; i < nvec; i += 32) {
    const uint4 v = __ldg(wr + i);
    uint2 o;
    o.x = pack4_int8(code_int8(bf16_lo(v.x), s), code_int8(bf16_hi(v.x), s),
                     code_int8(bf16_lo(v.y), s), code_int8(bf16_hi(v.y), s));
    o.y = pack4_int8(code_int8(bf16_lo(v.z), s), code_int8(bf16_hi(v.z), s),
                     code_int8(bf16_lo(v.w), s), code_int8(bf16_hi(v.w), s));
    qr[i] = o;
  }
}

// One warp per (pair of rows, group).  Each lane holds PER = gs/32
// consecutive values of both rows.
template <int PER>
__global__ void __launch_bounds__(256) quant_uint4_kernel(const __nv_bfloat16* __restrict__ w,
                                                          int64_t row_pairs, int cols, int groups,
                                                          uint8_t* __restrict__ qw,
                                                          __half* __restrict__ sc,
                                                          uint8_t* __restrict__ qz) {
  const int64_t item = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (item >= row_pairs * groups) return;
  const unsigned lane = threadIdx.x & 31;
  const int64_t pair = item / groups;
  const int g = (int)(item % groups);
  const int gs = PER * 32;
  int zrow[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int64_t row = pair * 2 + rr;
    const __nv_bfloat16* src = w + row * cols + (int64_t)g * gs + lane * PER;
    float v[PER];
    float lo = 0.0f, hi = 0.0f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      v[i] = __bfloat162float(src[i]);
      lo = fminf(lo, v[i]);
      hi = fmaxf(hi, v[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const __half s16 = __float2half_rn(__fdiv_rn(hi - lo, 15.0f));
    const float s = __half2float(s16);
    float z = 0.0f;
    int qv[PER];
    if (s > 0.0f) {
      z = fminf(fmaxf(rintf(__fdiv_rn(-lo, s)), 0.0f), 15.0f);
#pragma unroll
      for (int i = 0; i < PER; ++i)
        qv[i] = (int)fminf(fmaxf(rintf(__fdiv_rn(v[i], s)) + z, 0.0f), 15.0f);
    } else {
#pragma unroll
      for (int i = 0; i < PER; ++i) qv[i] = 0;
    }
    zrow[rr] = (int)z;
    if (lane == 0) sc[row * groups + g] = s16;
    uint8_t* dst = qw + row * (cols / 2) + ((int64_t)g * gs + lane * PER) / 2;
    if (PER >= 2) {
#pragma unroll
      for (int i = 0; i + 1 < PER; i += 2) dst[i / 2] = (uint8_t)(qv[i] | (qv[i + 1] << 4));
    } else {
      const int other = __shfl_down_sync(0xffffffffu, qv[0], 1);
      if ((lane & 1) == 0) dst[0] = (uint8_t)(qv[0] | (other << 4));
    }
  }
  if (lane == 0) qz[pair * groups + g] = (uint8_t)(zrow[0] | (zrow[1] << 4));
}

}  // namespace

cudaError_t launch_quant_int8(const void* w, int64_t rows, int64_t cols, int8_t* q, float* scale,
                              cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  quant_int8_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(w), rows,
                                                      (int)(cols / 8), q, scale);
  return cudaGetLastError();
}

cudaError_t launch_quant_uint4(const void* w, int64_t rows, int64_t cols, int gs, uint8_t* qw,
                               uint16_t* sc, uint8_t* qz, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int groups = (int)(cols / gs);
  const int64_t items = rows / 2 * groups;
  const unsigned blocks = (unsigned)((items + 7) / 8);
  const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(w);
  __half* s = reinterpret_cast<__half*>(sc);
  switch (gs) {
    case 32: quant_uint4_kernel<1><<<blocks, 256, 0, st>>>(wb, rows / 2, (int)cols, groups, qw, s, qz); break;
    case 64: quant_uint4_kernel<2><<<blocks, 256, 0, st>>>(wb, rows / 2, (int)cols, groups, qw, s, qz); break;
    case 128: quant_uint4_kernel<4><<<blocks, 256, 0, st>>>(wb, rows / 2, (int)cols, groups, qw, s, qz); break;
    case 256: quant_uint4_kernel<8><<<blocks, 256, 0, st>>>(wb, rows / 2, (int)cols, groups, qw, s, qz); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
