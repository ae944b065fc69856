// Thin inline-PTX wrappers for the Blackwell (sm_100 family) features the
// tensor-core kernels use: mbarriers, TMA tile loads, TMEM allocation,
// tcgen05.mma / commit / ld / st and the tcgen05 fences.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mq {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------------ TMA --
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

// L2 cache policy for data read once per pass (streamed weights): its lines
// are the first to go, so that what is reused (activations, partial sums,
// the kernels' own code) stays in L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_2d / tma_load_4d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int x, int y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int c0, int c1, int c2, int c3, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "l"(pol)
      : "memory");
}

// Bulk copy of `bytes` contiguous bytes (16-byte aligned, a multiple of 16)
// from global to shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16, one CTA.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One MMA step: 16 MMAs of K = 16 into the same accumulator, A from 16
// consecutive 8-column slices of tensor memory, B slice kk at descriptor
// b_desc + Okk (a start-address offset in 16-byte units).  The first MMA
// accumulates only if `accumulate` is nonzero, the others always.  All 16 are
// issued from one asm statement, with no instruction of the compiler's
// between them.
template <uint32_t O1, uint32_t O2, uint32_t O3, uint32_t O4, uint32_t O5, uint32_t O6,
          uint32_t O7, uint32_t O8, uint32_t O9, uint32_t O10, uint32_t O11, uint32_t O12,
          uint32_t O13, uint32_t O14, uint32_t O15>
__device__ __forceinline__ void mma_ts_x16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pa;\n\t.reg .b64 bd;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 pa, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n\t"
      "setp.eq.b32 pa, %3, %3;\n\t"
      "add.s32 ta, %1, 8;\n\tadd.s64 bd, %2, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 16;\n\tadd.s64 bd, %2, %6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 24;\n\tadd.s64 bd, %2, %7;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 32;\n\tadd.s64 bd, %2, %8;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 40;\n\tadd.s64 bd, %2, %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 48;\n\tadd.s64 bd, %2, %10;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 56;\n\tadd.s64 bd, %2, %11;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 64;\n\tadd.s64 bd, %2, %12;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 72;\n\tadd.s64 bd, %2, %13;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 80;\n\tadd.s64 bd, %2, %14;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 88;\n\tadd.s64 bd, %2, %15;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 96;\n\tadd.s64 bd, %2, %16;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 104;\n\tadd.s64 bd, %2, %17;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 112;\n\tadd.s64 bd, %2, %18;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "add.s32 ta, %1, 120;\n\tadd.s64 bd, %2, %19;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, pa;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate),
      "n"(O1), "n"(O2), "n"(O3), "n"(O4), "n"(O5), "n"(O6), "n"(O7), "n"(O8), "n"(O9), "n"(O10), "n"(O11), "n"(O12), "n"(O13), "n"(O14), "n"(O15)
      : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns; thread t owns lane (taddr.lane + t).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// tcgen05.ld of N consecutive 32-bit columns (one per register) for the
// warp's 32 lanes, together with its tcgen05.wait::ld.  The load fills its
// destination registers asynchronously while the compiler treats an asm's
// outputs as ready at once, so any instruction the compiler placed between a
// separate load and wait (a use, or a register copy) could read them early.
// One asm statement leaves no such gap.  Global loads issued before the call
// stay in flight across it.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols_sync(uint32_t taddr, uint32_t (&v)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tmem_ld32_sync(taddr, v);
  else tmem_ld16_sync(taddr, v);
}

// ------------------------------------------------------- descriptors --
// Shared-memory matrix descriptor (tcgen05 format): K-major operand stored
// with the 128-byte swizzle, rows of 128 bytes, 8-row core groups 1024 bytes
// apart.  `addr` must lie in a 1024-byte aligned swizzle atom.
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);         // start address
  d |= (uint64_t)(16u >> 4) << 16;                // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                         // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                         // swizzle: 128 B
  return d;
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> f32, A and B K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// Instruction descriptor, kind::f16: f16 x f16 -> f32, A and B K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | ((uint32_t)(N >> 3) << 17)   // N / 8   (A, B formats 0 = f16)
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

}  // namespace ptx
}  // namespace mq
