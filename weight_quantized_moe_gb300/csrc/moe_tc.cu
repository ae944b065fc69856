// Tensor-core expert GEMMs for sm_103a (tcgen05 + TMA + TMEM).
//
// fused_experts' two grouped GEMMs (gate/up with SiLU-and-mul, then down
// with the router-weighted scatter), restated for Blackwell:
//
//   D[128 weight rows x BN token-slots] = W[rows, K] . X[slots, K]^T
//
// * The weight tile is the MMA's A operand.  TMA stages the int8 codes in
//   shared memory, one 16 KB box (128 rows x 128 bytes) per K step; for the
//   gate/up GEMM a 4-D tensor map fetches the 64 gate rows and the matching
//   64 up rows in that one box.  Converter warpgroups turn the codes into
//   f16 (bf16 in the 8-bit down GEMM; exact, every int8 value is both) and
//   write them straight into tensor memory with tcgen05.st, so shared
//   memory never holds 16-bit weights.  The per-channel scale is applied
//   once per output in the epilogue (sum_k x*(q*s) = s * sum_k x*q).
// * The activations (token rows gathered per expert block) are the B
//   operand: TMA tiles with the 128-byte swizzle in a second, short ring,
//   read by tcgen05.mma from shared memory.
// * Accumulators live in tensor memory, double-buffered across work units.
// * One persistent CTA per SM walks the work units (expert block, weight
//   tile, K split).  Warp roles: 0 weight producer (TMA), 1 MMA issuer,
//   2 activation producer (TMA, and the uint4 scale staging), then two
//   converter groups taking alternate MMA steps (3-10; uint4: 3-18, two
//   warps per tensor-memory lane quarter), then 4 epilogue warps, then the
//   second MMA issuer of 16- and 32-token tiles.  The one-launch layer
//   (moe_layer_tc) runs the gate/up and the down GEMM in one kernel.
// * Every mbarrier wait is bounded: after kWaitNs the CTA flags
//   MQ_DEV_WAIT_TIMEOUT, stops issuing work, drains its own copies and MMAs
//   (with a bound again), frees its tensor memory and exits.
#include "common.cuh"
#include "dequant.cuh"
#include "sm100_ptx.cuh"

#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <type_traits>

namespace {

using namespace mq::ptx;
using namespace mq::dq;

constexpr int kBK = 128;                  // K elements per weight stage (one 16 KB TMA box)
constexpr int kG = 2;                     // weight stages per MMA step
constexpr int kTileM = 128;               // weight rows per tile (MMA M)
constexpr int kAColsPerK = kBK / 2;       // TMEM columns per weight stage (16-bit pairs)
constexpr int kAColsPerStep = kG * kAColsPerK;
constexpr int kABytes = kTileM * kBK;     // int8 A tile per weight stage (16 KB)
constexpr int kConvGroups = 2;            // converter warpgroups (alternate MMA steps)
constexpr int kConvWarp0 = 3;             // warps 0: A producer, 1: MMA, 2: B producer
constexpr int kEpiWarp0 = kConvWarp0 + 4 * kConvGroups;  // first epilogue warp
constexpr int kIssuer2Warp = kEpiWarp0 + 4;  // second MMA issuer (16- and 32-token tiles)
constexpr unsigned long long kWaitNs = 1000000000ull;
constexpr int kRasterGroup = 8;           // weight tiles per raster group
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBudget = 212 * 1024;   // A ring + B ring
constexpr int kMaxSteps = 4;              // MMA-step ring depth (max)
constexpr int kMaxVirt = 6;               // barrier slots of the MMA-step ring (max)
constexpr int kUnitList = 512;            // work units per CTA decoded once into shared memory
// uint4: a work unit's group scales ([128 tile rows][G] f16) and zero points
// ([64 row pairs][G] bytes) are staged in shared memory, double-buffered
// across units, when they fit a buffer of kStageBytes (G <= 25)
constexpr int kStageBytes = 8192;
inline bool stage_fits(int G) { return 128 * G * 2 + 64 * G <= kStageBytes; }

// Pipeline shape per token-tile width BN.
//
// * The int8 weight ring (16 KB entries) is as deep as shared memory allows:
//   HBM needs about 200 KB in flight per SM.
// * Synchronisation with the MMA issuer happens per MMA step of kG weight
//   stages (16 MMAs): the wait and commit around a step cost several MMAs'
//   worth of issue time, so a step batches 16 of them.
// * Tensor memory holds two accumulator buffers (one, below, for uint4
//   64-token tiles) and kSteps converted-A
//   stages of kG * 64 columns; the activation ring has kBSlots slots (as
//   many, or six for 16-token tiles), and one MMA commit per step frees a
//   stage and a slot.
// * One tcgen05.mma takes about 80 cycles to issue whatever N is, and the
//   issuing thread's wait and commit around each 16-MMA step add about a
//   third to that; two threads issuing at once reach twice the rate.  For
//   16- and 32-token tiles a second issuer thread takes every other step;
//   each issuer accumulates its steps into its own half of the accumulator
//   (kNI = 2 halves, added in a fixed order by the epilogue).  Step st uses
//   tensor-memory stage st % 3: a converter group converts its next step
//   while its issuer's MMAs still read the previous one.  With one stage
//   per issuer (st % 2) the two alternated, and the Mixtral-shaped gate/up
//   launch at T=64 took 184 us against 163 us with three; the 8-bit down
//   GEMM kept one issuer then (its bf16 conversion needed a third stage),
//   and with three stages two issuers serve it too (T=64: 106 -> 99 us).
// * uint4 64-token tiles take two issuers as well.  Two accumulator buffers
//   of two halves would leave room for two stages only, so they keep one
//   buffer and three stages: the MMAs of a unit wait for the epilogue of the
//   previous one, which costs less than a lone issuer's wait and commit per
//   step (W4A16 E=64 at T=64: gate/up 100.8 -> 90.2 us, down 57.5 -> 53.3
//   us).  8-bit 64-token tiles keep one issuer and two buffers: their down
//   GEMM in the fine-grained layer (K = 768, three steps per unit) went from
//   22.5 to 28.5 us with one buffer.
template <int BN, int NI, int SB = 0>
struct TileCfg {
  static constexpr int kNI = NI;                // MMA issuer threads
  // accumulator buffers of kNI halves: two (the epilogue of a unit overlaps
  // the next unit's MMAs), or one where two would leave two issuers fewer
  // than three stages (64-row tiles)
  static constexpr int kAccBufs =
      (kNI == 2 && 2 * kNI * BN + 3 * kAColsPerStep > (int)kTmemCols) ? 1 : 2;
  static constexpr int kACol0 = kAccBufs * kNI * BN;
  static constexpr int kStepFit = ((int)kTmemCols - kACol0) / kAColsPerStep;
  // one issuer: as many stages as fit (at most kMaxSteps); two issuers:
  // three where they fit, so that a converter group's next step can be
  // converted while its issuer's MMAs of the previous one still read their
  // stage (with two stages, one per issuer, conversion and MMAs alternated)
  static constexpr int kSteps =
      kNI == 2 ? (kStepFit >= 3 ? 3 : 2) : (kStepFit > kMaxSteps ? kMaxSteps : kStepFit);
  // barrier slots of the step ring: step st uses stage st % kSteps and the
  // barriers of slot st % kVirt.  Two issuers with three stages: six slots,
  // so that each slot serves one issuer and one converter group only (st % 6
  // fixes st % 2 and st % 3) and every parity wait is exact
  static constexpr int kVirt = (kNI == 2 && kSteps == 3) ? 6 : kSteps;
  // activation ring slots (step st in slot st % kBSlots): as many as the
  // stages, or, for 16-token tiles with six barrier slots, six (8 KB each),
  // so that a step's activation tile is requested six steps ahead and its
  // L2 latency stays off the converters' path
  static constexpr int kBSlots = (kVirt == 6 && BN == 16) ? 6 : kSteps;
  // converter warps per group: one per tensor-memory lane quarter, or for
  // uint4 (SB > 0) two, each converting half of a stage's K: uint4 -> f16
  // with the group scale costs about twice the instructions of int8 per
  // weight, and one warp per quarter left the converters the bottleneck
  static constexpr int kWPG = SB > 0 ? 8 : 4;
  static constexpr int kConvW0 = kConvWarp0;
  static constexpr int kEpiW0 = kConvW0 + kWPG * kConvGroups;  // first epilogue warp
  static constexpr int kIss2W = kEpiW0 + 4;                    // second MMA issuer
  static constexpr int kThreads = (kEpiW0 + 4 + (kNI - 1)) * 32;
  static constexpr int kBBytesK = BN * kBK * 2;     // activations per weight stage
  static constexpr int kBBytes = kG * kBBytesK;     // activations per MMA step
  static constexpr int kAFit = (kSmemBudget - SB - kBSlots * kBBytes) / kABytes;
  static constexpr int kAStagesSmem = kAFit > 12 ? 12 : kAFit;
  static_assert(kACol0 + kSteps * kAColsPerStep <= (int)kTmemCols, "tensor memory budget");
  static_assert(kSteps >= 2, "MMA-step depth");
  static_assert(kNI == 1 || kStepFit >= 2, "two issuers: at least one stage each");
  static_assert(kVirt <= kMaxVirt, "barrier slots");
  static_assert(kBSlots == kSteps || kBSlots == kVirt, "activation slots");
  static_assert(kAStagesSmem >= 3, "weight ring depth");
};

// Warp-MMA consumer mode (few token-slots per expert): no tensor memory and
// no MMA issuer; each converter warp multiplies its converted weight rows
// straight from registers with mma.sync (m16n8k16, f32 accumulate).  The
// activation ring is kSteps MMA steps deep -- an even number, so that every
// slot serves one converter group only (step st uses slot st % kSteps and
// belongs to group st % 2): each converter warp has then itself seen the
// slot's previous fill land, which makes its parity wait exact.  The two
// groups' partial sums reach the epilogue through kPBufs shared-memory
// buffers of [group][column][row] floats (row stride kPStride keeps the
// converters' scattered stores and the epilogue's row reads free of bank
// conflicts).
template <int BN, int SB = 0>
struct SyncCfg {
  static constexpr int kNI = 1;
  static constexpr int kAccBufs = 2;
  static constexpr int kWPG = 4;
  static constexpr int kConvW0 = kConvWarp0;
  static constexpr int kEpiW0 = kEpiWarp0;
  static constexpr int kIss2W = kIssuer2Warp;
  static constexpr int kThreads = (kEpiWarp0 + 4) * 32;
  static constexpr int kSteps = 4;
  static constexpr int kVirt = kSteps;
  static constexpr int kBSlots = kSteps;
  static_assert(kSteps % 2 == 0, "one converter group per activation slot");
  static constexpr int kACol0 = 0;
  static constexpr int kBBytesK = BN * kBK * 2;
  static constexpr int kBBytes = kG * kBBytesK;
  static constexpr int kPStride = kTileM + 4;
  static constexpr int kPBytes = kConvGroups * BN * kPStride * 4;
  static constexpr int kPBufs = BN <= 16 ? 2 : 1;
  static constexpr int kAFit =
      (kSmemBudget + 4096 - SB - kSteps * kBBytes - kPBufs * kPBytes) / kABytes;
  static constexpr int kAStagesSmem = (kAFit > 12 ? 12 : kAFit) & ~1;
  static_assert(kAStagesSmem >= 4, "weight ring depth");
};

template <int MODE, int BITS, int BN, bool SYNC>
struct CfgSel {
  using type = TileCfg<BN, (BN <= 32 || (BN == 64 && BITS == 4)) ? 2 : 1,
                       BITS == 4 ? 2 * kStageBytes : 0>;
};
template <int MODE, int BITS, int BN>
struct CfgSel<MODE, BITS, BN, true> {
  using type = SyncCfg<BN, BITS == 4 ? 2 * kStageBytes : 0>;
};
template <int MODE, int BITS, int BN, bool SYNC = false>
using CfgOf = typename CfgSel<MODE, BITS, BN, SYNC>::type;

// Shared memory of the warp-MMA mode's partial-sum buffers (0 otherwise).
template <bool SYNC, int BN>
constexpr int partial_bytes() {
  if constexpr (SYNC) return SyncCfg<BN>::kPBufs * SyncCfg<BN>::kPBytes;
  else return 0;
}

// Shared memory of the uint4 scale staging buffers.
template <int BITS>
constexpr int stage_bytes() {
  return BITS == 4 ? 2 * kStageBytes : 0;
}

struct TcParams {
  int H, I, E, k, S;
  int ksteps;        // weight stages per row: ceil(K / stage K)
  int MT;            // weight tiles per expert
  int splits;        // K splits
  const int32_t* sorted;
  const int32_t* offsets;       // [E + 1] padded expert segments (16-slot blocks)
  const int32_t* chunk_expert;  // expert of each token tile
  const int32_t* chunk_start;   // [E + 1] first token tile of each expert
  const int32_t* counts;        // [E] token-slots of each expert (warp-MMA mode)
  const void* scale;      // 8-bit: scales of this GEMM's weights (kind below)
  int scale_kind;         // 8-bit scales: 0 float32, 1 float16, 2 bfloat16
  int scale_per_tensor;   // 8-bit: one scale per expert instead of one per row
  uint32_t xmask;         // 8-bit codes: 0x80808080 for int8, 0 for uint8 (moe_wna16)
  const uint8_t* zrow;    // 8-bit uint8 codes: zero point per row [E * rows], or null (128)
  int rw_on_input;        // down GEMM: the router weight was applied to the input
  const __half* gscale;   // uint4: f16 group scales [rows, G]
  const uint8_t* gzero;   // uint4: zero points [rows / 2, G], even row in the low nibble
  int G;                  // uint4: groups per row (K / group_size)
  int gs;                 // uint4: group size
  int has_zp;             // uint4: 0 -> implicit zero 8
  int stage;              // uint4: group scales / zeros staged in shared memory per unit
  int gs_log2;            // uint4: log2(group size)
  const float* topk_w;
  __nv_bfloat16* act;     // gate/up output [cap, I]
  float* ypart;           // down output [splits, S, H]
  const float* xinv;      // gate/up: per activation row, 1 / (its power-of-two scale)
  // fused layer: per token tile, the count of gate/up epilogue warps done
  // with its act columns (zeroed by the align kernel); the down GEMM waits
  // for dep_target of them
  int* dep;
  int dep_target;
  // 8-bit down GEMM: act was converted to f16 in place (exact, with the row
  // scales in xinv), so the weights are converted to f16 as well
  int down_f16;
  unsigned* status;
};

// Work unit: token tile (rows [row0, row0 + n) of the expert-sorted
// activations, n <= BN a multiple of 16, all of expert e), weight tile mt
// and K split.
struct Unit {
  int e, row0, n, mt, split;
  int ch;      // token tile (chunk) index
  int single;  // the expert has one token tile: its weight tiles are read once
};

template <int N>
struct IC {
  static constexpr int value = N;
};

// Work unit u -> Unit.  Each expert's segment is cut into token tiles of at
// most BN rows (its chunks); units of one expert are contiguous, and inside
// an expert groups of kRasterGroup weight tiles sweep all of its token
// tiles, so a weight tile is reused from L2 by the tiles that run at the
// same time.
template <int BN>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  const int V = p.MT * p.splits;
  const int c0 = u / V;
  const int e = p.chunk_expert[c0];
  const int cs = p.chunk_start[e];
  const int nce = p.chunk_start[e + 1] - cs;
  const int ue = u - cs * V;
  const int g = ue / (kRasterGroup * nce);
  const int r = ue - g * kRasterGroup * nce;
  const int gsz = min(kRasterGroup, V - g * kRasterGroup);
  const int bl = r / gsz;
  const int v = g * kRasterGroup + (r - bl * gsz);
  Unit out;
  out.e = e;
  out.ch = cs + bl;
  out.single = nce == 1;
  out.row0 = p.offsets[e] + bl * BN;
  out.n = min(BN, p.offsets[e + 1] - out.row0);
  out.mt = v % p.MT;
  out.split = v / p.MT;
  return out;
}

__device__ __forceinline__ int4 pack_unit(const Unit& w) {
  return make_int4(w.e, w.row0, w.mt | (w.split << 16) | (w.single << 31), w.n | (w.ch << 8));
}

// Unit number i of this CTA (u = first unit + i * gridDim.x): from the list
// decoded in the prologue (`len` entries), or decoded on the spot past its
// end.
template <int BN>
__device__ __forceinline__ Unit cta_unit(const TcParams& p, const int4* ulist, int i, int u,
                                         int len = kUnitList) {
  if (i < len) {
    const int4 v = ulist[i];
    Unit w;
    w.e = v.x;
    w.row0 = v.y;
    w.mt = v.z & 0xffff;
    w.split = (v.z >> 16) & 0x7fff;
    w.single = (int)((unsigned)v.z >> 31);
    w.n = v.w & 255;
    w.ch = v.w >> 8;
    return w;
  }
  return decode_unit<BN>(p, u);
}

struct alignas(16) SharedCtl {
  uint64_t fullA[16];
  uint64_t emptyA[16];
  uint64_t fullB[kMaxVirt];
  uint64_t afull[kMaxVirt];     // converted A (and its activations) ready for the MMA
  uint64_t stepfree[kMaxVirt];  // MMAs of the step done: TMEM A stage and B stage free
  uint64_t accfull[2];
  uint64_t accempty[2];
  uint64_t fullS[2];    // uint4 staging: a unit's scales and zeros landed
  uint64_t emptyS[2];   // uint4 staging: the 8 converter warps are done with them
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, SharedCtl* ctl,
                                             unsigned* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = mq::global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (ctl->abort_flag) return false;
      if (mq::global_timer_ns() - t0 > kWaitNs) {
        ctl->abort_flag = 1;
        mq::flag(status, MQ_DEV_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait.  Every lane polls the same barrier (one shared
// access per poll, all lanes see the same phase), so the warp stays
// converged; the verdict is agreed with one vote.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, SharedCtl* ctl,
                                          unsigned* status, int lane) {
  (void)lane;
  bool ok = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, ok)) return true;
  ok = ok || wait_bounded(bar, parity, ctl, status);
  return __all_sync(0xffffffffu, ok);
}

// Same, for long waits off the critical path (the epilogue waiting for a
// whole tile): a short sleep between polls leaves the issue slots to the
// converter warps.
__device__ __forceinline__ bool warp_wait_sleepy(uint64_t* bar, uint32_t parity, SharedCtl* ctl,
                                                 unsigned* status, int lane) {
  int ok = 0;
  if (lane == 0) {
    const unsigned long long t0 = mq::global_timer_ns();
    for (;;) {
      if (mbar_try_wait(bar, parity)) {
        ok = 1;
        break;
      }
      if (ctl->abort_flag) break;
      if (mq::global_timer_ns() - t0 > kWaitNs) {
        ctl->abort_flag = 1;
        mq::flag(status, MQ_DEV_WAIT_TIMEOUT);
        break;
      }
      __nanosleep(256);
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Fused layer, producer side: after this warp's act stores, make them
// visible at GPU scope (and to the tensor-memory-access proxy that loads
// them) before adding 1 to the token tile's counter.
__device__ __forceinline__ void dep_signal(int* cnt, int lane) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicAdd(cnt, 1);
  }
  __syncwarp();
}

// Fused layer, consumer side (warp-uniform): lane 0 polls the counter with
// acquire loads until it reaches target, bounded like every other wait.
__device__ __forceinline__ bool dep_wait(const int* cnt, int target, SharedCtl* ctl,
                                         unsigned* status, int lane) {
  int ok = 0;
  if (lane == 0) {
    const unsigned long long t0 = mq::global_timer_ns();
    for (uint32_t n = 0;; ++n) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= target) {
        ok = 1;
        break;
      }
      if (ctl->abort_flag) break;
      if ((n & 15u) == 15u && mq::global_timer_ns() - t0 > kWaitNs) {
        ctl->abort_flag = 1;
        mq::flag(status, MQ_DEV_WAIT_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Wait used while draining after an abort: ignores the abort flag, still
// bounded in time.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = mq::global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (mq::global_timer_ns() - t0 > kWaitNs) return;
  }
}

// 8-bit scale number i of this GEMM's weights, as float.
__device__ __forceinline__ float load_scale(const TcParams& p, int64_t i) {
  if (p.scale_kind == 1) return __half2float(static_cast<const __half*>(p.scale)[i]);
  if (p.scale_kind == 2) return __bfloat162float(static_cast<const __nv_bfloat16*>(p.scale)[i]);
  return static_cast<const float*>(p.scale)[i];
}

// 16-byte chunk c of a 128-byte swizzled shared-memory row.
__device__ __forceinline__ uint4 ld_chunk(const uint8_t* row, uint32_t c, uint32_t sw) {
  return *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
}

__device__ __forceinline__ uint4 sel4(bool p, const uint4& a, const uint4& b) {
  return make_uint4(p ? a.x : b.x, p ? a.y : b.y, p ? a.z : b.z, p ? a.w : b.w);
}

// Zero point and scale of one weight row at K position k (uint4), each
// broadcast to both f16 halves.
__device__ __forceinline__ void group_words(const TcParams& p, int wrow, int k, uint32_t& zz,
                                            uint32_t& ss) {
  const int g = k / p.gs;
  uint32_t z = 8, sb = 0;  // past the row's end: scale 0 (the activations there are 0 too)
  if (g < p.G) {
    sb = __half_as_ushort(p.gscale[(int64_t)wrow * p.G + g]);
    if (p.has_zp) z = (p.gzero[(int64_t)(wrow >> 1) * p.G + g] >> (4 * (wrow & 1))) & 15u;
  }
  zz = (0x6400u | z) * 0x00010001u;
  ss = sb * 0x00010001u;
}

// --------------------------------------------------------------------------
// Warp-MMA mode (SYNC): the converter warps multiply, the epilogue warps
// finish.  Used for experts that hold a few token-slots (token tiles of 16
// or 32 rows), where one tcgen05.mma per 2 KB of weights costs more issue
// time than the weight stream leaves.
//
// Converter warp (group grp, quarter wq) owns 32 rows of the 128-row weight
// tile: two m16 MMA tiles.  Lane (g, t) holds, for each of its 4 rows, the
// 16-byte chunks t and t + 4 of each 128-byte weight-stage row (int8: K
// [16t, 16t + 16) and [64 + 16t, ...); uint4: [32t, 32t + 32) and
// [128 + 32t, ...)), and from the activation tile the same K range of token
// row 8 tg + g.  MMA k-slice j takes codes [4j, 4j + 4) of a chunk as the
// logical columns (2t, 2t+1, 2t+8, 2t+9), so A and B agree on the K behind
// every column.  Fragment row g reads tile row rg = (g >> 1) | ((g & 1) << 2)
// of its 8-row group: the two rows a quarter-warp reads differ by 4 in the
// 128-byte swizzle phase, so the reads are free of bank conflicts.  In the
// gate/up GEMM fragment rows 0-7 are gate rows i and rows 8-15 the up rows
// i; the epilogue pairs them.
// --------------------------------------------------------------------------
// Not volatile: the MMA is a pure function of its registers, and the
// compiler may then schedule the surrounding shared-memory loads and
// conversions across it.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16)
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Waits until the shared-memory loads that produced `v` have returned (an
// instruction that reads the registers), so that the slot they came from can
// be handed back to the TMA producer while the values are still being used.
template <int N>
__device__ __forceinline__ void consume(const uint4 (&v)[N]) {
  uint32_t x = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) x ^= v[i].x ^ v[i].y ^ v[i].z ^ v[i].w;
  uint32_t sink;
  asm volatile("mov.b32 %0, %1;" : "=r"(sink) : "r"(x));
}

// Row of the 128-row weight tile held by fragment row (tau, h) of lane
// group g in converter quarter wq.
template <int MODE>
__device__ __forceinline__ int sync_tile_row(int wq, int tau, int h, int rg) {
  return MODE == 1 ? (h ? 64 : 0) + 16 * wq + 8 * tau + rg : 32 * wq + 16 * tau + 8 * h + rg;
}

// Weight row (within the expert) of tile row br of weight tile mt.
template <int MODE>
__device__ __forceinline__ int sync_weight_row(const TcParams& p, int mt, int br) {
  return MODE == 1 ? (br >= 64 ? p.I : 0) + mt * 64 + (br & 63) : mt * kTileM + br;
}

template <int MODE, int BITS, int BN, typename C>
__device__ __forceinline__ void conv_sync(const TcParams& p, const int4* ulist, int total,
                                          const uint8_t* sA, const uint8_t* sB, float* partials,
                                          const uint8_t* sS, SharedCtl* ctl, int warp, int lane) {
  constexpr int kEntryK = BITS == 8 ? 128 : 256;
  constexpr int kGA = 256 / kEntryK;
  constexpr int NAG = C::kAStagesSmem / kConvGroups;
  constexpr int ND = C::kSteps;
  constexpr int TG = BN / 8;                  // 8-token MMA groups
  constexpr int kBox = BN * 128;              // bytes of one 64-K activation box
  constexpr bool kBf16 = MODE == 2;           // down GEMM: bf16 act, bf16 weights
  constexpr int PS = C::kPStride;
  const int grp = (warp - kConvWarp0) >> 2;
  const int wq = (warp - kConvWarp0) & 3;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int rg = (g >> 1) | ((g & 1) << 2);
  int br[2][2];  // tile rows [tau][h]
#pragma unroll
  for (int tau = 0; tau < 2; ++tau)
#pragma unroll
    for (int h = 0; h < 2; ++h) br[tau][h] = sync_tile_row<MODE>(wq, tau, h, rg);
  const int rows_e = MODE == 1 ? 2 * p.I : p.H;
  int lit = 0, st = 0;
  bool ok = true;
  for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
    const Unit w = cta_unit<BN>(p, ulist, ui, u);
    const int ks0 = w.split * p.ksteps / p.splits;
    const int ks1 = (w.split + 1) * p.ksteps / p.splits;
    // real token-slots of this tile (the rest of its rows are padding)
    const int nreal = p.counts ? max(1, min(w.n, p.counts[w.e] - (w.row0 - p.offsets[w.e]))) : w.n;
    const int ntg = min(TG, (nreal + 7) >> 3);
    // 8-bit: 1024 + z (f16) or 2^23 + z (bf16) of this thread's rows
    uint32_t zz8[2][2];
    float zf8[2][2];
    int64_t wrow[2][2];  // global weight rows
#pragma unroll
    for (int tau = 0; tau < 2; ++tau)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        wrow[tau][h] = (int64_t)w.e * rows_e + sync_weight_row<MODE>(p, w.mt, br[tau][h]);
        uint32_t z = 128u;
        if (BITS == 8 && p.zrow) z = p.zrow[wrow[tau][h]];
        zz8[tau][h] = (0x6400u | z) * 0x00010001u;
        zf8[tau][h] = 8388608.0f + (float)z;
      }
    // two accumulator sets (even / odd k-slices, 8-bit) so that an MMA rarely
    // waits for the previous one on its accumulator; added at the unit end
    constexpr int NS = (BITS == 8 && TG <= 2) ? 2 : 1;
    // uint4: the unit's staged group scales (waited for by every converter
    // warp on every unit, so that its parity waits stay exact)
    const uint8_t* stg = sS + (ui & 1) * kStageBytes;
    if (BITS == 4 && p.stage) {
      ok = warp_wait(&ctl->fullS[ui & 1], (ui >> 1) & 1, ctl, p.status, lane);
      if (!ok) break;
    }
    float acc[NS][2][TG][4];
#pragma unroll
    for (int q = 0; q < NS; ++q)
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < TG; ++b)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[q][a][b][r] = 0.0f;
    for (int ks = ks0; ks < ks1; ks += kGA, ++st) {
      const int nk = min(kGA, ks1 - ks);
      if (st % kConvGroups != grp) continue;
      const int d = st % ND;
      // the step's activations (exact parity: slot d serves this group only,
      // and this warp waited for its previous fill itself)
      ok = warp_wait(&ctl->fullB[d], (st / ND) & 1, ctl, p.status, lane);
      if (!ok) break;
      const uint8_t* bstep = sB + d * C::kBBytes;
      for (int j = 0; j < nk && ok; ++j, ++lit) {
        const int sa = grp * NAG + lit % NAG;
        // uint4: group scales and zero points of this stage's two K halves,
        // loaded before the tile wait
        float gsc[2][2][2];
        uint32_t gzz[2][2][2];
        if constexpr (BITS == 4) {
          constexpr uint32_t kMagic = kBf16 ? 0x4300u : 0x6400u;
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            // a K half past the row's end (K = 128 mod 256) has no group
            const int gi = min(((ks + j) * kEntryK + 128 * k2) >> p.gs_log2, p.G - 1);
#pragma unroll
            for (int tau = 0; tau < 2; ++tau)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int64_t row = wrow[tau][h];
                uint32_t z = 8u;
                if (p.stage) {
                  const int tr = br[tau][h];
                  gsc[tau][h][k2] = __half2float(__ushort_as_half(
                      reinterpret_cast<const uint16_t*>(stg)[tr * p.G + gi]));
                  if (p.has_zp) z = (stg[256 * p.G + (tr >> 1) * p.G + gi] >> (4 * (tr & 1))) & 15u;
                } else {
                  gsc[tau][h][k2] = __half2float(p.gscale[row * p.G + gi]);
                  if (p.has_zp) z = (p.gzero[(row >> 1) * p.G + gi] >> (4 * (int)(row & 1))) & 15u;
                }
                gzz[tau][h][k2] = (kMagic | z) * 0x00010001u;
              }
          }
        }
        ok = warp_wait(&ctl->fullA[sa], (lit / NAG) & 1, ctl, p.status, lane);
        if (!ok) break;
        const uint8_t* a = sA + sa * kABytes;
        // this thread's 8 chunks of the stage into registers; the slot goes
        // back to the producer as soon as every lane's loads have returned,
        // so that the ring's slots are in flight to HBM rather than held
        // through the conversion and the MMAs
        uint4 pcl[8];  // [tau][h][k2] = pcl[4 tau + 2 h + k2]: chunks t and t + 4
#pragma unroll
        for (int tau = 0; tau < 2; ++tau)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2)
              pcl[4 * tau + 2 * h + k2] =
                  ld_chunk(a + br[tau][h] * 128, (uint32_t)(t + 4 * k2), (uint32_t)rg);
        consume(pcl);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->emptyA[sa]);
        if constexpr (BITS == 8) {
          uint4 pc[2][2][2];
#pragma unroll
          for (int tau = 0; tau < 2; ++tau)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) pc[tau][h][k2] = pcl[4 * tau + 2 * h + k2];
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            uint32_t lo[2][2][4], hi[2][2][4];  // [tau][h][jj]
#pragma unroll
            for (int tau = 0; tau < 2; ++tau)
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                  if constexpr (kBf16)
                    int8x4_to_bf16x4(word_of(pc[tau][h][k2], jj), p.xmask, zf8[tau][h],
                                     lo[tau][h][jj], hi[tau][h][jj]);
                  else
                    int8x4_to_f16x4(word_of(pc[tau][h][k2], jj), p.xmask, zz8[tau][h],
                                    lo[tau][h][jj], hi[tau][h][jj]);
                }
            // activation box 2j + k2 (64 K), row 8 tg + g, chunks 2t and 2t + 1
            const uint8_t* bb = bstep + (2 * j + k2) * kBox;
#pragma unroll
            for (int tg = 0; tg < TG; ++tg) {
              if (tg >= ntg) break;
              const int n = 8 * tg + g;
              const uint4 b0 = ld_chunk(bb + n * 128, (uint32_t)(2 * t), (uint32_t)(n & 7));
              const uint4 b1 = ld_chunk(bb + n * 128, (uint32_t)(2 * t + 1), (uint32_t)(n & 7));
              const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
              // consecutive MMAs go to different accumulators: an MMA waits
              // for the previous one on its accumulator
#pragma unroll
              for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int tau = 0; tau < 2; ++tau)
                  mma16816<kBf16>(acc[(jj & 1) % NS][tau][tg], lo[tau][0][jj], lo[tau][1][jj],
                                  hi[tau][0][jj], hi[tau][1][jj], bw[2 * jj], bw[2 * jj + 1]);
            }
          }
        } else {
          const int kdim = MODE == 1 ? p.H : p.I;
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            if ((ks + j) * kEntryK + 128 * k2 >= kdim) break;  // half-filled last stage
            uint4 pc[2][2];  // [tau][h]: chunk t + 4 k2 of the row
#pragma unroll
            for (int tau = 0; tau < 2; ++tau)
#pragma unroll
              for (int h = 0; h < 2; ++h) pc[tau][h] = pcl[4 * tau + 2 * h + k2];
            // the group's partial sums, in two sets (one per octet of an
            // octet pair) so that consecutive MMAs use different accumulators
            float part[2][2][TG][4];
#pragma unroll
            for (int o2 = 0; o2 < 2; ++o2)
#pragma unroll
              for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                for (int b2 = 0; b2 < TG; ++b2)
#pragma unroll
                  for (int r = 0; r < 4; ++r) part[o2][a2][b2][r] = 0.0f;
            // two octet pairs of the 32-code chunk (16 K each)
#pragma unroll
            for (int op = 0; op < 2; ++op) {
              // activations: K [32t + 128 k2, +32) in box 2 k2 + (t >> 1),
              // chunks 4 (t & 1) + 2 op and + 1
              const uint8_t* bb = bstep + (2 * k2 + (t >> 1)) * kBox;
              uint32_t bw[TG][8];
#pragma unroll
              for (int tg = 0; tg < TG; ++tg) {
                if (tg >= ntg) break;
                const int n = 8 * tg + g;
                const uint32_t c0 = (uint32_t)(4 * (t & 1) + 2 * op);
                const uint4 b0 = ld_chunk(bb + n * 128, c0, (uint32_t)(n & 7));
                const uint4 b1 = ld_chunk(bb + n * 128, c0 + 1, (uint32_t)(n & 7));
                bw[tg][0] = b0.x; bw[tg][1] = b0.y; bw[tg][2] = b0.z; bw[tg][3] = b0.w;
                bw[tg][4] = b1.x; bw[tg][5] = b1.y; bw[tg][6] = b1.z; bw[tg][7] = b1.w;
              }
#pragma unroll
              for (int tau = 0; tau < 2; ++tau) {
                uint32_t wv[2][2][4];  // [h][octet in pair][word]
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                  for (int oo = 0; oo < 2; ++oo)
                    uint4x8_to_16<kBf16>(word_of(pc[tau][h], 2 * op + oo), gzz[tau][h][k2],
                                         wv[h][oo]);
#pragma unroll
                for (int oo = 0; oo < 2; ++oo)
#pragma unroll
                  for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                    for (int tg = 0; tg < TG; ++tg) {
                      if (tg >= ntg) break;
                      mma16816<kBf16>(part[oo][tau][tg], wv[0][oo][2 * jj], wv[1][oo][2 * jj],
                                      wv[0][oo][2 * jj + 1], wv[1][oo][2 * jj + 1],
                                      bw[tg][4 * oo + 2 * jj], bw[tg][4 * oo + 2 * jj + 1]);
                    }
              }
            }
#pragma unroll
            for (int tau = 0; tau < 2; ++tau)
#pragma unroll
              for (int tg = 0; tg < TG; ++tg)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                  acc[0][tau][tg][r] = fmaf(gsc[tau][r >> 1][k2],
                                            part[0][tau][tg][r] + part[1][tau][tg][r],
                                            acc[0][tau][tg][r]);
          }
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->stepfree[d]);  // activation slot d is free
    }
    if (!ok) break;
    if (BITS == 4 && p.stage) {  // done with the unit's staged scales
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->emptyS[ui & 1]);
    }
    // hand this unit's partial sums to the epilogue (all 8 converter warps
    // arrive, a group without steps in the unit with zeros)
    const int buf = ui % C::kPBufs;
    const uint32_t par = C::kPBufs == 2 ? (((ui >> 1) & 1) ^ 1) : ((ui & 1) ^ 1);
    ok = warp_wait(&ctl->accempty[buf], par, ctl, p.status, lane);
    if (!ok) break;
    float* P = partials + (buf * kConvGroups + grp) * BN * PS;
#pragma unroll
    for (int tau = 0; tau < 2; ++tau)
#pragma unroll
      for (int tg = 0; tg < TG; ++tg)
#pragma unroll
        for (int r = 0; r < 4; ++r)
          P[(8 * tg + 2 * t + (r & 1)) * PS + br[tau][r >> 1]] =
              NS == 2 ? acc[0][tau][tg][r] + acc[NS - 1][tau][tg][r] : acc[0][tau][tg][r];
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->accfull[buf]);
  }
}

template <int MODE, int BITS, int BN, typename C>
__device__ __forceinline__ void epi_sync(const TcParams& p, const int4* ulist, int total,
                                         const float* partials, SharedCtl* ctl, int warp,
                                         int lane) {
  constexpr int PS = C::kPStride;
  const int e = (warp - kEpiWarp0) * 32 + lane;  // 0..127
  mq::pdl_wait();
  for (int u = blockIdx.x, t = 0; u < total; u += gridDim.x, ++t) {
    const Unit w = cta_unit<BN>(p, ulist, t, u);
    // per-column values (column = lane): MODE 1 the activation row scale
    // (times the router weight when it applies to the input), MODE 2 the
    // token-slot and its router weight; loaded before the wait
    float colf = MODE == 1 ? 1.0f : 0.0f;
    int colslot = p.S;
    if (lane < w.n) {
      if (MODE == 1) colf = p.xinv[w.row0 + lane];
      if (MODE == 2 || p.rw_on_input) colslot = p.sorted[w.row0 + lane];
    }
    if (MODE == 1 && p.rw_on_input) colf *= colslot < p.S ? p.topk_w[colslot] : 0.0f;
    if (MODE == 2 && colslot < p.S) colf = p.rw_on_input ? 1.0f : p.topk_w[colslot];
    const int buf = t % C::kPBufs;
    const uint32_t par = C::kPBufs == 2 ? ((t >> 1) & 1) : (t & 1);
    float sc0 = 1.0f, sc1 = 1.0f;
    int col_out = 0;
    if (MODE == 1) {
      const int i = e & 63;
      const int64_t wr = (int64_t)w.e * 2 * p.I + w.mt * 64 + i;
      if (BITS == 8) {
        sc0 = load_scale(p, p.scale_per_tensor ? w.e : wr);
        sc1 = load_scale(p, p.scale_per_tensor ? w.e : wr + p.I);
      }
      col_out = w.mt * 64 + (BITS == 8 ? i : permute_octet(i));
    } else if (BITS == 8) {
      sc0 = load_scale(p, p.scale_per_tensor ? w.e : (int64_t)w.e * p.H + w.mt * kTileM + e);
    }
    if (!warp_wait_sleepy(&ctl->accfull[buf], par, ctl, p.status, lane)) break;
    const float* P0 = partials + (buf * kConvGroups) * BN * PS;
    const float* P1 = P0 + BN * PS;
    if (MODE == 1) {
      // threads 0-63: even columns, 64-127: odd columns; pair i = e & 63
      const int i = e & 63;
      for (int c = e >> 6; c < w.n; c += 2) {
        const float xs = __shfl_sync(0xffffffffu, colf, c);
        const float gt = (P0[c * PS + i] + P1[c * PS + i]) * sc0 * xs;
        const float up = (P0[c * PS + 64 + i] + P1[c * PS + 64 + i]) * sc1 * xs;
        const float a = __fdividef(gt * up, 1.0f + __expf(-gt));  // silu(g) * up
        p.act[(int64_t)(w.row0 + c) * p.I + col_out] = __float2bfloat16_rn(a);
      }
    } else {
      float* yp = p.ypart + (int64_t)w.split * p.S * p.H + w.mt * kTileM + e;
      for (int c = 0; c < w.n; ++c) {
        const int sl = __shfl_sync(0xffffffffu, colslot, c);
        const float f = __shfl_sync(0xffffffffu, colf, c);
        if (sl < p.S) yp[(int64_t)sl * p.H] = (P0[c * PS + e] + P1[c * PS + e]) * sc0 * f;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->accempty[buf]);
  }
}

// f16 operands carry an exact power-of-two scale per activation row (xinv
// undoes it in the epilogue); the 8-bit down GEMM runs bf16 operands on act
// as written.
// MODE 1: gate/up GEMM, SiLU-and-mul epilogue -> act (bf16).
// MODE 2: down GEMM on act (uint4: converted in place to scaled f16 in
//         between), router-weighted epilogue -> ypart.
//
// `st` numbers MMA steps (256 K, i.e. kGA weight stages of 16 KB, of one
// work unit) in schedule order; step st belongs to converter group
// st % kConvGroups and uses tensor-memory / activation slot st % ND.
//
// A phase-parity wait is exact only if the waiter knows that the barrier's
// previous phase has completed (a barrier two phases behind shows the parity
// being waited for).  Hence: the weight ring is split into one half per
// converter group, each with its own count of weight stages (one sequential
// consumer per slot); a converter waits for its step's activations only
// after it has seen the MMAs of the slot's previous use complete.
//
// FUSED: the whole expert MLP of an 8-bit layer in one persistent launch.
// Phase 1 is the gate/up GEMM (p, tmA, tmB), phase 2 the down GEMM (p2,
// tmA2, tmB2) on the same rings and tensor memory; every role walks its
// phase-1 units, then its phase-2 units, so the weight stream runs on
// across the boundary.  A down unit's activation tile (act rows of one
// token tile) is loaded only once all gate/up units of that tile have
// stored their act columns: each of the 4 epilogue warps of a gate/up unit
// adds 1 to the tile's counter (release), and the activation producer of a
// down unit waits (acquire, bounded) until the counter reaches 4 x the
// gate/up tiles per expert.  Phase 2 continues the round-robin over the
// concatenated unit list, and every CTA finishes its gate/up units before
// its down units: a down unit only waits for gate/up units, which wait for
// nothing outside their CTA, so every wait ends once all CTAs are resident
// (one CTA per SM, grid <= SMs).
template <int MODE, int BITS, int BN, bool SYNC, bool FUSED, bool F16D>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                          const TcParams& p, const CUtensorMap& tmA2,
                                          const CUtensorMap& tmB2, const TcParams& p2) {
  using C = CfgOf<MODE, BITS, BN, SYNC>;
  static_assert(!FUSED || (MODE == 1 && BITS == 8 && !SYNC &&
                           std::is_same<CfgOf<1, 8, BN>, CfgOf<2, 8, BN>>::value),
                "fused layer: 8-bit, tensor-core consumers, one tile shape for both GEMMs");
  // one weight stage = 128 rows x 128 bytes: 128 K of int8 or 256 K of uint4
  constexpr int kEntryK = BITS == 8 ? 128 : 256;
  constexpr int kGA = 256 / kEntryK;  // weight stages per MMA step (256 K)
  constexpr int kEntryCols = kEntryK / 2;
  constexpr int NA = C::kAStagesSmem;
  constexpr int NAG = NA / kConvGroups;  // weight-ring slots per converter group
  static_assert(kConvGroups == 2 && NAG >= 2, "two converter groups, two slots each");
  constexpr int ND = C::kSteps;
  constexpr int NV = C::kVirt;  // barrier slots of the step ring (stage st % ND, slot st % NV)
  constexpr int NB = C::kBSlots;  // activation ring slots (st % NB)
  constexpr int kBBytesK = C::kBBytesK;
  constexpr int kBBytes = C::kBBytes;
  constexpr int kACol0 = C::kACol0;
  // MMAs always run N = BN: a token tile's rows past its n belong to other
  // tiles (or are zero fill), and the accumulator columns they produce are
  // never read.  A compile-time descriptor keeps the issue loop short.
  // The 8-bit down GEMM reads act as written, in bf16 (weights converted to
  // bf16, exactly); every other GEMM runs f16 operands (kBf16M, kIdescM per
  // GEMM phase below).
  // In warp-MMA mode both down GEMMs read act as written (bf16); uint4
  // weights enter as the exact q - z and their group scale multiplies each
  // group's float32 partial sum.
  static_assert(NA <= 16, "ring sizes");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;                 // NA x 16 KB (int8 codes, 128-byte swizzle)
  uint8_t* sB = smem + NA * kABytes;  // NB x kG x 2 x BN x 128 B (16-bit, 128-byte swizzle)
  float* partials = reinterpret_cast<float*>(sB + NB * kBBytes);  // warp-MMA mode only
  constexpr int kPartBytes = partial_bytes<SYNC, BN>();
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(sB + NB * kBBytes + kPartBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The first TMA of each map waits for its descriptor (a kernel parameter
  // in global memory): start both fetches before the set-up below, so that
  // they overlap it.
  if (threadIdx.x == 32) tma_prefetch_desc(&tmA);
  if (threadIdx.x == 64) tma_prefetch_desc(&tmB);
  if (FUSED && threadIdx.x == 96) tma_prefetch_desc(&tmA2);
  if (FUSED && threadIdx.x == 128) tma_prefetch_desc(&tmB2);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NA; ++s) {
      mbar_init(&ctl->fullA[s], 1);
      mbar_init(&ctl->emptyA[s], C::kWPG);  // the warps of the converter group
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&ctl->fullB[s], 1);
      mbar_init(&ctl->afull[s], C::kWPG);
      // MMA commit; warp-MMA mode: the 4 warps of the step's converter group
      mbar_init(&ctl->stepfree[s], SYNC ? 4 : 1);
    }
    for (int s = 0; s < 2; ++s) {
      // one commit per issuer; warp-MMA mode: all 8 converter warps
      mbar_init(&ctl->accfull[s], SYNC ? 4 * kConvGroups : C::kNI);
      mbar_init(&ctl->accempty[s], 4);
      mbar_init(&ctl->fullS[s], 1);
      mbar_init(&ctl->emptyS[s], C::kWPG * kConvGroups);
    }
    mbar_init(&ctl->drain, C::kNI);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (!SYNC && warp == 0) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Decode this CTA's work units once, all threads in parallel, so that no
  // role waits on the schedule's global loads at a unit boundary (the fused
  // layer: half of the list for each GEMM).
  constexpr int kUL = FUSED ? kUnitList / 2 : kUnitList;
  const int total = p.chunk_start[p.E] * p.MT * p.splits;
  const int total2 = FUSED ? p2.chunk_start[p2.E] * p2.MT * p2.splits : 0;
  // the fused layer's down units continue the round-robin after the gate/up
  // units: unit u2 is item total + u2 of the concatenated list
  const int u02 = FUSED ? (int)((blockIdx.x + gridDim.x - (unsigned)total % gridDim.x) % gridDim.x) : 0;
  int4* ulist = reinterpret_cast<int4*>(ctl + 1);
  int4* ulist2 = ulist + kUL;
  uint8_t* sS = reinterpret_cast<uint8_t*>(ulist + kUnitList);  // uint4 staging, 2 buffers
  for (int i = threadIdx.x; i < kUL; i += C::kThreads) {
    const int u = blockIdx.x + i * gridDim.x;
    if (u >= total) break;
    ulist[i] = pack_unit(decode_unit<BN>(p, u));
  }
  if constexpr (FUSED)
    for (int i = threadIdx.x; i < kUL; i += C::kThreads) {
      const int u = u02 + i * gridDim.x;
      if (u >= total2) break;
      ulist2[i] = pack_unit(decode_unit<BN>(p2, u));
    }
  // Runs fn once per GEMM phase with that phase's parameters, tensor maps,
  // unit list, unit count and this CTA's first unit.
  auto phases = [&](auto&& fn) {
    fn(IC<MODE>{}, p, tmA, tmB, static_cast<const int4*>(ulist), total, (int)blockIdx.x);
    if constexpr (FUSED) fn(IC<2>{}, p2, tmA2, tmB2, static_cast<const int4*>(ulist2), total2, u02);
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = SYNC ? 0u : ctl->tmem_base;
  // The unit list (from the align kernel, two or more launches back) and the
  // weights do not depend on the previous kernel: the weight stream starts
  // at once.  The activations (and, in the epilogue, their row scales) come
  // from the previous kernel: the roles that read them wait for it first.
  mq::pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------ A producer (int8 weights) ----
    // The whole warp walks the schedule (so it stays converged); lane 0
    // issues the copies.
    int st = 0;
    int lit0 = 0, lit1 = 0;  // weight stages issued into each group's half of the ring
    bool ok = true;
    // The weight tiles of an expert with a single token tile are read once
    // per pass: first out of L2, so that what is reused (activations,
    // partial sums, the kernel's code) stays (Mixtral-shaped T=1 gate/up
    // 57.4 -> 49.7 us, T=64 165 -> 155 us).  Experts with several token
    // tiles share each weight tile between them through L2 (their units run
    // side by side), and keep the default policy (with evict-first,
    // prefill at T=4096 lost 4 % in the gate/up GEMM).
    const uint64_t wpol = l2_policy_evict_first();
    phases([&](auto ph_tag, const TcParams& prm, const CUtensorMap& mA, const CUtensorMap& mB,
               const int4* ul, int tot, int u0) {
      constexpr int M = decltype(ph_tag)::value;
      for (int u = u0, ui = 0; u < tot && ok; u += gridDim.x, ++ui) {
        const Unit w = cta_unit<BN>(prm, ul, ui, u, kUL);
        const int ks0 = w.split * prm.ksteps / prm.splits;
        const int ks1 = (w.split + 1) * prm.ksteps / prm.splits;
        for (int ks = ks0; ks < ks1 && ok; ks += kGA, ++st) {
          const int g = st % kConvGroups;
          const int nk = min(kGA, ks1 - ks);
          for (int j = 0; j < nk; ++j) {
            const int n = g ? lit1 : lit0;
            const int s = g * NAG + n % NAG;
            ok = warp_wait(&ctl->emptyA[s], ((n / NAG) & 1) ^ 1, ctl, prm.status, lane);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(&ctl->fullA[s], kABytes);
              uint8_t* a = sA + s * kABytes;
              // {K, row in half, gate/up half, expert}: 64 gate rows then 64 up rows
              if (M == 1 && w.single)
                tma_load_4d_hint(a, &mA, &ctl->fullA[s], (ks + j) * 128, w.mt * 64, 0, w.e, wpol);
              else if (M == 1)
                tma_load_4d(a, &mA, &ctl->fullA[s], (ks + j) * 128, w.mt * 64, 0, w.e);
              else if (w.single)
                tma_load_2d_hint(a, &mA, &ctl->fullA[s], (ks + j) * 128, w.e * prm.H + w.mt * kTileM,
                                 wpol);
              else
                tma_load_2d(a, &mA, &ctl->fullA[s], (ks + j) * 128, w.e * prm.H + w.mt * kTileM);
            }
            __syncwarp();
            if (g) ++lit1; else ++lit0;
          }
        }
      }
    });
    // Never leave with copies in flight: wait for the last load issued into
    // each slot of both halves.
    if (lane == 0) {
      for (int g = 0; g < kConvGroups; ++g) {
        const int n = g ? lit1 : lit0;
        for (int d = 1; d <= (n < NAG ? n : NAG); ++d) {
          const int j = n - d;
          wait_drain(&ctl->fullA[g * NAG + j % NAG], (j / NAG) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------ B producer (activations) ----
    mq::pdl_wait();
    int st = 0;
    bool ok = true;
    int nstaged = 0;  // units whose uint4 scales were staged
    phases([&](auto ph_tag, const TcParams& prm, const CUtensorMap& mA, const CUtensorMap& mB,
               const int4* ul, int tot, int u0) {
      constexpr int M = decltype(ph_tag)::value;
      int dep_ch = -1;  // fused layer: the last token tile whose gate/up outputs were waited for
      for (int u = u0, ui = 0; u < tot && ok; u += gridDim.x, ++ui) {
        const Unit w = cta_unit<BN>(prm, ul, ui, u, kUL);
        const int ks0 = w.split * prm.ksteps / prm.splits;
        const int ks1 = (w.split + 1) * prm.ksteps / prm.splits;
        if (BITS == 4 && prm.stage) {
          // the unit's group scales (and zero points): one contiguous block per
          // 64 (gate/up) or 128 (down) weight rows, 16-byte aligned because
          // tiles start at multiples of 64 rows.  Staged here rather than by
          // the weight producer, whose stream would otherwise stall until the
          // converters have finished the unit two back (this producer runs at
          // most ND steps ahead of the MMAs, so it seldom waits here)
          const int b = ui & 1;
          ok = warp_wait(&ctl->emptyS[b], ((ui >> 1) & 1) ^ 1, ctl, prm.status, lane);
          if (!ok) break;
          if (lane == 0) {
            uint8_t* dst = sS + b * kStageBytes;
            const uint32_t sbytes = 128u * prm.G * 2u;
            const uint32_t zbytes = prm.has_zp ? 64u * prm.G : 0u;
            mbar_arrive_expect_tx(&ctl->fullS[b], sbytes + zbytes);
            if (M == 1) {
              const int64_t r0 = (int64_t)w.e * 2 * prm.I + w.mt * 64;  // gate rows; up rows + I
              bulk_load(dst, prm.gscale + r0 * prm.G, sbytes / 2, &ctl->fullS[b]);
              bulk_load(dst + sbytes / 2, prm.gscale + (r0 + prm.I) * prm.G, sbytes / 2, &ctl->fullS[b]);
              if (prm.has_zp) {
                bulk_load(dst + sbytes, prm.gzero + (r0 >> 1) * prm.G, zbytes / 2, &ctl->fullS[b]);
                bulk_load(dst + sbytes + zbytes / 2, prm.gzero + ((r0 + prm.I) >> 1) * prm.G, zbytes / 2,
                          &ctl->fullS[b]);
              }
            } else {
              const int64_t r0 = (int64_t)w.e * prm.H + w.mt * kTileM;
              bulk_load(dst, prm.gscale + r0 * prm.G, sbytes, &ctl->fullS[b]);
              if (prm.has_zp) bulk_load(dst + sbytes, prm.gzero + (r0 >> 1) * prm.G, zbytes, &ctl->fullS[b]);
            }
          }
          __syncwarp();
          ++nstaged;
        }
        if constexpr (FUSED && M == 2) {
          // the token tile's act rows: every gate/up unit of the tile is done
          if (w.ch != dep_ch) {
            ok = dep_wait(prm.dep + w.ch, prm.dep_target, ctl, prm.status, lane);
            if (!ok) break;
            dep_ch = w.ch;
          }
        }
        for (int ks = ks0; ks < ks1; ks += kGA, ++st) {
          const int nboxes = min(kGA, ks1 - ks) * kEntryK / 64;  // 64-K activation boxes
          const int d = st % NB;  // activation slot
          const int v = st % NV;  // the step's barriers
          if (st >= NB) {  // the MMAs of the slot's previous fill (step st - NB) are done
            ok = warp_wait(&ctl->stepfree[(st - NB) % NV], ((st - NB) / NV) & 1, ctl, prm.status,
                           lane);
            if (!ok) break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&ctl->fullB[v], nboxes * (kBBytesK / 2));
            uint8_t* b = sB + d * kBBytes;
            for (int j = 0; j < nboxes; ++j)  // past K the box reads the fill value 0
              tma_load_2d(b + j * (kBBytesK / 2), &mB, &ctl->fullB[v], ks * kEntryK + 64 * j,
                          w.row0);
          }
          __syncwarp();
        }
      }
    });
    if (lane == 0) {
      const int n = st < NB ? st : NB;
      for (int dd = 1; dd <= n; ++dd) {
        const int j = st - dd;
        wait_drain(&ctl->fullB[j % NV], (j / NV) & 1);
      }
      for (int d = 1; d <= (nstaged < 2 ? nstaged : 2); ++d) {
        const int j = nstaged - d;
        wait_drain(&ctl->fullS[j & 1], (j >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (SYNC && warp == 1) {
    // warp-MMA mode: no MMA issuer
  } else if (warp == 1 || (C::kNI == 2 && warp == C::kIss2W)) {
    // ------------------------------------------------- MMA issuer ----
    // One thread runs this loop: it alone waits, issues and commits, so the
    // rest of the warp has nothing to agree on.  Per 256-K step: one wait
    // (the converted A stage; the converters have also seen the step's
    // activations land), the 16 MMAs from one asm statement, one commit.
    // With two issuers, issuer ip takes the steps st with st % 2 == ip and
    // accumulates them into half ip of the unit's accumulator buffer.
    if (lane == 0) {
      constexpr uint32_t kBoxD = (uint32_t)(kBBytesK / 2) >> 4;  // one 64-K activation box
      constexpr uint32_t kStageD = (uint32_t)kBBytes >> 4;        // one activation stage
      // descriptor of stage 0's first K slice; stage d's differs only in the
      // start-address field (address >> 4, no carry below 256 KB)
      const uint64_t b_desc0 = smem_desc_k_sw128(smem_addr(sB));
      const int ip = warp == 1 ? 0 : 1;
      int st = 0, t = 0;
      bool ok = true;
      phases([&](auto ph_tag, const TcParams& prm, const CUtensorMap& mA, const CUtensorMap& mB,
               const int4* ul, int tot, int u0) {
        constexpr int M = decltype(ph_tag)::value;
        // operand type: bf16 in the 8-bit down GEMM (unless act was converted
        // to f16 in place: F16D) and in the warp-MMA mode, else f16
        constexpr uint32_t kIdescM = (M == 2 && (BITS == 8 || SYNC) && !F16D)
                                         ? idesc_bf16_f32(kTileM, BN)
                                         : idesc_f16_f32(kTileM, BN);
        for (int u = u0, ui = 0; u < tot && ok; u += gridDim.x, ++t, ++ui) {
          const Unit w = cta_unit<BN>(prm, ul, ui, u, kUL);
          const int ks0 = w.split * prm.ksteps / prm.splits;
          const int ks1 = (w.split + 1) * prm.ksteps / prm.splits;
          const int buf = t % C::kAccBufs;
          ok = wait_bounded(&ctl->accempty[buf], ((t / C::kAccBufs) & 1) ^ 1, ctl, prm.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + (buf * C::kNI + ip) * BN;
          uint32_t acc = 0;  // the first step of this issuer in the unit overwrites
          for (int ks = ks0; ks < ks1; ks += kGA, ++st) {
            if (C::kNI == 2 && (st & 1) != ip) continue;
            const int dc = st % ND;                          // A stage and activation slot
            const int vc = st % NV;                          // their barriers
            const uint32_t phc = (uint32_t)(st / NV) & 1u;  // parity of this use
            const int nmma = min(kGA, ks1 - ks) * kEntryK / 16;  // K = 16 per MMA
            ok = wait_bounded(&ctl->afull[vc], phc, ctl, prm.status);
            if (!ok) break;
            tc_fence_after();
            // four K slices of 16 (32 bytes) per 64-K activation box
            const uint64_t b_desc = b_desc0 + (uint64_t)((st % NB) * kStageD);
            const uint32_t a_tmem = tmem + kACol0 + dc * kAColsPerStep;
            if (nmma == 16) {
              mma_ts_x16<2, 4, 6, kBoxD, kBoxD + 2, kBoxD + 4, kBoxD + 6, 2 * kBoxD, 2 * kBoxD + 2,
                         2 * kBoxD + 4, 2 * kBoxD + 6, 3 * kBoxD, 3 * kBoxD + 2, 3 * kBoxD + 4,
                         3 * kBoxD + 6>(d_tmem, a_tmem, b_desc, kIdescM, acc);
            } else {
              for (int kk = 0; kk < nmma; ++kk)
                mma_ts(d_tmem, a_tmem + kk * 8, b_desc + (uint64_t)((kk >> 2) * kBoxD + (kk & 3) * 2),
                       kIdescM, kk > 0 ? 1u : acc);
            }
            acc = 1;
            mma_commit(&ctl->stepfree[vc]);
          }
          if (!ok) break;
          mma_commit(&ctl->accfull[buf]);
        }
      });
      // every MMA issued here must finish before tensor memory is freed
      mma_commit(&ctl->drain);
      wait_drain(&ctl->drain, 0);
    }
    __syncwarp();
  } else if (SYNC && warp < C::kEpiW0) {
    if constexpr (SYNC)
      conv_sync<MODE, BITS, BN, C>(p, ulist, total, sA, sB, partials, sS, ctl, warp, lane);
  } else if (SYNC) {
    if constexpr (SYNC) epi_sync<MODE, BITS, BN, C>(p, ulist, total, partials, ctl, warp, lane);
  } else if (warp < C::kEpiW0) {
    // -------------------------------------------------- converters ----
    // Per MMA step of this group: for each weight stage, wait for the tile
    // in this group's half of the ring, read this thread's row into
    // registers, convert it (int8: exact; uint4: (q - z) * s per group),
    // write it into the step's tensor-memory A stage and hand the slot back.
    // Then wait for the step's activations and tell the MMA issuer.
    const int cw = warp - C::kConvW0;
    const int grp = cw / C::kWPG;  // takes the steps with st % kConvGroups == grp
    const int q = warp & 3;        // tensor-memory lane quarter of this warp
    const int r = q * 32 + lane;
    // uint4 with two warps per quarter: this warp's half of each stage's K
    constexpr int NH = C::kWPG / 4;   // parts of a stage's row (1 or 2)
    constexpr int NCH = 8 / NH;       // 16-byte chunks of its row per thread
    const int khalf = (cw % C::kWPG) >> 2;
    const uint32_t tcol = ((uint32_t)(q * 32) << 16) + kACol0;
    int lit = 0, st = 0;  // lit: weight stages consumed by this group
    bool ok = true;
    phases([&](auto ph_tag, const TcParams& prm, const CUtensorMap& mA, const CUtensorMap& mB,
               const int4* ul, int tot, int u0) {
      constexpr int M = decltype(ph_tag)::value;
      constexpr bool kBf16M = M == 2 && (BITS == 8 || SYNC) && !F16D;
      // this thread's row of the weight tile: gate/up lanes (2i, 2i+1) hold
      // gate row i and up row i (rotated read order keeps the pair on
      // distinct banks); down: row r
      const int i_gu = q * 16 + (lane >> 1);
      const int srow = M == 1 ? ((lane & 1) ? 64 + i_gu : i_gu) : r;
      const int rot = (M == 1 && (lane & 1)) ? NCH / 2 : 0;
      const uint32_t sw = srow & 7;  // 128-byte swizzle phase of this row
      const bool rt = rot != 0;
      for (int u = u0, ui = 0; u < tot && ok; u += gridDim.x, ++ui) {
        const Unit w = cta_unit<BN>(prm, ul, ui, u, kUL);
        const int ks0 = w.split * prm.ksteps / prm.splits;
        const int ks1 = (w.split + 1) * prm.ksteps / prm.splits;
        // this thread's weight row (uint4 group scales and zero points)
        const int wrow = M == 1 ? w.e * 2 * prm.I + ((lane & 1) ? prm.I : 0) + w.mt * 64 + q * 16 + (lane >> 1)
                                   : w.e * prm.H + w.mt * kTileM + r;
        // 8-bit: 1024 + zero point of this row (128 unless uint8 codes carry zeros)
        const uint32_t zz8 = (BITS == 8 && prm.zrow) ? (0x6400u | prm.zrow[wrow]) * 0x00010001u : 0x64806480u;
        const float zf8 = 8388608.0f + (float)((BITS == 8 && prm.zrow) ? prm.zrow[wrow] : 128u);
        // uint4: the unit's staged group scales (every converter warp waits for
        // every unit's buffer, so that its parity waits stay exact)
        const uint8_t* stg = sS + (ui & 1) * kStageBytes;
        // this row's staged scales and zero points (row srow of the tile)
        const uint16_t* srow16 = reinterpret_cast<const uint16_t*>(stg) + srow * prm.G;
        const uint8_t* zrow8 = stg + 256 * prm.G + (srow >> 1) * prm.G;
        const int zsh = 4 * (srow & 1);
        if (BITS == 4 && prm.stage) {
          ok = warp_wait(&ctl->fullS[ui & 1], (ui >> 1) & 1, ctl, prm.status, lane);
          if (!ok) break;
        }
        for (int ks = ks0; ks < ks1; ks += kGA, ++st) {
          const int nk = min(kGA, ks1 - ks);
          if (st % kConvGroups != grp) continue;
          const int d = st % ND;  // tensor-memory A stage and activation slot
          const int v = st % NV;  // their barriers
          for (int j = 0; j < nk && ok; ++j, ++lit) {
            const int sa = grp * NAG + lit % NAG;
            uint32_t zz[NCH], ss[NCH];  // uint4: per 32-K chunk, issued before the tile wait
            if constexpr (BITS == 4) {
              if (prm.stage) {
                // chunk c of this thread's part of the 256-K stage lies in group
                // g0 + (32 c >> log2 gs): one staged lookup per distinct group
                // (gs is a power of two, at least 32)
                const int g0 = ((ks + j) * kEntryK + khalf * 32 * NCH) >> prm.gs_log2;
                const int csh = prm.gs_log2 - 5;  // chunks per group = 2^csh
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                  if ((c & ((1 << csh) - 1)) == 0) {
                    const int g = g0 + (c >> csh);
                    uint32_t z = 8, sb = 0;  // past the row's end: scale 0
                    if (g < prm.G) {
                      sb = srow16[g];
                      if (prm.has_zp) z = (zrow8[g] >> zsh) & 15u;
                    }
                    zz[c] = (0x6400u | z) * 0x00010001u;
                    ss[c] = sb * 0x00010001u;
                  } else {
                    zz[c] = zz[c - 1];
                    ss[c] = ss[c - 1];
                  }
                }
              } else {
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                  group_words(prm, wrow, (ks + j) * kEntryK + 32 * (khalf * NCH + c), zz[c], ss[c]);
              }
            }
            ok = warp_wait(&ctl->fullA[sa], (lit / NAG) & 1, ctl, prm.status, lane);
            if (!ok) break;
            const uint8_t* row = sA + sa * kABytes + srow * 128;
            // x[c] holds chunk khalf * NCH + ((c + rot) % NCH) of the row
            uint4 x[NCH];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
              x[c] = ld_chunk(row, (uint32_t)(khalf * NCH + ((c + rot) & (NCH - 1))), sw);
            if (j == 0) {
              // the MMAs that last read this tensor-memory stage (step st - ND)
              // must be done
              if (st >= ND) {
                ok = warp_wait(&ctl->stepfree[(st - ND) % NV], ((st - ND) / NV) & 1, ctl,
                               prm.status, lane);
                if (!ok) break;
              }
              tc_fence_after();
            }
            const uint32_t tbase = tmem + tcol + d * kAColsPerStep + j * kEntryCols + khalf * (kEntryCols / NH);
            if constexpr (BITS == 8) {
              // the stage's codes as 16-bit words (bf16 or f16), into tensor memory
              auto conv8 = [&](auto bf) {
                constexpr bool kB = decltype(bf)::value;
#pragma unroll
                for (int h = 0; h < NCH / 4; ++h) {
                  uint32_t words[32];
#pragma unroll
                  for (int c = 0; c < 4; ++c) {
                    // chunk 4h + c of this part sits in x[4h + c] (rot 0) or
                    // x[(4h + c + NCH / 2) % NCH] (rotated)
                    const int cl = 4 * h + c;
                    const uint4 cv = sel4(rt, x[(cl + NCH / 2) & (NCH - 1)], x[cl]);
                    if constexpr (kB) convert16_bf16(cv, prm.xmask, zf8, &words[c * 8]);
                    else convert16(cv, prm.xmask, zz8, &words[c * 8]);
                  }
                  tmem_st32(tbase + h * 32, words);
                }
              };
              conv8(std::integral_constant<bool, kBf16M>{});
            } else {
#pragma unroll
              for (int h = 0; h < NCH / 2; ++h) {
                uint32_t words[32];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                  const int c = 2 * h + c2;  // chunk of this part: 32 codes
                  const uint4 v = sel4(rt, x[(c + NCH / 2) & (NCH - 1)], x[c]);
                  uint4x8_to_f16(v.x, zz[c], ss[c], &words[c2 * 16 + 0]);
                  uint4x8_to_f16(v.y, zz[c], ss[c], &words[c2 * 16 + 4]);
                  uint4x8_to_f16(v.z, zz[c], ss[c], &words[c2 * 16 + 8]);
                  uint4x8_to_f16(v.w, zz[c], ss[c], &words[c2 * 16 + 12]);
                }
                tmem_st32(tbase + h * 32, words);
              }
            }
            // The slot goes back only now that the loaded registers have been
            // consumed: a shared-memory load that has issued may still be
            // reading, and the next fill of the slot (TMA) would overtake it.
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->emptyA[sa]);
          }
          if (!ok) break;
          // the step's activations (exact: the MMAs that read this slot's
          // previous fill are done, so its barrier is at most this phase behind)
          ok = warp_wait(&ctl->fullB[v], (st / NV) & 1, ctl, prm.status, lane);
          if (!ok) break;
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->afull[v]);
        }
        if (!ok) break;
        if (BITS == 4 && prm.stage) {  // done with the unit's staged scales
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->emptyS[ui & 1]);
        }
      }
    });
  } else {
    // ---------------------------------------------------- epilogue ----
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const bool odd = (lane & 1) != 0;
    // accumulator columns per tcgen05.ld (two issuers: two halves are
    // loaded); the gate/up epilogue takes 16 at a time in every tile shape:
    // its unrolled SiLU body is then half the code, and the first unit's
    // epilogue -- which runs that code cold -- ends sooner (fine-grained
    // layer at T=512, one-launch kernel: 98.3 -> 91.6 us)
    constexpr int CH = C::kNI == 2 ? 16 : (BN < 32 ? BN : 32);
    mq::pdl_wait();
    int t = 0;
    int est = 0;  // schedule index of the unit's first MMA step
    bool ok = true;
    phases([&](auto ph_tag, const TcParams& prm, const CUtensorMap& mA, const CUtensorMap& mB,
               const int4* ul, int tot, int u0) {
      constexpr int M = decltype(ph_tag)::value;
      constexpr int CHM = M == 1 ? 16 : CH;
      constexpr bool kBf16M = M == 2 && (BITS == 8 || SYNC) && !F16D;
      for (int u = u0, ui = 0; u < tot && ok; u += gridDim.x, ++t, ++ui) {
        const Unit w = cta_unit<BN>(prm, ul, ui, u, kUL);
        const int buf = t % C::kAccBufs;
        const int nsteps = ((w.split + 1) * prm.ksteps / prm.splits - w.split * prm.ksteps / prm.splits + kGA - 1) / kGA;
        // two issuers: both halves hold partial sums when the unit has two or
        // more steps; with one step only half (first step % 2) was written
        const bool both = C::kNI == 2 && nsteps >= 2;
        const int half0 = (C::kNI == 2 && !both) ? (est & 1) : 0;
        est += nsteps;
        // Per-column values of the tile, loaded while its MMAs still run (a
        // unit of a few MMA steps would otherwise wait on these dependent
        // loads): column i * 32 + lane in element i.  M 1: the activation
        // row scale; M 2: the token-slot (S for padding) and its factor
        // (activation row scale x router weight).
        constexpr int NP = (BN + 31) / 32;
        float colf[NP];
        int colslot[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          const int cc = i * 32 + lane;
          colf[i] = M == 1 ? 1.0f : 0.0f;
          colslot[i] = prm.S;
          if (cc < w.n) {
            if (M == 1) colf[i] = prm.xinv[w.row0 + cc];
            if (M == 2 || prm.rw_on_input) colslot[i] = prm.sorted[w.row0 + cc];
          }
        }
        if (M == 1 && prm.rw_on_input) {
          // router weight on the input: W13 . (w x) = w (W13 . x), applied to
          // the float32 accumulators with the row scale
#pragma unroll
          for (int i = 0; i < NP; ++i) colf[i] *= colslot[i] < prm.S ? prm.topk_w[colslot[i]] : 0.0f;
        }
        if (M == 2) {
#pragma unroll
          for (int i = 0; i < NP; ++i)
            if (colslot[i] < prm.S)
              colf[i] = (kBf16M ? 1.0f : prm.xinv[w.row0 + i * 32 + lane]) *
                        (prm.rw_on_input ? 1.0f : prm.topk_w[colslot[i]]);
        }
        // this thread's per-channel scale (8-bit), likewise loaded before the wait
        float sc_pre = 1.0f;
        if (BITS == 8) {
          int64_t srow_g;
          if (M == 1)
            srow_g = (int64_t)w.e * 2 * prm.I + (odd ? prm.I : 0) + w.mt * 64 + q * 16 + (lane >> 1);
          else
            srow_g = (int64_t)w.e * prm.H + w.mt * kTileM + r;
          sc_pre = load_scale(prm, prm.scale_per_tensor ? w.e : srow_g);
        }
        if (!warp_wait_sleepy(&ctl->accfull[buf], (t / C::kAccBufs) & 1, ctl, prm.status, lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (buf * C::kNI + half0) * BN;
        // accumulator columns [c0, c0 + W) into v: half 0 (+ half 1), in that order
        auto load_acc = [&](auto wtag, int c0, auto& v) {
          constexpr int W = decltype(wtag)::value;
          tmem_ld_cols_sync<W>(taddr + c0, v);
          if (C::kNI == 2 && both) {
            uint32_t v2[W];
            tmem_ld_cols_sync<W>(taddr + BN + c0, v2);
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v2[j]));
          }
        };
        if (M == 1) {
          // lanes (2i, 2i+1) hold gate row i and up row i; per pair of
          // columns (jj, jj + HALF) the even lane finishes column jj and the
          // odd lane column jj + HALF, after one exchange
          // int8: per-channel scale here; uint4: group scales were applied to A
          const float sc = sc_pre;
          // uint4 runs the down GEMM in the K order [0,4,1,5,2,6,3,7] per octet
          const int col = w.mt * 64 + q * 16 + (BITS == 8 ? (lane >> 1) : permute_octet(lane >> 1));
          // xv: element c0 / 32 of colf (column c0 + cj on lane (c0 & 31) + cj)
          auto body = [&](auto wtag, int c0, float xv) {
            constexpr int W = decltype(wtag)::value;
            constexpr int HW = W / 2;
            uint32_t v[W];
            load_acc(wtag, c0, v);
#pragma unroll
            for (int jj = 0; jj < HW; ++jj) {
              const float lo = __uint_as_float(v[jj]) * sc;       // own row, column jj
              const float hi = __uint_as_float(v[jj + HW]) * sc;  // own row, column jj + HW
              const float got = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
              const int cj = odd ? jj + HW : jj;
              const float xs = __shfl_sync(0xffffffffu, xv, (c0 & 31) + cj);
              const float g = (odd ? got : lo) * xs;
              const float up = (odd ? hi : got) * xs;
              const float a = __fdividef(g * up, 1.0f + __expf(-g));  // silu(g) * up
              prm.act[(int64_t)(w.row0 + c0 + cj) * prm.I + col] = __float2bfloat16_rn(a);
            }
          };
          int c0 = 0;
          for (; c0 + CHM <= w.n; c0 += CHM) {
            float xv = colf[0];
#pragma unroll
            for (int i = 1; i < NP; ++i)
              if ((c0 >> 5) == i) xv = colf[i];
            body(IC<CHM>{}, c0, xv);
          }
          if (CHM > 16 && c0 < w.n) {  // n is a multiple of 16
            float xv = colf[0];
#pragma unroll
            for (int i = 1; i < NP; ++i)
              if ((c0 >> 5) == i) xv = colf[i];
            body(IC<16>{}, c0, xv);
          }
        } else {
          const int h = w.mt * kTileM + r;
          const float sc = sc_pre;
          float* yp = prm.ypart + (int64_t)w.split * prm.S * prm.H;
          // slot, f: element c0 / 32 of colslot, colf (column c0 + jj on lane (c0 & 31) + jj)
          auto body = [&](auto wtag, int c0, int slot, float f) {
            constexpr int W = decltype(wtag)::value;
            uint32_t v[W];
            load_acc(wtag, c0, v);
#pragma unroll
            for (int jj = 0; jj < W; ++jj) {
              const int sj = __shfl_sync(0xffffffffu, slot, (c0 & 31) + jj);
              const float fj = __shfl_sync(0xffffffffu, f, (c0 & 31) + jj);
              if (sj < prm.S) yp[(int64_t)sj * prm.H + h] = __uint_as_float(v[jj]) * sc * fj;
            }
          };
          int c0 = 0;
          for (; c0 + CHM <= w.n; c0 += CHM) {
            int sl = colslot[0];
            float fc = colf[0];
#pragma unroll
            for (int i = 1; i < NP; ++i)
              if ((c0 >> 5) == i) {
                sl = colslot[i];
                fc = colf[i];
              }
            body(IC<CHM>{}, c0, sl, fc);
          }
          if (CHM > 16 && c0 < w.n) {  // n is a multiple of 16
            int sl = colslot[0];
            float fc = colf[0];
#pragma unroll
            for (int i = 1; i < NP; ++i)
              if ((c0 >> 5) == i) {
                sl = colslot[i];
                fc = colf[i];
              }
            body(IC<16>{}, c0, sl, fc);
          }
        }
        // fused layer: this warp's act columns of the token tile are stored
        if constexpr (FUSED && M == 1) dep_signal(prm.dep + w.ch, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->accempty[buf]);
      }
    });
  }

  tc_fence_before();
  __syncthreads();
  if (!SYNC && warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One expert GEMM (MODE 1 gate/up, 2 down).  F16D: the 8-bit down GEMM on
// f16 operands (act converted to f16 in place beforehand).
template <int MODE, int BITS, int BN, bool SYNC, bool F16D = false>
__global__ void __launch_bounds__(CfgOf<MODE, BITS, BN, SYNC>::kThreads, 1)
    moe_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ TcParams p) {
  gemm_body<MODE, BITS, BN, SYNC, false, F16D>(tmA, tmB, p, tmA, tmB, p);
}

// Both expert GEMMs of an 8-bit layer in one launch (FUSED above).
template <int BN>
__global__ void __launch_bounds__(CfgOf<1, 8, BN, false>::kThreads, 1)
    moe_layer_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tmA2,
                 const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ TcParams p2) {
  gemm_body<1, 8, BN, false, true, false>(tmA, tmB, p, tmA2, tmB2, p2);
}

// Rows of x gathered into expert-sorted order as f16, each scaled by a power
// of two 2^e chosen so that the row's largest magnitude lands in
// [2^14, 2^15): bf16 -> f16 is then exact except for elements below 2^-28
// of the row maximum (f16 subnormals).  xinv[p] = 2^-e undoes it in the
// epilogue.  Padding rows are zeros.
// 8 activations of one uint4 (bf16 or f16), times wmul.
__device__ __forceinline__ void act8(const uint4& v, bool f16, float wmul, float* f) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (f16) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&u[j]));
      f[2 * j] = t.x * wmul;
      f[2 * j + 1] = t.y * wmul;
    } else {
      f[2 * j] = mq::bf16_lo(u[j]) * wmul;
      f[2 * j + 1] = mq::bf16_hi(u[j]) * wmul;
    }
  }
}

// x is bf16, or f16 (act_f16).
template <bool PERM>
__global__ void __launch_bounds__(128) gather_rows_f16(const void* __restrict__ xv,
                                                       const int32_t* __restrict__ sorted,
                                                       const int32_t* __restrict__ num_padded,
                                                       int k, int S, int H, int act_f16,
                                                       __half* __restrict__ xs,
                                                       float* __restrict__ xinv) {
  __shared__ float wmax[4];
  const int p = blockIdx.x;
  mq::pdl_wait();  // sorted and num_padded come from the previous kernel
  mq::pdl_trigger();
  if (p >= *num_padded) return;
  const int s = sorted[p];
  uint4* dst = reinterpret_cast<uint4*>(xs + (int64_t)p * H);  // one K octet per uint4
  const int n = H / 8;
  if (s >= S) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) xinv[p] = 1.0f;
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xv) + (int64_t)(s / k) * H);
  const bool f16 = act_f16 != 0;
  const float wmul = 1.0f;
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    float f[8];
    act8(src[i], f16, wmul, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  int ex = 0;
  if (m > 0.0f) frexpf(m, &ex);  // m = f * 2^ex, f in [0.5, 1)
  int e = 15 - ex;               // m * 2^e in [2^14, 2^15)
  e = max(-120, min(120, e));
  const float scale = ldexpf(1.0f, e);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    float f[8];
    act8(src[i], f16, wmul, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] *= scale;
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // natural order: pair (2j, 2j+1); octet order [0,4,1,5,2,6,3,7]: pair (j, j+4)
      const __half2 h = PERM ? __floats2half2_rn(f[j], f[j + 4]) : __floats2half2_rn(f[2 * j], f[2 * j + 1]);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) xinv[p] = ldexpf(1.0f, -e);
}

// uint4 weights (f16 down-GEMM operands): act rows [0, num_padded)
// converted in place from bf16 to f16, each row scaled by a power of two 2^e
// so that its largest magnitude lands in [2^14, 2^15) (exact, as in
// gather_rows_f16); xinv[p] = 2^-e.
__global__ void __launch_bounds__(256) act_rows_to_f16(uint16_t* act, const int32_t* num_padded,
                                                       int I, float* __restrict__ xinv) {
  __shared__ float wmax[8];
  const int p = blockIdx.x;
  mq::pdl_wait();  // act comes from the previous kernel
  mq::pdl_trigger();
  if (p >= *num_padded) return;
  uint4* row = reinterpret_cast<uint4*>(act + (int64_t)p * I);
  const int n = I / 8;
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint4 v = row[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(mq::bf16_lo(u[j])), fabsf(mq::bf16_hi(u[j]))));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) m = fmaxf(m, wmax[w]);
  int ex = 0;
  if (m > 0.0f) frexpf(m, &ex);
  int e = 15 - ex;
  e = max(-120, min(120, e));
  const float scale = ldexpf(1.0f, e);
  // each thread rewrites exactly the vectors it read: in place is safe
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint4 v = row[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h = __floats2half2_rn(mq::bf16_lo(u[j]) * scale, mq::bf16_hi(u[j]) * scale);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    row[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) xinv[p] = ldexpf(1.0f, -e);
}

// out[t, :] = sum over valid slots j and K splits of ypart[split, t*k + j, :],
// in the order (j, split).  Without K splits (prefill plans) the partial
// sums are read once from HBM: eight slots' loads are all issued before
// their sums, so that enough bytes are in flight, with streaming cache hints.
// With K splits (decode plans, a few MB that the down GEMM just wrote to L2)
// a plain loop over the slots is faster.
__global__ void __launch_bounds__(256) combine_splits(const float* __restrict__ ypart,
                                                      const int32_t* __restrict__ ids, int T,
                                                      int k, int E, int H, int splits,
                                                      int out_f16, void* __restrict__ out) {
  constexpr int kBatch = 8;
  const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int H4 = H / 4;
  mq::pdl_wait();  // ypart comes from the previous kernel
  mq::pdl_trigger();
  if (i4 >= (int64_t)T * H4) return;
  const int t = (int)(i4 / H4);
  const int c = (int)(i4 % H4) * 4;
  const int64_t S = (int64_t)T * k;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (splits == 1) {
    for (int j0 = 0; j0 < k; j0 += kBatch) {
      float4 v[kBatch];
      bool ok[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int64_t s = (int64_t)t * k + j0 + b;
        ok[b] = false;
        if (j0 + b < k) {
          const int e = ids[s];
          ok[b] = e >= 0 && e < E;
          if (ok[b]) v[b] = __ldcs(reinterpret_cast<const float4*>(ypart + s * H + c));
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (ok[b]) {
          acc.x += v[b].x;
          acc.y += v[b].y;
          acc.z += v[b].z;
          acc.w += v[b].w;
        }
      }
    }
  } else {
    for (int j = 0; j < k; ++j) {
      const int64_t s = (int64_t)t * k + j;
      const int e = ids[s];
      if (e < 0 || e >= E) continue;
      for (int sp = 0; sp < splits; ++sp) {
        const float4 v = *reinterpret_cast<const float4*>(ypart + (sp * S + s) * H + c);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
  }
  uint2 o;
  if (out_f16) {
    __half2 lo = __floats2half2_rn(acc.x, acc.y);
    __half2 hi = __floats2half2_rn(acc.z, acc.w);
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
  }
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + (int64_t)t * H + c) = o;
}

// ------------------------------------------------------------ host side --
int g_num_sms = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// Tensor map of `rank` dims; dims[0] is innermost, strides are in bytes for
// dims 1..rank-1.
cudaError_t make_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                     const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                     CUtensorMapSwizzle sw) {
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// At least 120 KB so that only one CTA fits on an SM: each CTA allocates all
// 512 tensor-memory columns.
template <int MODE, int BITS, int BN, bool SYNC>
constexpr size_t smem_for() {
  using C = CfgOf<MODE, BITS, BN, SYNC>;
  const size_t part = (size_t)partial_bytes<SYNC, BN>();
  const size_t need = 1024 + (size_t)C::kAStagesSmem * kABytes + (size_t)C::kBSlots * C::kBBytes +
                      part + sizeof(SharedCtl) + kUnitList * sizeof(int4) +
                      (size_t)stage_bytes<BITS>();
  return need < 120 * 1024 ? 120 * 1024 : need;
}

template <int MODE, int BITS, int BN, bool SYNC, bool F16D = false>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const TcParams& p,
                        int max_units, cudaStream_t st) {
  constexpr size_t smem = smem_for<MODE, BITS, BN, SYNC>();
  static_assert(smem <= 227 * 1024, "shared memory");
  auto kern = moe_gemm_tc<MODE, BITS, BN, SYNC, F16D>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int sms = tc_num_sms();
  const int grid = max_units < sms ? max_units : sms;
  if (grid <= 0) return cudaSuccess;
  err = launch_pdl(kern, dim3(grid), dim3(CfgOf<MODE, BITS, BN, SYNC>::kThreads), smem, st, ta,
                   tb, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int MODE, int BITS>
cudaError_t launch_gemm_bn(int bn, bool sync, const CUtensorMap& ta, const CUtensorMap& tb,
                           const TcParams& p, int max_units, cudaStream_t st) {
  if (sync) {  // warp-MMA mode: 16-row tiles, and 32-row tiles for 8-bit codes
    if (bn == 16) return launch_gemm<MODE, BITS, 16, true>(ta, tb, p, max_units, st);
    if constexpr (BITS == 8)
      if (bn == 32) return launch_gemm<MODE, BITS, 32, true>(ta, tb, p, max_units, st);
    return cudaErrorInvalidValue;
  }
  if constexpr (MODE == 2 && BITS == 8) {
    if (p.down_f16) {  // f16 operands: 16- and 32-row tiles (batches of 8-64 tokens)
      if (bn == 16) return launch_gemm<2, 8, 16, false, true>(ta, tb, p, max_units, st);
      if (bn == 32) return launch_gemm<2, 8, 32, false, true>(ta, tb, p, max_units, st);
      return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return launch_gemm<MODE, BITS, 16, false>(ta, tb, p, max_units, st);
    case 32: return launch_gemm<MODE, BITS, 32, false>(ta, tb, p, max_units, st);
    case 64: return launch_gemm<MODE, BITS, 64, false>(ta, tb, p, max_units, st);
    case 128: return launch_gemm<MODE, BITS, 128, false>(ta, tb, p, max_units, st);
    default: return cudaErrorInvalidValue;
  }
}

// K elements per 16 KB weight stage, and stages per row of length K.
inline int entry_k(int bits) { return bits == 8 ? 128 : 256; }
inline int entries(int K, int bits) { return (K + entry_k(bits) - 1) / entry_k(bits); }

}  // namespace

TcPlan tc_plan(int T, int H, int I, int E, int k, int bits) {
  TcPlan pl;
  pl.sync1 = pl.sync2 = false;
  pl.layer = false;
  pl.f16down = false;
  const int64_t S = (int64_t)T * k;
  // Token-slots per tile at most (the MMA's N).  A tile is cut from one
  // expert's segment with the rows it has, so a larger bound costs shared
  // memory for the activation ring (a shallower weight ring) and activation
  // traffic, while a smaller one streams an expert's weights once per tile
  // (the tiles of one expert run side by side, so the second pass mostly
  // hits L2).  Up to 32 tokens: 16 (32 from 17 tokens in 8-bit layers of
  // many experts, below).  Up to 64 tokens: 32 for layers of a
  // few large experts, whose loads are near-uniform (measured on the
  // Mixtral-shaped layer, E=8, at T=64: gate/up 186.3 us with 64-row tiles,
  // 178.3 us with 32-row tiles and two MMA issuers), 64 for layers of many
  // small experts, where a few experts take most tokens (fine-grained E=128
  // with Zipf routing at T=64: step 66.9 us with 64-row tiles, 69.2 us with
  // 32-row ones).  Beyond 64 tokens, 128.
  // 8-bit layers of many experts take 32-row tiles from 17 tokens (Zipf
  // routing puts most tokens on a few experts: fine-grained T=32 step 51.5
  // -> 46.4 us; W4A16 and the Mixtral-shaped layer lose 0.3-1 % with them).
  int bn = T > 64 ? 128
                  : (T > 32 ? (E <= 16 ? 32 : 64) : (T > 16 && E > 16 && bits == 8 ? 32 : 16));
  // uint4 layers of more than 16 experts keep 16- and 32-row tiles while the
  // mean number of slots per expert stays below 10 and 28.  A uint4 stage
  // costs as many MMAs as an int8 step for half the bytes, and the small
  // tiles run the deepest pipeline: two issuers, two accumulator buffers,
  // three tensor-memory stages.  W4A16 E=64, k=6, uniform routing, step in
  // us with the L2 flushed, tiles 16 / 32 / default:
  // T=64 152 / 158 / 161 (64-row), T=128 161 / 159 / 186, T=192 231 / 162 /
  // 189, T=256 268 / 171 / 191, T=384 - / 253 / 197 (128-row).
  if (bits == 4 && E > 16) {
    if (S <= 10 * (int64_t)E) bn = 16;
    else if (S <= 28 * (int64_t)E) bn = 32;
  }
  pl.bn = bn;
  // K splits of the down GEMM.  Decode batches: the split count whose units
  // (live experts x H / 128 x splits) fill the SMs most evenly (dec_splits;
  // Mixtral-shaped T=1: 7 splits, 448 units, 2.95 waves, against 8 splits'
  // 3.37 waves).  Larger batches: enough units (about 600, four per SM) to
  // keep every SM streaming, each split keeping at least two MMA steps.
  const int64_t live = S < E ? S : E;
  const int64_t blocks = live > S / bn ? live : S / bn;
  const int mt2 = H / kTileM;
  const int steps2 = (I + 255) / 256;
  int splits = 1;
  if (T <= 64) {
    splits = dec_splits(T, H, I, E, k, bits);
  } else {
    while (splits < 8 && blocks * mt2 * splits < 600 && steps2 / (splits * 2) >= 2) splits *= 2;
  }
  pl.splits = splits;
  return pl;
}

int tc_num_sms() {
  if (g_num_sms == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      g_num_sms = n;
  }
  return g_num_sms > 0 ? g_num_sms : 148;
}

cudaError_t launch_gather_rows(const MoeArgs& a, void* xs, float* xinv, cudaStream_t st) {
  if (a.cap == 0) return cudaSuccess;
  const cudaError_t err = launch_pdl(
      a.bits == 8 ? gather_rows_f16<false> : gather_rows_f16<true>, dim3((unsigned)a.cap),
      dim3(128), 0, st, a.x, a.sorted, a.num_padded, a.k, a.T * a.k, a.H,
      (a.flags & MQ_FWD_ACT_F16) ? 1 : 0, static_cast<__half*>(xs), xinv);
  return err != cudaSuccess ? err : cudaGetLastError();
}

namespace {

void common_params(TcParams& p, const MoeArgs& a) {
  p.H = a.H; p.I = a.I; p.E = a.E; p.k = a.k; p.S = a.T * a.k;
  p.sorted = a.sorted; p.offsets = a.offsets;
  p.chunk_expert = a.chunk_expert; p.chunk_start = a.chunk_start;
  p.counts = a.counts;
  p.topk_w = a.topk_w;
  p.status = a.status;
  p.gs = a.bits == 8 ? 0 : a.group_size;
  p.has_zp = a.has_zp;
  p.stage = 0;
  p.gs_log2 = 0;
  for (int g = p.gs; g > 1; g >>= 1) ++p.gs_log2;
  p.act = nullptr;
  p.ypart = nullptr;
  p.scale_kind = (a.flags & MQ_FWD_SCALE_F16) ? 1 : (a.flags & MQ_FWD_SCALE_BF16) ? 2 : 0;
  p.scale_per_tensor = (a.flags & MQ_FWD_SCALE_PER_TENSOR) ? 1 : 0;
  p.xmask = (a.flags & MQ_FWD_W8_UINT8) ? 0u : 0x80808080u;
  p.zrow = nullptr;
  p.rw_on_input = (a.flags & MQ_FWD_ROUTER_WEIGHT_ON_INPUT) ? 1 : 0;
  p.xinv = nullptr;
  p.dep = nullptr;
  p.dep_target = 0;
  p.down_f16 = 0;
  p.scale = nullptr;
  p.gscale = nullptr;
  p.gzero = nullptr;
  p.G = 0;
}

}  // namespace

namespace {

// Tensor maps and parameters of the gate/up GEMM; mu bounds its work units.
cudaError_t prep_gemm1(const MoeArgs& a, const TcPlan& pl, const void* xs, const float* xinv,
                       CUtensorMap& ta, CUtensorMap& tb, TcParams& p, int& mu) {
  cudaError_t err = get_encoder();
  if (err != cudaSuccess) return err;
  // weight rows in bytes: H int8 codes or H/2 bytes of packed uint4 codes
  const uint64_t rb = a.bits == 8 ? (uint64_t)a.H : (uint64_t)a.H / 2;
  {
    // w13 [E, 2, I, rb] viewed as {rb, I, 2, E}: one box = 64 gate rows + 64 up rows
    const cuuint64_t dims[4] = {rb, (cuuint64_t)a.I, 2, (cuuint64_t)a.E};
    const cuuint64_t strides[3] = {rb, (cuuint64_t)a.I * rb, (cuuint64_t)2 * a.I * rb};
    const cuuint32_t box[4] = {128, 64, 2, 1};
    err = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, a.w13, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.H, (cuuint64_t)a.cap};
    const cuuint64_t strides[1] = {(cuuint64_t)a.H * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)pl.bn};
    err = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xs, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }
  common_params(p, a);
  p.ksteps = entries(a.H, a.bits);
  p.MT = a.I / 64;
  p.splits = 1;
  if (a.bits == 8) {
    p.scale = a.s13;
    p.zrow = a.has_zp ? a.z13 : nullptr;
  } else {
    p.gscale = static_cast<const __half*>(a.s13);
    p.gzero = a.z13;
    p.G = a.H / a.group_size;
    p.stage = stage_fits(p.G) ? 1 : 0;
  }
  p.act = a.act;
  p.xinv = xinv;
  const int64_t units = (a.cap / a.bm) * (int64_t)p.MT;  // token tiles <= 16-slot blocks
  mu = (int)(units < (1 << 30) ? units : (1 << 30));
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm1_tc(const MoeArgs& a, const TcPlan& pl, const void* xs,
                            const float* xinv, cudaStream_t st) {
  CUtensorMap ta, tb;
  TcParams p;
  int mu = 0;
  const cudaError_t err = prep_gemm1(a, pl, xs, xinv, ta, tb, p, mu);
  if (err != cudaSuccess) return err;
  return a.bits == 8 ? launch_gemm_bn<1, 8>(pl.bn, pl.sync1, ta, tb, p, mu, st)
                     : launch_gemm_bn<1, 4>(pl.bn, pl.sync1, ta, tb, p, mu, st);
}

cudaError_t launch_act_to_f16(const MoeArgs& a, float* act_inv, cudaStream_t st) {
  if (a.cap == 0) return cudaSuccess;
  const cudaError_t err =
      launch_pdl(act_rows_to_f16, dim3((unsigned)a.cap), dim3(256), 0, st,
                 reinterpret_cast<uint16_t*>(a.act), a.num_padded, a.I, act_inv);
  return err != cudaSuccess ? err : cudaGetLastError();
}

namespace {

// Tensor maps and parameters of the down GEMM; mu bounds its work units.
cudaError_t prep_gemm2(const MoeArgs& a, const TcPlan& pl, const float* act_inv, float* ypart,
                       CUtensorMap& ta, CUtensorMap& tb, TcParams& p, int& mu) {
  cudaError_t err = get_encoder();
  if (err != cudaSuccess) return err;
  const uint64_t rb = a.bits == 8 ? (uint64_t)a.I : (uint64_t)a.I / 2;
  {
    const cuuint64_t dims[2] = {rb, (cuuint64_t)a.E * a.H};
    const cuuint64_t strides[1] = {rb};
    const cuuint32_t box[2] = {128, kTileM};
    err = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.w2, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.I, (cuuint64_t)a.cap};
    const cuuint64_t strides[1] = {(cuuint64_t)a.I * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)pl.bn};
    // act: bf16 as written by the gate/up GEMM (8-bit, and uint4 in warp-MMA
    // mode), or f16 after the in-place conversion (uint4, tensor cores)
    err = make_map(&tb, ((a.bits == 8 && !pl.f16down) || pl.sync2) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, a.act, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
  }
  common_params(p, a);
  p.ksteps = entries(a.I, a.bits);
  p.MT = a.H / kTileM;
  p.splits = pl.splits;
  if (a.bits == 8) {
    p.scale = a.s2;
    p.zrow = a.has_zp ? a.z2 : nullptr;
  } else {
    p.gscale = static_cast<const __half*>(a.s2);
    p.gzero = a.z2;
    p.G = a.I / a.group_size;
    p.stage = stage_fits(p.G) ? 1 : 0;
  }
  p.ypart = ypart;
  p.xinv = act_inv;
  p.down_f16 = (a.bits == 8 && pl.f16down && !pl.sync2) ? 1 : 0;
  const int64_t units = (a.cap / a.bm) * (int64_t)p.MT * p.splits;
  mu = (int)(units < (1 << 30) ? units : (1 << 30));
  return cudaSuccess;
}

template <int BN>
cudaError_t launch_layer(const CUtensorMap& ta, const CUtensorMap& tb, const TcParams& p,
                         const CUtensorMap& ta2, const CUtensorMap& tb2, const TcParams& p2,
                         int max_units, cudaStream_t st) {
  constexpr size_t smem = smem_for<1, 8, BN, false>();
  static_assert(smem <= 227 * 1024, "shared memory");
  auto kern = moe_layer_tc<BN>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // at most one CTA per SM (shared memory and all tensor-memory columns):
  // with grid <= SMs every CTA becomes resident, which the down units'
  // waits for other CTAs' gate/up units rely on
  const int sms = tc_num_sms();
  const int grid = max_units < sms ? max_units : sms;
  if (grid <= 0) return cudaSuccess;
  err = launch_pdl(kern, dim3(grid), dim3(CfgOf<1, 8, BN, false>::kThreads), smem, st, ta, tb, p,
                   ta2, tb2, p2);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm2_tc(const MoeArgs& a, const TcPlan& pl, const float* act_inv,
                            float* ypart, cudaStream_t st) {
  CUtensorMap ta, tb;
  TcParams p;
  int mu = 0;
  const cudaError_t err = prep_gemm2(a, pl, act_inv, ypart, ta, tb, p, mu);
  if (err != cudaSuccess) return err;
  return a.bits == 8 ? launch_gemm_bn<2, 8>(pl.bn, pl.sync2, ta, tb, p, mu, st)
                     : launch_gemm_bn<2, 4>(pl.bn, pl.sync2, ta, tb, p, mu, st);
}

namespace {
std::atomic<int> g_layer_wait_extra{0};
}  // namespace

int set_layer_wait_extra(int extra) { return g_layer_wait_extra.exchange(extra); }

cudaError_t launch_layer_tc(const MoeArgs& a, const TcPlan& pl, const void* xs,
                            const float* xinv, float* ypart, cudaStream_t st) {
  if (a.bits != 8 || pl.sync1 || pl.sync2 || pl.f16down || a.dep == nullptr)
    return cudaErrorInvalidValue;
  CUtensorMap ta, tb, ta2, tb2;
  TcParams p, p2;
  int mu1 = 0, mu2 = 0;
  cudaError_t err = prep_gemm1(a, pl, xs, xinv, ta, tb, p, mu1);
  if (err != cudaSuccess) return err;
  err = prep_gemm2(a, pl, nullptr, ypart, ta2, tb2, p2, mu2);
  if (err != cudaSuccess) return err;
  // each gate/up unit's 4 epilogue warps count once per token tile
  p.dep = a.dep;
  p2.dep = a.dep;
  p2.dep_target = 4 * p.MT + g_layer_wait_extra.load();
  const int64_t mu = (int64_t)mu1 + mu2;
  const int m = (int)(mu < (1 << 30) ? mu : (1 << 30));
  switch (pl.bn) {
    case 16: return launch_layer<16>(ta, tb, p, ta2, tb2, p2, m, st);
    case 32: return launch_layer<32>(ta, tb, p, ta2, tb2, p2, m, st);
    case 64: return launch_layer<64>(ta, tb, p, ta2, tb2, p2, m, st);
    case 128: return launch_layer<128>(ta, tb, p, ta2, tb2, p2, m, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_splits(const MoeArgs& a, const float* ypart, int splits,
                                  cudaStream_t st) {
  const int64_t n = (int64_t)a.T * (a.H / 4);
  if (n == 0) return cudaSuccess;
  const cudaError_t err =
      launch_pdl(combine_splits, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, ypart,
                 a.topk_ids, a.T, a.k, a.E, a.H, splits, (a.flags & MQ_FWD_ACT_F16) ? 1 : 0, a.out);
  return err != cudaSuccess ? err : cudaGetLastError();
}

bool dec_supported(int bits, int group_size, int H, int I) {
  if (bits == 8) return true;
  return bits == 4 && (group_size == 128 || group_size == 256) && H % 128 == 0 && I % 128 == 0;
}

int dec_splits(int T, int H, int I, int E, int k, int bits) {
  // K splits of the down GEMM at decode sizes: the split count whose units
  // (live experts x H / 128 x splits) fill the SMs most evenly, the last
  // wave nearly full; fewer splits win near-ties (each adds partial sums to
  // write and combine), and a unit keeps at least 4 MMA steps (256 K each:
  // shorter units spend more on hand-off and pipeline turn-around than the
  // even waves save -- W4A16 E=64 at T=8, 6 steps: down 39 us unsplit, 53 us
  // in two).  Mixtral-shaped T=1: 7 splits, 2.95 waves (down 38.9 -> 35.3 us
  // against 8 splits' 3.37 waves).
  (void)bits;
  const int64_t S = (int64_t)T * k;
  const int64_t live = S < E ? S : E;
  const int steps = (I + 255) / 256;
  const int sms = tc_num_sms();
  int best = 1;
  double best_eff = -1.0;
  for (int sp = 1; sp <= 8; ++sp) {
    if (sp > 1 && steps / sp < 4) break;
    const int64_t units = live * (H / kTileM) * sp;
    const double waves = (double)units / (double)sms;
    const double eff = waves / std::ceil(waves) - (sp - 1) * 0.01;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = sp;
    }
  }
  return best;
}
