// C ABI of libmoeq.so: argument validation, workspace layout and launches.
// Every exported function is declared, with its contract, in include/moeq.h.
#include "common.cuh"

#include <atomic>
#include <cmath>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <vector>

#define MQ_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// ---------------------------------------------------------------------------
// Launch accounting and optional per-kernel CUDA-event timing.
// ---------------------------------------------------------------------------
std::atomic<long long> g_launches{0};
std::atomic<int> g_prof_on{0};
std::mutex g_prof_mu;
struct ProfRec {
  int slot;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
double g_prof_ms[MQ_PROF_SLOTS];
long long g_prof_n[MQ_PROF_SLOTS];

cudaEvent_t pool_event() {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Counts one kernel launch and, while profiling is on, brackets it with a
// pair of events on its stream.
struct LaunchScope {
  int slot;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  LaunchScope(int s, cudaStream_t stream) : slot(s), st(stream) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_prof_on.load(std::memory_order_relaxed)) {
      a = pool_event();
      if (a) cudaEventRecord(a, st);
    }
  }
  ~LaunchScope() {
    if (!a) return;
    cudaEvent_t b = pool_event();
    if (!b) return;
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_pending.push_back({slot, a, b});
  }
};

thread_local char g_msg[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t err, const char* what) {
  return fail(MQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device status word (one per device, in this library's module).
__device__ unsigned g_dev_status;

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Workspace layout of moe_quant_forward: align arrays (16-slot blocks) and
// the chunk table of the GEMMs' token tiles, gathered activations (f16) and
// their row scales, act (bf16, then f16 in place) and its row scales,
// split-K partial outputs (fp32).
constexpr int kAlignBlock = 16;

// Which consumers the expert GEMMs run.  With a few token-slots per expert
// the converter warps can multiply with warp-level MMAs themselves
// (TcPlan::sync1 / sync2; token tiles of 16 or 32 rows) instead of feeding
// the tcgen05.mma issuers.  That mode was the faster gate/up GEMM for 8-bit
// batches of up to 32 tokens while each converter group had one
// tensor-memory stage (Mixtral-shaped T=8: 150 vs 163 us per launch).  With
// three stages shared by two issuers, tcgen05 is faster at every size
// measured (Mixtral-shaped gate/up T=1: 56.4 vs 57.8 us, T=8: 148.6 vs
// 158.3, T=32: 161.7 vs 174.0; fine-grained T=8: 25.1 vs 26.0), so the
// default takes tcgen05 and the warp-MMA mode runs when forced
// (MQ_FWD_PATH_DECODE).  Each mma.sync takes about 8 cycles of its
// scheduler's issue that dequant instructions cannot overlap.

// The one-launch layer by default where it measured faster than two
// launches (fine-grained E=128, k=8, H=2048, I=768 with Zipf routing, step
// with the L2 flushed: T=128 83.0 -> 77.2 us, T=512 132.4 -> 124.1 us): layers
// of many small experts with 128-row token tiles, where each GEMM alone runs
// few MMA steps per SM.  At T=64 (64-row tiles) both take 59-60 us, at
// T=4096 both 574 us; Mixtral-shaped layers (E=8) lose with it (T=64: 291 ->
// 305 us, as 64-row tiles replace the 32-row ones).  For one or two tokens
// in layers of a few experts the down GEMM's start-up hides behind the
// gate/up GEMM's tail: Mixtral-shaped T=1 step 79.6 -> 76.5 us (L2 flushed:
// 90.7 -> 85.3), T=2 80.1 -> 77.7 us; from T=4 on two launches are as fast
// or faster.
bool layer_default(int T, int E) { return E > 16 ? (T > 64 && T <= 2048) : T <= 2; }

TcPlan fwd_plan(int T, int H, int I, int E, int k, int bits, int group_size, unsigned flags) {
  TcPlan pl = tc_plan(T, H, I, E, k, bits);
  const bool ok = dec_supported(bits, group_size, H, I);
  if (flags & MQ_FWD_PATH_TENSOR_CORE) return pl;
  if (flags & MQ_FWD_PATH_LAYER) {  // 8-bit only (checked by the caller)
    pl.layer = true;
    return pl;
  }
  if (flags & MQ_FWD_PATH_DECODE) {
    if (!ok) return pl;
    pl.sync1 = pl.sync2 = true;
    // an expert receives at most one slot per token: up to 16 tokens every
    // expert fits one 16-row tile (uint4 keeps 16-row tiles: their register
    // budget holds two 8-token MMA groups)
    pl.bn = (bits == 8 && T > 16) ? 32 : 16;
    // the workspace holds the warp-MMA splits for batches where that mode is
    // the default's size class, else the tcgen05 plan's
    if (T <= 64) pl.splits = dec_splits(T, H, I, E, k, bits);
    return pl;
  }
  // default: tcgen05 for both GEMMs; one launch for both GEMMs of 8-bit
  // layers of many experts (measured rule above)
  (void)ok;
  if (bits == 8 && layer_default(T, E)) pl.layer = true;
  // 8-bit down GEMM on f16 operands after the in-place act -> f16 pass, for
  // layers of a few experts at 8-64 tokens: the f16 conversion of the codes
  // takes about half the instructions of bf16, which outweighs the pass
  // (Mixtral-shaped step T=64 248.3 -> 240.7 us, T=8 218.7 -> 213.1 us; T=1
  // 79.5 -> 81.9, fine-grained T=64 51.9 -> 57.4, prefill T=4096 2456 ->
  // 2556 us, where the pass costs more than it saves)
  if (bits == 8 && !pl.layer && E <= 16 && T >= 8 && T <= 64) pl.f16down = true;
  return pl;
}

struct WsLayout {
  size_t sorted, block_expert, offsets, num_padded, chunk_expert, chunk_start, counts, dep, xs,
      xinv, act, act_inv, y, topk_w, topk_ids, total;
  int64_t cap;
  TcPlan plan;
};

// with_route: the forward routes itself (router logits in), holding topk_w
// and topk_ids in the workspace too.
WsLayout ws_layout(int T, int H, int I, int E, int k, int bits, int group_size,
                   bool with_route = false) {
  WsLayout L;
  L.plan = tc_plan(T, H, I, E, k, bits);
  // partial outputs for every consumer choice (the warp-MMA plan's splits
  // and the tcgen05 plan's), so that a forced choice fits the same workspace
  const TcPlan fp = fwd_plan(T, H, I, E, k, bits, group_size, MQ_FWD_PATH_DECODE);
  const int ysplits = L.plan.splits > fp.splits ? L.plan.splits : fp.splits;
  const int bm = kAlignBlock;
  const int64_t S = (int64_t)T * k;
  const int64_t cap = moe_align_capacity(T, k, E, bm);
  L.cap = cap;
  size_t off = 0;
  L.sorted = off;       off += align256(sizeof(int32_t) * (size_t)cap);
  L.block_expert = off; off += align256(sizeof(int32_t) * (size_t)(cap / bm));
  L.offsets = off;      off += align256(sizeof(int32_t) * (size_t)(E + 1));
  L.num_padded = off;   off += align256(sizeof(int32_t));
  L.chunk_expert = off; off += align256(sizeof(int32_t) * (size_t)(cap / bm));
  L.chunk_start = off;  off += align256(sizeof(int32_t) * (size_t)(E + 1));
  L.counts = off;       off += align256(sizeof(int32_t) * (size_t)E);
  L.dep = off;          off += align256(sizeof(int32_t) * (size_t)(cap / bm));
  L.xs = off;           off += align256(sizeof(__half) * (size_t)cap * (size_t)H);
  L.xinv = off;         off += align256(sizeof(float) * (size_t)cap);
  L.act = off;          off += align256(sizeof(__nv_bfloat16) * (size_t)cap * (size_t)I);
  L.act_inv = off;      off += align256(sizeof(float) * (size_t)cap);
  L.y = off;            off += align256(sizeof(float) * (size_t)ysplits * (size_t)S * (size_t)H);
  L.topk_w = off;       if (with_route) off += align256(sizeof(float) * (size_t)S);
  L.topk_ids = off;     if (with_route) off += align256(sizeof(int32_t) * (size_t)S);
  L.total = off;
  return L;
}

bool fmt_ok(int bits, int group_size, int has_zp) {
  if (bits == 8) return group_size == -1 && has_zp == 0;
  if (bits == 4)
    return (group_size == 32 || group_size == 64 || group_size == 128 || group_size == 256) &&
           (has_zp == 0 || has_zp == 1);
  return false;
}

}  // namespace

int mq_set_error(int status, const char* msg) { return fail(status, "%s", msg); }

MQ_EXPORT const char* mq_status_string(int status) {
  switch (status) {
    case MQ_OK: return "ok";
    case MQ_ERR_INVALID_ARG: return "invalid argument";
    case MQ_ERR_UNSUPPORTED: return "unsupported";
    case MQ_ERR_CUDA: return "CUDA error";
    case MQ_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

MQ_EXPORT const char* mq_last_error_message(void) { return g_msg; }

MQ_EXPORT long long mq_kernel_launch_count(void) { return g_launches.load(); }

MQ_EXPORT int mq_test_layer_wait_extra(int extra) {
  if (extra < 0) return fail(MQ_ERR_INVALID_ARG, "extra must be >= 0");
  set_layer_wait_extra(extra);
  return MQ_OK;
}

MQ_EXPORT int mq_profile_enable(int on) {
  g_prof_on.store(on ? 1 : 0);
  return MQ_OK;
}

MQ_EXPORT int mq_profile_read(double* total_ms, long long* launches, int n_slots) {
  if (!total_ms || !launches || n_slots < 1) return fail(MQ_ERR_INVALID_ARG, "bad profile buffers");
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    recs.swap(g_prof_pending);
  }
  int status = MQ_OK;
  for (const ProfRec& r : recs) {
    float ms = 0.0f;
    cudaError_t err = cudaEventSynchronize(r.b);
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, r.a, r.b);
    if (err != cudaSuccess) status = cuda_fail(err, "mq_profile_read");
    g_prof_ms[r.slot] += ms;
    g_prof_n[r.slot] += 1;
  }
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (const ProfRec& r : recs) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  for (int i = 0; i < n_slots; ++i) {
    total_ms[i] = i < MQ_PROF_SLOTS ? g_prof_ms[i] : 0.0;
    launches[i] = i < MQ_PROF_SLOTS ? g_prof_n[i] : 0;
  }
  for (int i = 0; i < MQ_PROF_SLOTS; ++i) {
    g_prof_ms[i] = 0.0;
    g_prof_n[i] = 0;
  }
  return status;
}

MQ_EXPORT int mq_device_status(void* stream, uint32_t* flags) {
  if (!flags) return fail(MQ_ERR_INVALID_ARG, "flags is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return cuda_fail(err, "mq_device_status: stream synchronize");
  unsigned v = 0;
  err = cudaMemcpyFromSymbol(&v, g_dev_status, sizeof(v));
  if (err != cudaSuccess) return cuda_fail(err, "mq_device_status: read");
  const unsigned zero = 0;
  err = cudaMemcpyToSymbol(g_dev_status, &zero, sizeof(zero));
  if (err != cudaSuccess) return cuda_fail(err, "mq_device_status: clear");
  *flags = v;
  return MQ_OK;
}

MQ_EXPORT int moe_quantize_int8_per_channel(const void* w, int64_t rows, int64_t cols, int8_t* q,
                                            float* scale, void* stream) {
  if (rows < 0 || cols < 0) return fail(MQ_ERR_INVALID_ARG, "negative size");
  if (cols % 8 || cols > (int64_t(1) << 31) - 8)
    return fail(MQ_ERR_INVALID_ARG, "cols must be a multiple of 8 below 2^31");
  if (rows == 0) return MQ_OK;
  if (cols == 0) return fail(MQ_ERR_INVALID_ARG, "cols must be positive");
  if (!w || !q || !scale) return fail(MQ_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w) || !aligned16(q)) return fail(MQ_ERR_INVALID_ARG, "w and q must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(MQ_PROF_QUANT, st);
  cudaError_t err = launch_quant_int8(w, rows, cols, q, scale, st);
  return err == cudaSuccess ? MQ_OK : cuda_fail(err, "quantize_int8 launch");
}

MQ_EXPORT int moe_quantize_uint4_group(const void* w, int64_t rows, int64_t cols, int group_size,
                                       uint8_t* qweight, uint16_t* scales, uint8_t* qzeros,
                                       void* stream) {
  if (rows < 0 || cols <= 0) return fail(MQ_ERR_INVALID_ARG, "bad size");
  if (rows % 2) return fail(MQ_ERR_INVALID_ARG, "rows must be even (zero points pack two rows)");
  if (!(group_size == 32 || group_size == 64 || group_size == 128 || group_size == 256))
    return fail(MQ_ERR_INVALID_ARG, "group_size must be 32, 64, 128 or 256");
  if (cols % group_size) return fail(MQ_ERR_INVALID_ARG, "group_size must divide cols");
  if (cols > (int64_t(1) << 30)) return fail(MQ_ERR_INVALID_ARG, "cols too large");
  if (rows == 0) return MQ_OK;
  if (!w || !qweight || !scales || !qzeros) return fail(MQ_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w) || !aligned16(qweight)) return fail(MQ_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(MQ_PROF_QUANT, st);
  cudaError_t err = launch_quant_uint4(w, rows, cols, group_size, qweight, scales, qzeros, st);
  return err == cudaSuccess ? MQ_OK : cuda_fail(err, "quantize_uint4 launch");
}

MQ_EXPORT int moe_topk_route(const float* logits, int T, int E, int k, int renormalize,
                             float* topk_w, int32_t* topk_ids, void* stream) {
  if (T < 0) return fail(MQ_ERR_INVALID_ARG, "T must be >= 0");
  if (E < 1 || E > 1024) return fail(MQ_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  if (k < 1 || k > E || k > 32) return fail(MQ_ERR_INVALID_ARG, "need 1 <= k <= min(E, 32)");
  if (T == 0) return MQ_OK;
  if (!logits || !topk_w || !topk_ids) return fail(MQ_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(MQ_PROF_ROUTE, st);
  cudaError_t err = launch_route(logits, T, E, k, renormalize ? 1 : 0, topk_w, topk_ids, st);
  return err == cudaSuccess ? MQ_OK : cuda_fail(err, "route launch");
}

// mq_route_opts -> RouteOpts, with the checks moe_topk_route_ex documents.
static int route_opts_from(const mq_route_opts* opts, int E, int k, RouteOpts* o) {
  if (!opts) return fail(MQ_ERR_INVALID_ARG, "null route options");
  if (opts->scoring_func != MQ_SCORING_SOFTMAX && opts->scoring_func != MQ_SCORING_SIGMOID)
    return fail(MQ_ERR_INVALID_ARG, "unknown scoring_func %d", opts->scoring_func);
  const int G = opts->num_expert_group;
  if (G < 0 || G > 32) return fail(MQ_ERR_INVALID_ARG, "num_expert_group must be in [0, 32]");
  if (G > 1) {
    if (E % G) return fail(MQ_ERR_INVALID_ARG, "num_expert_group must divide E");
    if (opts->topk_group < 1 || opts->topk_group > G)
      return fail(MQ_ERR_INVALID_ARG, "topk_group must be in [1, num_expert_group]");
    if ((int64_t)k > (int64_t)opts->topk_group * (E / G))
      return fail(MQ_ERR_INVALID_ARG, "k exceeds the experts of topk_group groups");
  }
  if (!std::isfinite(opts->routed_scaling_factor))
    return fail(MQ_ERR_INVALID_ARG, "routed_scaling_factor must be finite");
  if (opts->e_score_correction_bias && !aligned16(opts->e_score_correction_bias))
    return fail(MQ_ERR_INVALID_ARG, "e_score_correction_bias must be 16-byte aligned");
  o->scoring = opts->scoring_func;
  o->renorm = opts->renormalize ? 1 : 0;
  o->groups = G > 1 ? G : 0;
  o->topk_group = G > 1 ? opts->topk_group : 0;
  o->bias = opts->e_score_correction_bias;
  o->scale = opts->routed_scaling_factor;
  return MQ_OK;
}

MQ_EXPORT int moe_topk_route_ex(const float* logits, int T, int E, int k,
                                const mq_route_opts* opts, float* topk_w, int32_t* topk_ids,
                                void* stream) {
  if (T < 0) return fail(MQ_ERR_INVALID_ARG, "T must be >= 0");
  if (E < 1 || E > 1024) return fail(MQ_ERR_UNSUPPORTED, "E must be in [1, 1024]");
  if (k < 1 || k > E || k > 32) return fail(MQ_ERR_INVALID_ARG, "need 1 <= k <= min(E, 32)");
  RouteOpts o;
  const int rc = route_opts_from(opts, E, k, &o);
  if (rc != MQ_OK) return rc;
  if (T == 0) return MQ_OK;
  if (!logits || !topk_w || !topk_ids) return fail(MQ_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(MQ_PROF_ROUTE, st);
  cudaError_t err = launch_route_ex(logits, T, E, k, o, topk_w, topk_ids, st);
  return err == cudaSuccess ? MQ_OK : cuda_fail(err, "route launch");
}

MQ_EXPORT int64_t moe_align_capacity(int T, int k, int E, int block_m) {
  if (T < 0 || k < 1 || E < 1 || block_m < 1) return -1;
  const int64_t S = (int64_t)T * k;
  const int64_t cap = S + (int64_t)(E < S ? E : S) * (block_m - 1);
  return (cap + block_m - 1) / block_m * block_m;
}

MQ_EXPORT int moe_align_block(const int32_t* topk_ids, int T, int k, int E, int block_m,
                              int32_t* sorted_slot_ids, int32_t* block_expert,
                              int32_t* expert_offsets, int32_t* num_padded, int64_t capacity,
                              void* stream) {
  if (T < 0 || k < 1 || E < 1) return fail(MQ_ERR_INVALID_ARG, "bad T, k or E");
  if (E > 1024) return fail(MQ_ERR_UNSUPPORTED, "E must be <= 1024");
  if (block_m < 1 || block_m > 1024) return fail(MQ_ERR_INVALID_ARG, "block_m must be in [1, 1024]");
  if ((int64_t)T * k > (int64_t(1) << 30)) return fail(MQ_ERR_UNSUPPORTED, "too many slots");
  if (capacity < moe_align_capacity(T, k, E, block_m))
    return fail(MQ_ERR_INVALID_ARG, "capacity below moe_align_capacity()");
  if ((T > 0 && !topk_ids) || !sorted_slot_ids || !block_expert || !expert_offsets || !num_padded)
    return fail(MQ_ERR_INVALID_ARG, "null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = status_ptr();
  LaunchScope ls(MQ_PROF_ALIGN, st);
  cudaError_t err = launch_align(topk_ids, T, k, E, block_m, sorted_slot_ids, block_expert,
                                 expert_offsets, num_padded, status, st);
  return err == cudaSuccess ? MQ_OK : cuda_fail(err, "align launch");
}

MQ_EXPORT size_t moe_quant_forward_workspace(int T, int H, int I, int E, int k, int bits,
                                             int group_size) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || k < 1 || k > E) return 0;
  if (!fmt_ok(bits, group_size, 0)) return 0;
  return ws_layout(T, H, I, E, k, bits, group_size).total;
}

MQ_EXPORT int moe_quant_forward_ex(const void* x, int T, int H, int I, int E, int k, int bits,
                                   int group_size, int has_zp, const void* w13, const void* w2,
                                   const void* s13, const void* s2, const uint8_t* z13,
                                   const uint8_t* z2, const float* topk_w,
                                   const int32_t* topk_ids, void* workspace, size_t ws_bytes,
                                   void* out, unsigned flags, void* stream);

MQ_EXPORT int moe_quant_forward(const void* x, int T, int H, int I, int E, int k, int bits,
                                int group_size, int has_zp, const void* w13, const void* w2,
                                const void* s13, const void* s2, const uint8_t* z13,
                                const uint8_t* z2, const float* topk_w, const int32_t* topk_ids,
                                void* workspace, size_t ws_bytes, void* out, void* stream) {
  return moe_quant_forward_ex(x, T, H, I, E, k, bits, group_size, has_zp, w13, w2, s13, s2, z13,
                              z2, topk_w, topk_ids, workspace, ws_bytes, out, 0u, stream);
}

// The forward.  With logits (router logits [T, E]) it routes itself, into
// the workspace; otherwise topk_w / topk_ids are the caller's.
static int forward_impl(const void* x, int T, int H, int I, int E, int k, int bits,
                        int group_size, int has_zp, const void* w13, const void* w2,
                        const void* s13, const void* s2, const uint8_t* z13, const uint8_t* z2,
                        const float* topk_w, const int32_t* topk_ids, const float* logits,
                        const RouteOpts& ro, void* workspace, size_t ws_bytes, void* out,
                        unsigned flags, void* stream) {
  constexpr unsigned kW8Flags = MQ_FWD_W8_UINT8 | MQ_FWD_SCALE_F16 | MQ_FWD_SCALE_BF16 |
                                MQ_FWD_SCALE_PER_TENSOR;
  constexpr unsigned kAllFlags = kW8Flags | MQ_FWD_ACT_F16 | MQ_FWD_ROUTER_WEIGHT_ON_INPUT |
                                 MQ_FWD_PATH_TENSOR_CORE | MQ_FWD_PATH_DECODE |
                                 MQ_FWD_PATH_LAYER;
  if (T < 0 || H <= 0 || I <= 0 || E < 1) return fail(MQ_ERR_INVALID_ARG, "bad T, H, I or E");
  if (k < 1 || k > E || k > 32) return fail(MQ_ERR_INVALID_ARG, "need 1 <= k <= min(E, 32)");
  if (E > 1024) return fail(MQ_ERR_UNSUPPORTED, "E must be <= 1024");
  if (flags & ~kAllFlags) return fail(MQ_ERR_UNSUPPORTED, "unknown flags 0x%x", flags & ~kAllFlags);
  if (bits == 4 && (flags & kW8Flags))
    return fail(MQ_ERR_UNSUPPORTED, "uint8 codes and scale options apply to bits = 8 only");
  if ((flags & MQ_FWD_SCALE_F16) && (flags & MQ_FWD_SCALE_BF16))
    return fail(MQ_ERR_UNSUPPORTED, "scales are float16 or bfloat16, not both");
  {
    const unsigned paths = flags & (MQ_FWD_PATH_TENSOR_CORE | MQ_FWD_PATH_DECODE | MQ_FWD_PATH_LAYER);
    if (paths & (paths - 1))
      return fail(MQ_ERR_INVALID_ARG, "at most one of the MQ_FWD_PATH_* flags");
  }
  if ((flags & MQ_FWD_PATH_LAYER) && bits != 8)
    return fail(MQ_ERR_UNSUPPORTED, "the one-launch layer takes 8-bit codes");
  if ((flags & MQ_FWD_PATH_DECODE) && !dec_supported(bits, group_size, H, I))
    return fail(MQ_ERR_UNSUPPORTED, "the warp-MMA consumers take 8-bit codes or uint4 with group_size 128 or 256");
  const bool w8zp = bits == 8 && group_size == -1 && has_zp == 1 && (flags & MQ_FWD_W8_UINT8);
  if (!fmt_ok(bits, group_size, has_zp) && !w8zp)
    return fail(MQ_ERR_UNSUPPORTED,
                "format must be (8, -1, 0), (8, -1, 1) with uint8 codes, or (4, 32..256, 0|1)");
  if (H % 128 || I % 128) return fail(MQ_ERR_UNSUPPORTED, "H and I must be multiples of 128");
  if (bits == 4 && (H % group_size || I % group_size))
    return fail(MQ_ERR_UNSUPPORTED, "group_size must divide H and I");
  if ((int64_t)T * k > (int64_t(1) << 24)) return fail(MQ_ERR_UNSUPPORTED, "too many token-slots");
  if (T == 0) return MQ_OK;
  if (!x || !w13 || !w2 || !s13 || !s2 || !out || !workspace ||
      (logits ? false : (!topk_w || !topk_ids)))
    return fail(MQ_ERR_INVALID_ARG, "null pointer");
  if (has_zp && (!z13 || !z2)) return fail(MQ_ERR_INVALID_ARG, "null zero points");
  if (!has_zp && (z13 || z2)) return fail(MQ_ERR_INVALID_ARG, "zero points given with has_zp = 0");
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(out) || !aligned16(workspace))
    return fail(MQ_ERR_INVALID_ARG, "x, w13, w2, out and workspace must be 16-byte aligned");
  if (!aligned16(s13) || !aligned16(s2) || (z13 && !aligned16(z13)) || (z2 && !aligned16(z2)))
    return fail(MQ_ERR_INVALID_ARG, "scales and zero points must be 16-byte aligned");
  {
    const char* xb = static_cast<const char*>(x);
    const char* ob = static_cast<const char*>(out);
    const size_t nb = (size_t)T * H * 2;
    // out == x is fused_experts' inplace: x is read (gathered) before any
    // output is written
    if (ob != xb && ob < xb + nb && xb < ob + nb)
      return fail(MQ_ERR_INVALID_ARG, "out overlaps x (only out == x is allowed)");
  }
  const WsLayout L = ws_layout(T, H, I, E, k, bits, group_size, logits != nullptr);
  const TcPlan plan = fwd_plan(T, H, I, E, k, bits, group_size, flags);
  const int bm = kAlignBlock;
  if (ws_bytes < L.total)
    return fail(MQ_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, L.total);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  float* rw = logits ? reinterpret_cast<float*>(ws + L.topk_w) : nullptr;
  int32_t* rid = logits ? reinterpret_cast<int32_t*>(ws + L.topk_ids) : nullptr;
  if (logits) {
    topk_w = rw;
    topk_ids = rid;
  }
  MoeArgs a;
  a.x = x;
  a.flags = flags;
  a.T = T; a.H = H; a.I = I; a.E = E; a.k = k;
  a.bits = bits; a.group_size = group_size; a.has_zp = has_zp;
  a.w13 = w13; a.w2 = w2; a.s13 = s13; a.s2 = s2; a.z13 = z13; a.z2 = z2;
  a.topk_w = topk_w; a.topk_ids = topk_ids;
  a.out = out;
  a.status = status_ptr();
  a.sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  a.block_expert = reinterpret_cast<int32_t*>(ws + L.block_expert);
  a.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  a.num_padded = reinterpret_cast<int32_t*>(ws + L.num_padded);
  a.chunk_expert = reinterpret_cast<int32_t*>(ws + L.chunk_expert);
  a.chunk_start = reinterpret_cast<int32_t*>(ws + L.chunk_start);
  a.counts = reinterpret_cast<int32_t*>(ws + L.counts);
  a.dep = reinterpret_cast<int32_t*>(ws + L.dep);
  a.act = reinterpret_cast<__nv_bfloat16*>(ws + L.act);
  a.y = reinterpret_cast<float*>(ws + L.y);
  a.bm = bm;
  a.cap = L.cap;

  cudaError_t err;
  // the plain softmax router of small batches runs inside the align kernel
  const bool plain = route_opts_plain(ro);
  const bool fused = logits && plain && route_fused(T, k, E);
  if (logits && !fused) {  // otherwise the router kernel first
    LaunchScope ls(MQ_PROF_ROUTE, st);
    err = plain ? launch_route(logits, T, E, k, ro.renorm, rw, rid, st)
                : launch_route_ex(logits, T, E, k, ro, rw, rid, st);
    if (err != cudaSuccess) return cuda_fail(err, "forward: route launch");
  }
  const int chunk = plan.bn;  // token rows per tile of the chunk table
  {
    LaunchScope ls(MQ_PROF_ALIGN, st);
    if (fused)
      err = launch_route_align(logits, ro.renorm, rw, rid, T, k, E, bm, a.sorted, a.block_expert,
                               a.offsets, a.num_padded, a.status, st, chunk, a.chunk_expert,
                               a.chunk_start, a.counts, plan.layer ? a.dep : nullptr);
    else
      err = launch_align(topk_ids, T, k, E, bm, a.sorted, a.block_expert, a.offsets,
                         a.num_padded, a.status, st, chunk, a.chunk_expert, a.chunk_start,
                         a.counts, plan.layer ? a.dep : nullptr);
  }
  if (err != cudaSuccess) return cuda_fail(err, "forward: align launch");
  void* xs = ws + L.xs;
  float* xinv = reinterpret_cast<float*>(ws + L.xinv);
  {
    LaunchScope ls(MQ_PROF_GATHER, st);
    err = launch_gather_rows(a, xs, xinv, st);
  }
  if (err != cudaSuccess) return cuda_fail(err, "forward: gather launch");
  if (plan.layer) {
    {
      LaunchScope ls(MQ_PROF_LAYER, st);
      err = launch_layer_tc(a, plan, xs, xinv, a.y, st);
    }
    if (err != cudaSuccess) return cuda_fail(err, "forward: expert layer launch");
    LaunchScope ls(MQ_PROF_COMBINE, st);
    err = launch_combine_splits(a, a.y, plan.splits, st);
    if (err != cudaSuccess) return cuda_fail(err, "forward: combine launch");
    return MQ_OK;
  }
  {
    LaunchScope ls(MQ_PROF_GEMM1, st);
    err = launch_gemm1_tc(a, plan, xs, xinv, st);
  }
  if (err != cudaSuccess) return cuda_fail(err, "forward: gate/up GEMM launch");
  float* act_inv = reinterpret_cast<float*>(ws + L.act_inv);
  if ((bits == 4 && !plan.sync2) || plan.f16down) {
    // the tcgen05 uint4 down GEMM runs f16 operands (and the 8-bit one where
    // the plan says so); otherwise the 8-bit one and the warp-MMA mode read
    // bf16 act
    LaunchScope ls(MQ_PROF_ACTF16, st);
    err = launch_act_to_f16(a, act_inv, st);
    if (err != cudaSuccess) return cuda_fail(err, "forward: act conversion launch");
  }
  {
    LaunchScope ls(MQ_PROF_GEMM2, st);
    err = launch_gemm2_tc(a, plan, act_inv, a.y, st);
  }
  if (err != cudaSuccess) return cuda_fail(err, "forward: down GEMM launch");
  {
    LaunchScope ls(MQ_PROF_COMBINE, st);
    err = launch_combine_splits(a, a.y, plan.splits, st);
  }
  if (err != cudaSuccess) return cuda_fail(err, "forward: combine launch");
  return MQ_OK;
}

MQ_EXPORT int moe_quant_forward_ex(const void* x, int T, int H, int I, int E, int k, int bits,
                                   int group_size, int has_zp, const void* w13, const void* w2,
                                   const void* s13, const void* s2, const uint8_t* z13,
                                   const uint8_t* z2, const float* topk_w,
                                   const int32_t* topk_ids, void* workspace, size_t ws_bytes,
                                   void* out, unsigned flags, void* stream) {
  const RouteOpts none = {MQ_SCORING_SOFTMAX, 0, 0, 0, nullptr, 1.0f};
  return forward_impl(x, T, H, I, E, k, bits, group_size, has_zp, w13, w2, s13, s2, z13, z2,
                      topk_w, topk_ids, nullptr, none, workspace, ws_bytes, out, flags, stream);
}

MQ_EXPORT size_t moe_quant_forward_logits_workspace(int T, int H, int I, int E, int k, int bits,
                                                    int group_size) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || k < 1 || k > E) return 0;
  if (!fmt_ok(bits, group_size, 0)) return 0;
  return ws_layout(T, H, I, E, k, bits, group_size, true).total;
}

MQ_EXPORT int moe_quant_forward_logits(const void* x, const float* router_logits, int T, int H,
                                       int I, int E, int k, int renormalize, int bits,
                                       int group_size, int has_zp, const void* w13,
                                       const void* w2, const void* s13, const void* s2,
                                       const uint8_t* z13, const uint8_t* z2, void* workspace,
                                       size_t ws_bytes, void* out, unsigned flags, void* stream) {
  if (T > 0 && !router_logits) return fail(MQ_ERR_INVALID_ARG, "null router_logits");
  const RouteOpts ro = {MQ_SCORING_SOFTMAX, renormalize ? 1 : 0, 0, 0, nullptr, 1.0f};
  return forward_impl(x, T, H, I, E, k, bits, group_size, has_zp, w13, w2, s13, s2, z13, z2,
                      nullptr, nullptr, router_logits, ro, workspace, ws_bytes, out, flags, stream);
}

MQ_EXPORT int moe_quant_forward_logits_ex(const void* x, const float* router_logits, int T,
                                          int H, int I, int E, int k, const mq_route_opts* opts,
                                          int bits, int group_size, int has_zp, const void* w13,
                                          const void* w2, const void* s13, const void* s2,
                                          const uint8_t* z13, const uint8_t* z2, void* workspace,
                                          size_t ws_bytes, void* out, unsigned flags,
                                          void* stream) {
  if (k < 1 || k > E || k > 32) return fail(MQ_ERR_INVALID_ARG, "need 1 <= k <= min(E, 32)");
  RouteOpts ro;
  const int rc = route_opts_from(opts, E, k, &ro);
  if (rc != MQ_OK) return rc;
  if (T > 0 && !router_logits) return fail(MQ_ERR_INVALID_ARG, "null router_logits");
  return forward_impl(x, T, H, I, E, k, bits, group_size, has_zp, w13, w2, s13, s2, z13, z2,
                      nullptr, nullptr, router_logits, ro, workspace, ws_bytes, out, flags, stream);
}
