// moe_quant_forward_noalloc: the fused forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: a plugin
// hosted inside an application that owns all device memory through its own
// allocator and gives the plugin only its input and output buffers, or code
// on a path where an allocation (a synchronising call that may fail) is not
// allowed.  For them the forward's scratch lives in a fixed array compiled
// into this library.  Each GPU that loads the library holds that array until
// the process exits.
#include "common.cuh"

#include <mutex>
#include <stdio.h>

#define MQ_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device

// In host code `g_scratch` is only a stand-in for the symbol, not a device
// address: its device address is looked up below and passed to the kernels.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of this device's scratch array; looked up on the first call
// on each device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

MQ_EXPORT int moe_quant_forward_noalloc(const void* x, int T, int H, int I, int E, int k, int bits,
                                        int group_size, int has_zp, const void* w13,
                                        const void* w2, const void* s13, const void* s2,
                                        const uint8_t* z13, const uint8_t* z2,
                                        const float* topk_w, const int32_t* topk_ids, void* out,
                                        void* stream) {
  const size_t need = moe_quant_forward_workspace(T, H, I, E, k, bits, group_size);
  if (need == 0)  // the workspace query rejects these sizes; let the forward report why
    return moe_quant_forward(x, T, H, I, E, k, bits, group_size, has_zp, w13, w2, s13, s2, z13,
                             z2, topk_w, topk_ids, nullptr, 0, out, stream);
  char msg[256];
  if (need > kScratchBytes) {
    snprintf(msg, sizeof(msg),
             "moe_quant_forward_noalloc: these sizes need %zu bytes of scratch, more than its "
             "fixed %zu; use moe_quant_forward with a caller-provided workspace",
             need, kScratchBytes);
    return mq_set_error(MQ_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  const cudaError_t err = scratch_address(&scratch);
  if (err != cudaSuccess) {
    snprintf(msg, sizeof(msg), "moe_quant_forward_noalloc: scratch address lookup failed: %s",
             cudaGetErrorString(err));
    return mq_set_error(MQ_ERR_CUDA, msg);
  }
  // Nothing in the scratch has to start at zero: every region the forward
  // reads is written earlier in the same call.
  return moe_quant_forward(x, T, H, I, E, k, bits, group_size, has_zp, w13, w2, s13, s2, z13, z2,
                           topk_w, topk_ids, scratch, kScratchBytes, out, stream);
}
