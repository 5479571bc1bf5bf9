// moe_forward_decode_noalloc: the decode chain with its scratch in a fixed device array
// owned by this library, for callers that cannot allocate device memory themselves.
//
// Some callers have no way to call cudaMalloc: a plugin hosted inside another runtime that
// owns every device allocation and hands out no allocator, or a latency-critical serving
// loop that may not allocate because cudaMalloc can synchronise the whole device. moe_forward
// needs a caller-allocated workspace; this entry point instead uses the file-scope array
// below, so the caller passes only inputs and outputs.
//
// The array costs kStaticScratchBytes on every GPU that loads this library, until the
// process exits. All calls share it, so two calls that overlap on the GPU (different
// streams, or different host threads, without ordering between them) race on it. Its device
// address is looked up once per device and kept, so a cudaDeviceReset() (which reloads the
// device code) makes the kept address stale: the entry point is not for use after one.
#include <mutex>

#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)4 << 20;   // 4 MiB

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64];   // device address of g_static_scratch, per device ordinal

// Host code sees g_static_scratch only as a host-side stand-in; the kernels need its device
// address, looked up once per device with that device current (null on failure).
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" MOE_API moe_status_t moe_forward_decode_noalloc(const moe_config_t* cfg,
                                                           const moe_weights_t* weights,
                                                           const void* x, void* out,
                                                           void* stream) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (cfg->path == MOE_PATH_GROUPED) return MOE_ERR_UNSUPPORTED;
  moe_config_t c = *cfg;
  c.path = MOE_PATH_DECODE;
  size_t need = 0;
  moe_status_t s = moe_workspace_size(&c, &need);   // also validates the decode limits
  if (s != MOE_OK) return s;
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (c.num_tokens == 0) return MOE_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  void* scratch = scratch_address(dev);
  if (!scratch) return MOE_ERR_CUDA;
  // moe_forward clears every part of the scratch that must start at zero (the header with
  // its status word and counters, and the atomic accumulator) before using it.
  return moe_forward(&c, weights, x, out, scratch, kStaticScratchBytes, stream, nullptr, nullptr,
                     nullptr);
}

extern "C" MOE_API moe_status_t moe_noalloc_read_device_status(void* stream, int32_t* status) {
  if (!status) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  void* scratch = scratch_address(dev);
  if (!scratch) return MOE_ERR_CUDA;
  return moe_read_device_status(scratch, stream, status);
}
