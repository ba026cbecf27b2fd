// latent_moe_forward_noalloc: the layer forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin that an inference
// runtime calls with only its input and output buffers (the runtime owns every
// allocation), host code without an allocator of its own, or a latency path
// where cudaMalloc is not allowed because it may synchronise the device.  For
// them this entry point runs the same kernels as latent_moe_forward with its
// scratch in a fixed array that the library itself holds in device memory.
//
// The array is a file-scope __device__ variable of kStaticScratchBytes
// (32 MiB): every GPU that loads the library holds it until the process exits.
// Host code cannot use the variable's name as a device address; its address on
// a device comes from cudaGetSymbolAddress, called once per device (with that
// device current) by the first call made on that device, and cached.
#include <mutex>

#include "lmoe_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device (set up once).
int scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LMOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return LMOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return LMOE_OK;
}

}  // namespace

extern "C" int latent_moe_forward_noalloc(const lmoe_dims* dims, const lmoe_weights* weights,
                                          const lmoe_bf16* hidden, const float* router_logits,
                                          lmoe_bf16* out, const lmoe_debug* dbg, void* stream) {
  if (!dims) return LMOE_ERR_NULL;
  if (dims->T == 0) return latent_moe_forward(dims, weights, hidden, router_logits, out, nullptr,
                                              0, dbg, stream);
  const size_t need = latent_moe_workspace_bytes(dims);
  if (need == 0)   // invalid dims: let the regular entry point name the error
    return latent_moe_forward(dims, weights, hidden, router_logits, out, nullptr, 0, dbg, stream);
  if (need > kStaticScratchBytes) return LMOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != LMOE_OK) return st;
  return latent_moe_forward(dims, weights, hidden, router_logits, out, scratch,
                            kStaticScratchBytes, dbg, stream);
}
