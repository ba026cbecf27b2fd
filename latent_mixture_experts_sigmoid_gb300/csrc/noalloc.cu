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
// Host code cannot use the variable's name as a device address; every call
// looks the address up on the current device with cudaGetSymbolAddress.  The
// lookup is not cached, so a call made after a device reset or a new primary
// context gets the array of the live context, never a stale address.  With
// CUDA's lazy module loading, the first lookup on a device loads this
// library's module there: that reserves the 32 MiB and may synchronise the
// device, so a caller with a strict latency path makes its first call (or any
// other call of the library) on each device before that path, and before any
// stream capture.
#include "lmoe_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.
int scratch_on_current_device(void** addr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  *addr = p;
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
  return lmoe::forward_on_library_scratch(dims, weights, hidden, router_logits, out, scratch,
                                          kStaticScratchBytes, dbg, stream);
}
