// Internal declarations shared by the CUDA translation units of liblmoe.so.
// Nothing here is part of the public ABI (include/lmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/lmoe.h"

namespace lmoe {

constexpr int kNumSmsDefault = 152;

// Codes of the device error word (the first one written stays): 1-6 are the
// tensor-core GEMM's bounded waits; kErrExpertId is an expert id outside
// [0, E) handed to the pre-routed forward.
constexpr int kErrExpertId = 7;

// Device address of the error word of the current device.
int* device_error_word();

// The CUDA driver API's cuTensorMapEncodeTiled (looked up once), or nullptr.
void* tensor_map_encoder();

// latent_moe_forward on the library's own static scratch (device memory of
// the current device, so its pointer is not queried like a caller's).
int forward_on_library_scratch(const lmoe_dims* dims, const lmoe_weights* wt,
                               const lmoe_bf16* hidden, const float* router_logits,
                               lmoe_bf16* out, void* scratch, size_t scratch_bytes,
                               const lmoe_debug* dbg, void* stream);

// ---------------------------------------------------------------------------
// bf16 <-> fp32 on raw 16-bit patterns (round to nearest even on the way down)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t two) { return __uint_as_float(two << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t two) { return __uint_as_float(two & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

// ---------------------------------------------------------------------------
// SituGLU math (vLLM PR #50088, commit 2), fp32
// ---------------------------------------------------------------------------
//   out = beta*tanh(g/beta) * [linear_beta*tanh(u/linear_beta)  or  u] / (1 + e^{-g})
// Both tanh factors come from the hardware tanh (tanh.approx.f32: documented
// maximum relative error near 2^-11; an exhaustive run over every finite fp32
// input on GB300 measured 2^-16.5).  The sigmoid stays 1 / (1 + e^{-g}) from
// the hardware 2^x and reciprocal: 0.5 + 0.5*tanh(g/2) would cancel for very
// negative gates, where the output is tiny but must keep its relative
// accuracy.  Four transcendental ops per element (two tanh, one 2^x, one
// reciprocal) and about ten other instructions; a denominator beyond 2^126
// (gate below about -87) gives 0, the value to bf16 precision.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct SituParams {
  float beta, inv_beta, lbeta, inv_lbeta;
  int has_lbeta;
};

// Two elements at a time on the packed fp32 pipe (sm_100 f32x2 FMA/MUL/ADD,
// each lane rounded to nearest like the scalar form); the transcendental ops
// stay per element.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_make(uint32_t lo_bits, uint32_t hi_bits) {
  f32x2 d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo_bits), "r"(hi_bits));
  return d;
}
__device__ __forceinline__ f32x2 f2_splat(float x) {
  return f2_make(__float_as_uint(x), __float_as_uint(x));
}
__device__ __forceinline__ float f2_lo(f32x2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(f32x2 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// elementwise f(x) of a pair through a scalar transcendental op
#define LMOE_F2_APPLY(f, v) f2_make(__float_as_uint(f(f2_lo(v))), __float_as_uint(f(f2_hi(v))))

// bf16x2 gate / up in, fp32 pair out (lo, hi)
__device__ __forceinline__ f32x2 situ2_f32(uint32_t g2, uint32_t u2, const SituParams& p) {
  const f32x2 g = f2_make(g2 << 16, g2 & 0xFFFF0000u);
  const f32x2 u = f2_make(u2 << 16, u2 & 0xFFFF0000u);
  const f32x2 tg = LMOE_F2_APPLY(tanh_fast, f2_mul(g, f2_splat(p.inv_beta)));
  const f32x2 e = LMOE_F2_APPLY(ex2_fast, f2_mul(g, f2_splat(-1.4426950408889634f)));
  const f32x2 up = p.has_lbeta ? f2_mul(LMOE_F2_APPLY(tanh_fast, f2_mul(u, f2_splat(p.inv_lbeta))),
                                        f2_splat(p.lbeta))
                               : u;
  const f32x2 num = f2_mul(f2_mul(tg, f2_splat(p.beta)), up);
  const f32x2 r = LMOE_F2_APPLY(rcp_fast, f2_add(e, f2_splat(1.0f)));
  return f2_mul(num, r);
}

__device__ __forceinline__ uint32_t situ2(uint32_t g2, uint32_t u2, const SituParams& p) {
  const f32x2 o = situ2_f32(g2, u2, p);
  return pack_bf16x2(f2_lo(o), f2_hi(o));
}

inline SituParams make_situ_params(float beta, float lbeta) {
  SituParams p;
  p.beta = beta;
  p.inv_beta = 1.0f / beta;
  p.has_lbeta = lbeta > 0.0f;
  p.lbeta = p.has_lbeta ? lbeta : 1.0f;
  p.inv_lbeta = 1.0f / p.lbeta;
  return p;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation: it may start while its predecessor in the
// stream drains.  pdl_trigger() lets the next kernel be scheduled; pdl_wait()
// blocks until every prerequisite grid has completed and its memory is
// visible.  Nothing produced or read by an earlier kernel is touched before
// pdl_wait() (only constant weights may be prefetched).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with thread-block clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Host-side helpers
// ---------------------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
int num_sms();  // of the current device (cached per device)

// Launchers (return cudaError_t of the launch); arguments already validated.
// logits [T, E] fp32 with rows ld >= E elements apart
cudaError_t launch_route(const float* logits, long long ld, const float* bias, int T, int E, int k,
                         int renorm, float rsf, int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_situ(const uint16_t* in, uint16_t* out, long long N, int d, float beta,
                        float lbeta, cudaStream_t s);
cudaError_t launch_masked_situ(const uint16_t* in, uint16_t* out, const int32_t* counts, int E,
                               int T_max, int d, float beta, float lbeta, cudaStream_t s);

}  // namespace lmoe
