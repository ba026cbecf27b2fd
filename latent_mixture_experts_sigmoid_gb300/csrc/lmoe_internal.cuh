// Internal declarations shared by the CUDA translation units of liblmoe.so.
// Nothing here is part of the public ABI (include/lmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lmoe.h"

namespace lmoe {

constexpr int kNumSmsDefault = 152;

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
// SituGLU scalar math (vLLM PR #50088, commit 2), fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct SituParams {
  float beta, inv_beta, lbeta, inv_lbeta;
  int has_lbeta;
};

__device__ __forceinline__ float situ1(float g, float u, const SituParams& p) {
  const float sig = __fdividef(1.0f, 1.0f + __expf(-g));
  const float gate_out = p.beta * tanh_fast(g * p.inv_beta) * sig;
  const float up_out = p.has_lbeta ? p.lbeta * tanh_fast(u * p.inv_lbeta) : u;
  return gate_out * up_out;
}

__device__ __forceinline__ uint32_t situ2(uint32_t g2, uint32_t u2, const SituParams& p) {
  return pack_bf16x2(situ1(bf16_lo(g2), bf16_lo(u2), p), situ1(bf16_hi(g2), bf16_hi(u2), p));
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
// Host-side helpers
// ---------------------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
int num_sms();  // of the current device (cached per device)

// Launchers (return cudaError_t of the launch); arguments already validated.
cudaError_t launch_route(const float* logits, const float* bias, int T, int E, int k,
                         int renorm, float rsf, int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_situ(const uint16_t* in, uint16_t* out, long long N, int d, float beta,
                        float lbeta, cudaStream_t s);
cudaError_t launch_masked_situ(const uint16_t* in, uint16_t* out, const int32_t* counts, int E,
                               int T_max, int d, float beta, float lbeta, cudaStream_t s);

}  // namespace lmoe
