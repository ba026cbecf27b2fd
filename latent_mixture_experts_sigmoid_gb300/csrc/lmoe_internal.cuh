// Internal declarations shared by the CUDA translation units of liblmoe.so.
// Nothing here is part of the public ABI (include/lmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

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
// Written from the identities
//   tanh(a)    = -m / (2 + m),   m = e^{-2|a|} - 1   (sign restored separately)
//   sigmoid(g) = 1 / (1 + e^{-g})
// so that one reciprocal serves the whole product:
//   out = [beta*sgn(g)*(-m1)] * [linear_beta*sgn(u)*(-m2)  or  u]
//         / [(2 + m1) * (1 + e^{-g}) * (2 + m2  or  1)]
// m = e^z - 1 (z <= 0) comes from the hardware 2^x for |z| >= 0.2 and from
// its Taylor series to z^5 below that (no cancellation); relative error of
// every factor is about 1e-6, so the bf16 result is almost always the
// correctly rounded one.  A denominator beyond 2^126 (gate below about -87)
// gives 0, the value to bf16 precision.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float expm1_neg(float z) {   // e^z - 1 for z <= 0
  if (z > -0.2f) {
    float p = 1.0f / 120.0f;
    p = fmaf(p, z, 1.0f / 24.0f);
    p = fmaf(p, z, 1.0f / 6.0f);
    p = fmaf(p, z, 0.5f);
    p = fmaf(p, z, 1.0f);
    return p * z;
  }
  return ex2_fast(z * 1.4426950408889634f) - 1.0f;
}

struct SituParams {
  float beta, inv_beta, lbeta, inv_lbeta;
  int has_lbeta;
};

__device__ __forceinline__ float situ1(float g, float u, const SituParams& p) {
  const float m1 = expm1_neg(-2.0f * fabsf(g * p.inv_beta));
  const float e = ex2_fast(-g * 1.4426950408889634f);
  float num = copysignf(p.beta, g) * (-m1);
  float den = (2.0f + m1) * (1.0f + e);
  if (p.has_lbeta) {
    const float m2 = expm1_neg(-2.0f * fabsf(u * p.inv_lbeta));
    num *= copysignf(p.lbeta, u) * (-m2);
    den *= (2.0f + m2);
  } else {
    num *= u;
  }
  return __fdividef(num, den);
}

// Two elements at a time on the packed fp32 pipe (sm_100 f32x2 FMA/MUL/ADD,
// each lane rounded to nearest like the scalar form); the hardware 2^x and
// reciprocal stay per element.  Same formulation and accuracy as situ1.
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
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e^z - 1 for a pair of z <= 0 (Taylor series to z^5 above -0.2, else 2^x - 1)
__device__ __forceinline__ f32x2 expm1_neg2(f32x2 z) {
  f32x2 p = f2_fma(z, f2_splat(1.0f / 120.0f), f2_splat(1.0f / 24.0f));
  p = f2_fma(p, z, f2_splat(1.0f / 6.0f));
  p = f2_fma(p, z, f2_splat(0.5f));
  p = f2_fma(p, z, f2_splat(1.0f));
  const f32x2 small = f2_mul(p, z);
  const f32x2 t = f2_mul(z, f2_splat(1.4426950408889634f));
  const f32x2 big = f2_add(f2_make(__float_as_uint(ex2_fast(f2_lo(t))),
                                   __float_as_uint(ex2_fast(f2_hi(t)))),
                           f2_splat(-1.0f));
  const uint32_t lo = f2_lo(z) > -0.2f ? (uint32_t)small : (uint32_t)big;
  const uint32_t hi = f2_hi(z) > -0.2f ? (uint32_t)(small >> 32) : (uint32_t)(big >> 32);
  return f2_make(lo, hi);
}

// bf16x2 gate / up in, fp32 pair out (lo, hi)
__device__ __forceinline__ f32x2 situ2_f32(uint32_t g2, uint32_t u2, const SituParams& p) {
  const f32x2 g = f2_make(g2 << 16, g2 & 0xFFFF0000u);
  const f32x2 gabs = g & 0x7FFFFFFF7FFFFFFFull;
  const f32x2 m1 = expm1_neg2(f2_mul(gabs, f2_splat(-2.0f * p.inv_beta)));
  const f32x2 t = f2_mul(g, f2_splat(-1.4426950408889634f));
  const f32x2 e = f2_make(__float_as_uint(ex2_fast(f2_lo(t))), __float_as_uint(ex2_fast(f2_hi(t))));
  // -beta with the sign of g flipped: num = sgn(g) * beta * (-m1)
  const f32x2 nb = (g & 0x8000000080000000ull) ^ f2_splat(-p.beta);
  f32x2 num = f2_mul(nb, m1);
  f32x2 den = f2_mul(f2_add(m1, f2_splat(2.0f)), f2_add(e, f2_splat(1.0f)));
  const f32x2 u = f2_make(u2 << 16, u2 & 0xFFFF0000u);
  if (p.has_lbeta) {
    const f32x2 uabs = u & 0x7FFFFFFF7FFFFFFFull;
    const f32x2 m2 = expm1_neg2(f2_mul(uabs, f2_splat(-2.0f * p.inv_lbeta)));
    const f32x2 nl = (u & 0x8000000080000000ull) ^ f2_splat(-p.lbeta);
    num = f2_mul(num, f2_mul(nl, m2));
    den = f2_mul(den, f2_add(m2, f2_splat(2.0f)));
  } else {
    num = f2_mul(num, u);
  }
  // a denominator beyond 2^126 (gate below about -87) flushes its reciprocal
  // to 0, the value to bf16 precision
  const f32x2 r = f2_make(__float_as_uint(rcp_fast(f2_lo(den))),
                          __float_as_uint(rcp_fast(f2_hi(den))));
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
