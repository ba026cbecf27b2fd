// SituGLU gated activation, dense and masked (batched MoE) layouts.
//
// vLLM PR #50088, commit 2:
//   gate_out = beta * tanh(gate / beta) * sigmoid(gate)
//   up_out   = linear_beta * tanh(up / linear_beta)   (linear_beta > 0)
//   out      = gate_out * up_out
// commit 3: linear_beta <= 0 means unset and up passes through.  Arithmetic is
// fp32 and results go straight to the output buffer.  The masked kernel reads
// expert_num_tokens and never touches padded rows.
//
// Bandwidth-bound: every thread moves 16-byte vectors (8 bf16); the scalar
// math (one hardware 2^x per exponential, one reciprocal per element, relative
// error about 1e-6) lives with the other SituGLU users in lmoe_internal.cuh.
#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

__device__ __forceinline__ uint4 situ8(const uint4& g, const uint4& u, const SituParams& p) {
  uint4 o;
  o.x = situ2(g.x, u.x, p);
  o.y = situ2(g.y, u.y, p);
  o.z = situ2(g.z, u.z, p);
  o.w = situ2(g.w, u.w, p);
  return o;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Rows [row0, row0 + nrows) of a [*, 2d] -> [*, d] problem, vpr = d / 8.
__device__ __forceinline__ void situ_rows(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                                          long long row0, int nrows, int d, int vpr,
                                          const SituParams& p) {
  const int total = nrows * vpr;
  for (int j0 = threadIdx.x; j0 < total; j0 += kUnroll * kThreads) {
    uint4 g[kUnroll], u[kUnroll];
    long long oi[kUnroll];
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
      const int j = j0 + q * kThreads;
      oi[q] = -1;
      if (j < total) {
        const int r = j / vpr;
        const int c = j - r * vpr;
        const long long row = row0 + r;
        const uint16_t* src = in + row * (2LL * d) + (long long)c * 8;
        g[q] = ld_stream(reinterpret_cast<const uint4*>(src));
        u[q] = ld_stream(reinterpret_cast<const uint4*>(src + d));
        oi[q] = row * d + (long long)c * 8;
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll; ++q)
      if (oi[q] >= 0) *reinterpret_cast<uint4*>(out + oi[q]) = situ8(g[q], u[q], p);
  }
}

__global__ void __launch_bounds__(kThreads)
situ_dense_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, long long N,
                  int d, int rows_per_block, SituParams p) {
  pdl_trigger();
  pdl_wait();
  const long long row0 = (long long)blockIdx.x * rows_per_block;
  if (row0 >= N) return;
  const int nrows = (int)min((long long)rows_per_block, N - row0);
  situ_rows(in, out, row0, nrows, d, d / 8, p);
}

__global__ void __launch_bounds__(kThreads)
situ_masked_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out,
                   const int32_t* __restrict__ counts, int T_max, int d, int rows_per_block,
                   SituParams p) {
  pdl_trigger();
  pdl_wait();
  const int e = blockIdx.y;
  const int n = min(max(__ldg(counts + e), 0), T_max);
  const int r0 = blockIdx.x * rows_per_block;
  if (r0 >= n) return;
  const int nrows = min(rows_per_block, n - r0);
  situ_rows(in, out, (long long)e * T_max + r0, nrows, d, d / 8, p);
}

int rows_for(int d) {
  // about 4096 16-byte vectors (64 KiB of input) per block
  const int vpr = d / 8;
  return vpr >= 4096 ? 1 : 4096 / vpr;
}

}  // namespace

cudaError_t launch_situ(const uint16_t* in, uint16_t* out, long long N, int d, float beta,
                        float lbeta, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  // at least two blocks per SM when there are enough rows
  const long long spread = (N + 2LL * num_sms() - 1) / (2LL * num_sms());
  const int rpb = (int)(spread < rows_for(d) ? (spread < 1 ? 1 : spread) : rows_for(d));
  const long long blocks = (N + rpb - 1) / rpb;
  return launch_k(situ_dense_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, s, in, out, N, d,
                  rpb, make_situ_params(beta, lbeta));
}

cudaError_t launch_masked_situ(const uint16_t* in, uint16_t* out, const int32_t* counts, int E,
                               int T_max, int d, float beta, float lbeta, cudaStream_t s) {
  if (E <= 0 || T_max <= 0) return cudaSuccess;
  const int rpb = min(rows_for(d), T_max);
  dim3 grid((unsigned)ceil_div(T_max, rpb), (unsigned)E);
  return launch_k(situ_masked_kernel, grid, dim3(kThreads), 0, s, in, out, counts, T_max, d, rpb,
                  make_situ_params(beta, lbeta));
}

}  // namespace lmoe
