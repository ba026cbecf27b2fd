// Host interface of the permutation / scatter / combine / reduction kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

// The experts of a permutation split by token count (MXFP4 experts): experts
// with at least heavy_min tokens are heavy when there are at least min_heavy
// of them (else none is), the others with tokens light.
// light [E]: light[0 .. *n_light - 1] the light experts in expert order;
// h_expert / h_count / h_offset [H]: the heavy experts (expert, count, first
// row) in the first #heavy slots, count 0 in the others; h_prefix [H+1]: the
// grouped GEMM's tile prefix over the H slots (ceil(count / tile) token tiles
// a heavy expert).  H >= T*k / heavy_min.
struct HeavySplit {
  int heavy_min, min_heavy, H, tile;
  int32_t *light, *n_light, *h_expert, *h_count, *h_offset, *h_prefix;
};

// Scratch bytes launch_permute needs for T tokens and E experts.
size_t permute_scratch_bytes(int T, int E);

// ids [T,k] -> counts [E], offsets [E+1], tile_prefix [E+1] (prefix of
// ceil(count/tile)), row_of [T,k], tok_of_row [T*k].  E <= 1024.  An id
// outside [0, E) is read as 0 and, if err is given, recorded there
// (kErrExpertId) by the first pass.  split (optional): the experts also
// split by count.
cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int tile, void* scratch,
                           int32_t* counts, int32_t* offsets, int32_t* tile_prefix,
                           int32_t* row_of, int32_t* tok_of_row, int* err, cudaStream_t s,
                           const HeavySplit* split = nullptr);

// launch_permute followed by launch_scatter_rows in one launch of T blocks,
// for T <= 256, E <= 1024, k <= 32 (the small-T path).  active (optional,
// needs tile >= T): active[i] = the i-th expert with a nonzero count, for
// i < tile_prefix[E].  split (optional): the experts also split by count.
cudaError_t launch_permute_scatter_small(const int32_t* ids, int T, int k, int E, int tile,
                                         int32_t* counts, int32_t* offsets, int32_t* tile_prefix,
                                         int32_t* row_of, int32_t* tok_of_row, const uint16_t* Zb,
                                         const float* Zp, int S, long long split_stride,
                                         int ldz, int L, uint16_t* A, int32_t* active, int* err,
                                         cudaStream_t s, const HeavySplit* split = nullptr);

// A[row_of[t,j]] = Z[t] for j < k; Z from bf16 rows Zb ([T, L]) or from the sum
// of S fp32 partials Zp (split_stride elements apart, rows ldz >= L elements
// apart, Z in the first L columns).  L % 8 == 0, ldz % 4 == 0.
cudaError_t launch_scatter_rows(const uint16_t* Zb, const float* Zp, int S, long long split_stride,
                                int ldz, int T, int L, int k, const int32_t* row_of, uint16_t* A,
                                cudaStream_t s);

// out[t, c] = sum_s P[s*sstride + t*ldp + col0 + c] (s ascending), c < n, rows
// ldo apart.
cudaError_t launch_sum_splits_cols(const float* P, int S, long long sstride, int T, long long ldp,
                                   int col0, int n, long long ldo, float* out, cudaStream_t s);

// N[t] = bf16(RMSNorm(sum_j w[t,j] Y[row_of[t,j]]) * gamma).  L % 8 == 0, L <= 8192.
cudaError_t launch_combine_norm(const uint16_t* Y, const float* w, const int32_t* row_of, int T,
                                int k, int L, const uint16_t* gamma, float eps, uint16_t* N,
                                cudaStream_t s);

// out[i] = bf16(sum_s P[s][i] + a[i]) over n elements (n % 8 == 0); a is
// bf16(sum_s2 Q[s2][i]) when Q is given, add[i] when add is given, else 0.
cudaError_t launch_reduce_splits(const float* P, int S, long long sstride, const float* Q, int S2,
                                 long long qstride, const uint16_t* add, long long n,
                                 uint16_t* out, cudaStream_t s);

// out[T,d] = bf16(SituGLU(bf16(sum_s P[s]))) for a [T, 2d] partial GEMM output.
cudaError_t launch_reduce_situ(const float* P, int S, long long sstride, int T, int d, float beta,
                               float lbeta, uint16_t* out, cudaStream_t s);

}  // namespace lmoe
