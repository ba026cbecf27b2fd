// Data movement of the latent-MoE layer: token permutation into the
// expert-major layout, the scatter of the routed input into it, the top-k
// weighted combine fused with the latent RMSNorm, and the fixed-order
// reductions of split-K partials (with the fused SituGLU and epilogue add).
//
// Permutation (vLLM PR #50088, commits 2-3: the batched MoE layout with
// expert_num_tokens).  The layer stores it compactly: expert e owns rows
// offsets[e] .. offsets[e+1]-1, its (token, slot) pairs in ascending token
// order.  The order is fixed by the data, not by atomics: per 256-token block
// a shared-memory bitmap marks which tokens chose each expert; a token's rank
// inside an expert is the population count of the bits below it plus the
// counts of the earlier blocks.
//
// Combine + RMSNorm (vLLM PR #50088, commit 7: the routed output is summed
// before the output transform; vLLM latent_moe_runner page,
// _shard_up_proj_tail: transform.norm on the reduced latent):
//   C[t] = sum_j w[t,j] * Y[row_of[t,j]]   (fp32, j ascending)
//   N[t] = bf16(C[t] * rsqrt(mean(C[t]^2) + eps) * gamma)
#include "lmoe_internal.cuh"
#include "moe_data.cuh"

namespace lmoe {
namespace {

constexpr int kBlkTok = 256;     // tokens per permutation block
constexpr int kWords = kBlkTok / 32;

// Expert id of pair i.  Ids the library did not write itself (the pre-routed
// forward) may be out of range: such an id is read as expert 0, the same way
// by every pass, and the device error word records kErrExpertId.
__device__ __forceinline__ int expert_id(const int32_t* __restrict__ ids, long long i, int E,
                                         int* err) {
  const int e = __ldg(ids + i);
  if ((unsigned)e < (unsigned)E) return e;
  if (err) atomicCAS(err, 0, kErrExpertId);
  return 0;
}

// ---- permutation, pass 1: bitmaps and per-block counts -----------------------
__global__ void __launch_bounds__(kBlkTok)
perm_count_kernel(const int32_t* __restrict__ ids, int T, int k, int E,
                  uint32_t* __restrict__ bitmaps, int32_t* __restrict__ blk_cnt, int* err) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t bm[];   // [E][kWords]
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  const int t = b * kBlkTok + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = expert_id(ids, (long long)t * k + j, E, err);
      atomicOr(&bm[e * kWords + (threadIdx.x >> 5)], 1u << (threadIdx.x & 31));
    }
  }
  __syncthreads();
  uint32_t* gbm = bitmaps + (long long)b * E * kWords;
  for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) gbm[i] = bm[i];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kWords; ++w) c += __popc(bm[e * kWords + w]);
    blk_cnt[(long long)b * E + e] = c;
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* sh /* [32] */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = sh[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, si, o);
      if (lane >= o) si += n;
    }
    sh[lane] = si - s;                   // exclusive prefix of warp totals
    if (lane == 31) sh[32] = si;
  }
  __syncthreads();
  const int r = sh[warp] + incl - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

// ---- MXFP4 experts: split by token count -------------------------------------
// Called by every thread of one block of 1024 with its expert's count c
// (thread e = expert e, c = 0 for e >= E).  Experts with at least heavy_min
// tokens are heavy when there are at least min_heavy of them (else none is);
// the others with tokens are light.  light[0 .. *n_light - 1] the light
// experts (expert order); the first #heavy slots of h_expert / h_count /
// h_offset [H] the heavy ones (expert, count, first row), the other slots
// count 0; h_prefix [H+1] the grouped GEMM's tile prefix over the H slots
// (ceil(count / tile) token tiles a heavy expert).
__device__ void split_heavy_block(int c, int off, const HeavySplit& hs, int* sh) {
  const int e = threadIdx.x;
  bool heavy = c >= hs.heavy_min;
  int nh = 0, nl = 0, tiles = 0;
  const int hi = block_exclusive_scan(heavy ? 1 : 0, sh, &nh);
  if (nh < hs.min_heavy || nh > hs.H) {   // (nh > H cannot happen: H >= T*k / heavy_min)
    heavy = false;
    nh = 0;
  }
  const bool lite = c > 0 && !heavy;
  const int li = block_exclusive_scan(lite ? 1 : 0, sh, &nl);
  const int ht = block_exclusive_scan(heavy ? (c + hs.tile - 1) / hs.tile : 0, sh, &tiles);
  if (lite) hs.light[li] = e;
  if (heavy) {
    hs.h_expert[hi] = e;
    hs.h_count[hi] = c;
    hs.h_offset[hi] = off;
    hs.h_prefix[hi] = ht;
  }
  for (int j = nh + e; j < hs.H; j += blockDim.x) {
    hs.h_expert[j] = 0;
    hs.h_count[j] = 0;
    hs.h_offset[j] = 0;
  }
  for (int j = nh + e; j <= hs.H; j += blockDim.x) hs.h_prefix[j] = tiles;
  if (e == 0) hs.n_light[0] = nl;
}

// ---- permutation, pass 2: counts, offsets, tile prefix, block bases ----------
// One block of 1024 threads; expert e is handled by thread e (E <= 1024).
__global__ void __launch_bounds__(1024)
perm_scan_kernel(const int32_t* __restrict__ blk_cnt, int nblk, int E, int tile,
                 int32_t* __restrict__ blk_base, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ tile_prefix,
                 const HeavySplit hs) {
  pdl_trigger();
  pdl_wait();
  __shared__ int sh[33];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int b = 0; b < nblk; ++b) {
      const int c = blk_cnt[(long long)b * E + e];
      blk_base[(long long)b * E + e] = total;
      total += c;
    }
  }
  int all = 0, all_tiles = 0;
  const int off = block_exclusive_scan(e < E ? total : 0, sh, &all);
  const int ntile = (e < E) ? (total + tile - 1) / tile : 0;
  const int toff = block_exclusive_scan(ntile, sh, &all_tiles);
  if (e < E) {
    counts[e] = total;
    offsets[e] = off;
    tile_prefix[e] = toff;
    for (int b = 0; b < nblk; ++b) blk_base[(long long)b * E + e] += off;
  }
  if (e == 0) {
    offsets[E] = all;
    tile_prefix[E] = all_tiles;
  }
  if (hs.H > 0) split_heavy_block(e < E ? total : 0, off, hs, sh);
}

// ---- permutation in one block, for T <= 256 (one bitmap block) ---------------
// The three passes above fused: bitmaps, counts/offsets/tile prefix by a
// block scan, then every (token, slot) row.  1024 threads, E <= 1024.
__global__ void __launch_bounds__(1024)
perm_small_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int tile,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ tile_prefix, int32_t* __restrict__ row_of,
                  int32_t* __restrict__ tok_of_row, const HeavySplit hs, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t bm[1024 * kWords];
  __shared__ int soff[1024];
  __shared__ int sh[33];
  for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  const int t = threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = expert_id(ids, (long long)t * k + j, E, err);
      atomicOr(&bm[e * kWords + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
#pragma unroll
    for (int w = 0; w < kWords; ++w) c += __popc(bm[e * kWords + w]);
  }
  int all = 0, all_tiles = 0;
  const int off = block_exclusive_scan(c, sh, &all);
  const int toff = block_exclusive_scan(e < E ? (c + tile - 1) / tile : 0, sh, &all_tiles);
  if (e < E) {
    counts[e] = c;
    offsets[e] = off;
    tile_prefix[e] = toff;
    soff[e] = off;
  }
  if (e == 0) {
    offsets[E] = all;
    tile_prefix[E] = all_tiles;
  }
  if (hs.H > 0) split_heavy_block(e < E ? c : 0, off, hs, sh);
  __syncthreads();
  if (t < T) {
    const int w = t >> 5;
    const uint32_t below = (1u << (t & 31)) - 1u;
    for (int j = 0; j < k; ++j) {
      const int ej = expert_id(ids, (long long)t * k + j, E, nullptr);
      const uint32_t* m = bm + ej * kWords;
      int rank = __popc(m[w] & below);
      for (int i = 0; i < w; ++i) rank += __popc(m[i]);
      const int row = soff[ej] + rank;
      row_of[(long long)t * k + j] = row;
      tok_of_row[row] = t;
    }
  }
}

// ---- permutation, pass 3: row of every (token, slot) -------------------------
__global__ void __launch_bounds__(kBlkTok)
perm_rows_kernel(const int32_t* __restrict__ ids, int T, int k, int E,
                 const uint32_t* __restrict__ bitmaps, const int32_t* __restrict__ blk_base,
                 int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of_row) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int tl = threadIdx.x;
  const int t = b * kBlkTok + tl;
  if (t >= T) return;
  const uint32_t* gbm = bitmaps + (long long)b * E * kWords;
  const int w = tl >> 5;
  const uint32_t below = (1u << (tl & 31)) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = expert_id(ids, (long long)t * k + j, E, nullptr);
    const uint32_t* m = gbm + e * kWords;
    int rank = __popc(__ldg(m + w) & below);
    for (int i = 0; i < w; ++i) rank += __popc(__ldg(m + i));
    const int row = __ldg(blk_base + (long long)b * E + e) + rank;
    row_of[(long long)t * k + j] = row;
    tok_of_row[row] = t;
  }
}

// acc[0..7] += the 8 floats at P + s * stride + off for s = 0 .. S-1, added in
// ascending s; the loads of four splits are issued before any of their sums,
// so that a row of split partials costs about S/4 load latencies, not S.
__device__ __forceinline__ void sum8_splits(const float* __restrict__ P, int S, long long stride,
                                            long long off, float (&acc)[8]) {
  int s = 0;
  for (; s + 4 <= S; s += 4) {
    float4 a[4], c[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float4* p = reinterpret_cast<const float4*>(P + (s + b) * stride + off);
      a[b] = __ldg(p);
      c[b] = __ldg(p + 1);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      acc[0] += a[b].x; acc[1] += a[b].y; acc[2] += a[b].z; acc[3] += a[b].w;
      acc[4] += c[b].x; acc[5] += c[b].y; acc[6] += c[b].z; acc[7] += c[b].w;
    }
  }
  for (; s < S; ++s) {
    const float4* p = reinterpret_cast<const float4*>(P + s * stride + off);
    const float4 a = __ldg(p), c = __ldg(p + 1);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += c.x; acc[5] += c.y; acc[6] += c.z; acc[7] += c.w;
  }
}

// ---- permutation and scatter in one kernel, for small T (decode) -------------
// T blocks of 1024 threads (T <= 256, E <= 1024).  Every block rebuilds the
// whole counting sort of the T*k (token, slot) pairs in shared memory (bitmaps,
// counts, a block scan for the offsets), which for so few pairs costs less than
// a second launch; block 0 publishes counts, offsets, tile prefix and every
// row; block t then writes Z[t] (the fixed-order sum of the S fp32 split
// partials, or a bf16 row) into its k expert-major rows.
__global__ void __launch_bounds__(1024)
perm_scatter_small_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int tile,
                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                          int32_t* __restrict__ tile_prefix, int32_t* __restrict__ row_of,
                          int32_t* __restrict__ tok_of_row, const uint16_t* __restrict__ Zb,
                          const float* __restrict__ Zp, int S, long long split_stride, int ldz,
                          int L, uint16_t* __restrict__ A, int32_t* __restrict__ active,
                          const HeavySplit hs, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t bm[1024 * kWords];
  __shared__ int soff[1024];
  __shared__ int sh[33];
  __shared__ int srow[32];
  for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  if ((int)threadIdx.x < T) {
    const int tt = threadIdx.x;
    for (int j = 0; j < k; ++j) {
      const int e = expert_id(ids, (long long)tt * k + j, E, blockIdx.x == 0 ? err : nullptr);
      atomicOr(&bm[e * kWords + (tt >> 5)], 1u << (tt & 31));
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  int c = 0;
  if (e < E) {
#pragma unroll
    for (int w = 0; w < kWords; ++w) c += __popc(bm[e * kWords + w]);
  }
  int all = 0, all_tiles = 0;
  const int off = block_exclusive_scan(c, sh, &all);
  const int toff = block_exclusive_scan(e < E ? (c + tile - 1) / tile : 0, sh, &all_tiles);
  if (e < E) soff[e] = off;
  if (blockIdx.x == 0) {
    if (e < E) {
      counts[e] = c;
      offsets[e] = off;
      tile_prefix[e] = toff;
      // with tile >= every count an active expert owns exactly one tile, so
      // its tile offset is its rank among the active experts
      if (active && c > 0) active[toff] = e;
    }
    if (e == 0) {
      offsets[E] = all;
      tile_prefix[E] = all_tiles;
    }
    if (hs.H > 0) split_heavy_block(e < E ? c : 0, off, hs, sh);
  }
  __syncthreads();
  const int t = blockIdx.x;
  if ((int)threadIdx.x < k) {
    const int j = threadIdx.x;
    const int ej = expert_id(ids, (long long)t * k + j, E, nullptr);
    const uint32_t* m = bm + ej * kWords;
    const int w = t >> 5;
    int rank = __popc(m[w] & ((1u << (t & 31)) - 1u));
    for (int i = 0; i < w; ++i) rank += __popc(m[i]);
    const int row = soff[ej] + rank;
    row_of[(long long)t * k + j] = row;
    tok_of_row[row] = t;
    srow[j] = row;
  }
  __syncthreads();
  for (int v = threadIdx.x; v < L / 8; v += blockDim.x) {
    uint4 o;
    if (Zp) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      sum8_splits(Zp, S, split_stride, (long long)t * ldz + v * 8, acc);
      o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    } else {
      o = __ldg(reinterpret_cast<const uint4*>(Zb + (long long)t * L) + v);
    }
    for (int j = 0; j < k; ++j) reinterpret_cast<uint4*>(A + (long long)srow[j] * L)[v] = o;
  }
}

// ---- scatter of the routed input into the expert-major rows ------------------
// A[row_of[t, j], :] = Z[t, :] for every slot j, where Z[t] is either a bf16
// row or the bf16 rounding of the fixed-order sum of S fp32 split partials.
__global__ void __launch_bounds__(256)
scatter_rows_kernel(const uint16_t* __restrict__ Zb, const float* __restrict__ Zp, int S,
                    long long split_stride, int ldz, int L, int k,
                    const int32_t* __restrict__ row_of, uint16_t* __restrict__ A) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int nv = L / 8;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 o;
    if (Zp) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      sum8_splits(Zp, S, split_stride, (long long)t * ldz + v * 8, acc);
      o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    } else {
      o = __ldg(reinterpret_cast<const uint4*>(Zb + (long long)t * L) + v);
    }
    for (int j = 0; j < k; ++j) {
      const long long row = __ldg(row_of + (long long)t * k + j);
      reinterpret_cast<uint4*>(A + row * L)[v] = o;
    }
  }
}

// ---- combine + RMSNorm -------------------------------------------------------
// kMaxV: 8-element vectors per thread (L <= 8 * blockDim * kMaxV), a template
// parameter so that the accumulators of the common L <= 2048 take 8 registers
// and eight 256-thread blocks fit per SM.
template <int kMaxV>
__global__ void __launch_bounds__(256)
combine_norm_kernel(const uint16_t* __restrict__ Y, const float* __restrict__ w,
                    const int32_t* __restrict__ row_of, int k, int L,
                    const uint16_t* __restrict__ gamma, float eps, uint16_t* __restrict__ N) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int nv = L / 8;
  float acc[kMaxV][8];
  float ss = 0.0f;
#pragma unroll
  for (int q = 0; q < kMaxV; ++q) {
    const int v = threadIdx.x + q * blockDim.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[q][i] = 0.0f;
    if (v < nv) {
      for (int j = 0; j < k; ++j) {
        const float wj = __ldg(w + (long long)t * k + j);
        const long long row = __ldg(row_of + (long long)t * k + j);
        const uint4 y = __ldg(reinterpret_cast<const uint4*>(Y + row * L) + v);
        const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[q][2 * i] += wj * bf16_lo(yw[i]);
          acc[q][2 * i + 1] += wj * bf16_hi(yw[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += acc[q][i] * acc[q][i];
    }
  }
  // block reduction of the sum of squares
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    float s = lane < nw ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) red[0] = s;
  }
  __syncthreads();
  const float r = rsqrtf(red[0] / (float)L + eps);
#pragma unroll
  for (int q = 0; q < kMaxV; ++q) {
    const int v = threadIdx.x + q * blockDim.x;
    if (v < nv) {
      float g[8];
      if (gamma) {
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(gamma) + v);
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { g[2 * i] = bf16_lo(gw[i]); g[2 * i + 1] = bf16_hi(gw[i]); }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = 1.0f;
      }
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        pk[i] = pack_bf16x2(acc[q][2 * i] * r * g[2 * i], acc[q][2 * i + 1] * r * g[2 * i + 1]);
      reinterpret_cast<uint4*>(N + (long long)t * L)[v] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

// ---- fixed-order reduction of split-K partials -------------------------------
// out[r, c] = bf16( sum_s P[s, r, c] + a ), where a = bf16(sum_s2 Q[s2, r, c]) if
// Q is given, a = add[r, c] if add is given, else 0.
__global__ void __launch_bounds__(256)
reduce_splits_kernel(const float* __restrict__ P, int S, long long sstride,
                     const float* __restrict__ Q, int S2, long long qstride,
                     const uint16_t* __restrict__ add, long long n8, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < n8;
       v += (long long)gridDim.x * blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    sum8_splits(P, S, sstride, 8 * v, acc);
    if (Q) {
      float qa[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      sum8_splits(Q, S2, qstride, 8 * v, qa);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const uint32_t b2 = pack_bf16x2(qa[i], qa[i + 1]);   // the bf16 shared output
        acc[i] += bf16_lo(b2);
        acc[i + 1] += bf16_hi(b2);
      }
    } else if (add) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(add) + v);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) { acc[2 * i] += bf16_lo(aw[i]); acc[2 * i + 1] += bf16_hi(aw[i]); }
    }
    reinterpret_cast<uint4*>(out)[v] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

// SituGLU of split-K partials of a [T, 2d] GEMM output: G = bf16(sum_s P)
// (gate = columns 0..d-1, up = d..2d-1), out[T, d] = bf16(SituGLU(G)).
__global__ void __launch_bounds__(256)
reduce_situ_kernel(const float* __restrict__ P, int S, long long sstride, int T, int d,
                   SituParams sp, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const long long n8 = (long long)T * (d / 8);
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < n8;
       v += (long long)gridDim.x * blockDim.x) {
    const long long t = v / (d / 8);
    const int c = (int)(v - t * (d / 8)) * 8;
    float g[8] = {0, 0, 0, 0, 0, 0, 0, 0}, u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    sum8_splits(P, S, sstride, t * (2LL * d) + c, g);
    sum8_splits(P, S, sstride, t * (2LL * d) + c + d, u);
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t gb = pack_bf16x2(g[2 * i], g[2 * i + 1]);
      const uint32_t ub = pack_bf16x2(u[2 * i], u[2 * i + 1]);
      pk[i] = situ2(gb, ub, sp);
    }
    reinterpret_cast<uint4*>(out + t * d + c)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

int grid_for(long long n, int threads) {
  const long long b = (n + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 16;
  return (int)(b < cap ? (b < 1 ? 1 : b) : cap);
}

}  // namespace

static bool valid_split(const HeavySplit& h) {
  return h.H >= 1 && h.heavy_min >= 1 && h.tile >= 1 && h.light && h.n_light && h.h_expert &&
         h.h_count && h.h_offset && h.h_prefix;
}

size_t permute_scratch_bytes(int T, int E) {
  const long long nblk = (T + kBlkTok - 1) / kBlkTok;
  return (size_t)(nblk * E * kWords * 4 + 2 * nblk * E * 4);
}

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int tile, void* scratch,
                           int32_t* counts, int32_t* offsets, int32_t* tile_prefix,
                           int32_t* row_of, int32_t* tok_of_row, int* err, cudaStream_t s,
                           const HeavySplit* split) {
  const int nblk = (T + kBlkTok - 1) / kBlkTok;
  HeavySplit hs{};
  if (split) {
    if (!valid_split(*split)) return cudaErrorInvalidValue;
    hs = *split;
  }
  if (nblk == 1)
    return launch_k(perm_small_kernel, dim3(1), dim3(1024), 0, s, ids, T, k, E, tile, counts,
                    offsets, tile_prefix, row_of, tok_of_row, hs, err);
  uint32_t* bitmaps = reinterpret_cast<uint32_t*>(scratch);
  int32_t* blk_cnt = reinterpret_cast<int32_t*>(bitmaps + (size_t)nblk * E * kWords);
  int32_t* blk_base = blk_cnt + (size_t)nblk * E;
  const size_t sm = (size_t)E * kWords * 4;
  cudaError_t e = cudaFuncSetAttribute(perm_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sm);
  if (e != cudaSuccess) return e;
  e = launch_k(perm_count_kernel, dim3(nblk), dim3(kBlkTok), sm, s, ids, T, k, E, bitmaps, blk_cnt,
               err);
  if (e != cudaSuccess) return e;
  e = launch_k(perm_scan_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)blk_cnt, nblk, E,
               tile, blk_base, counts, offsets, tile_prefix, hs);
  if (e != cudaSuccess) return e;
  return launch_k(perm_rows_kernel, dim3(nblk), dim3(kBlkTok), 0, s, ids, T, k, E,
                  (const uint32_t*)bitmaps, (const int32_t*)blk_base, row_of, tok_of_row);
}

cudaError_t launch_permute_scatter_small(const int32_t* ids, int T, int k, int E, int tile,
                                         int32_t* counts, int32_t* offsets, int32_t* tile_prefix,
                                         int32_t* row_of, int32_t* tok_of_row, const uint16_t* Zb,
                                         const float* Zp, int S, long long split_stride,
                                         int ldz, int L, uint16_t* A, int32_t* active, int* err,
                                         cudaStream_t s, const HeavySplit* split) {
  if (T > kBlkTok || E > 1024 || k > 32 || (active && tile < T)) return cudaErrorInvalidValue;
  HeavySplit hs{};
  if (split) {
    if (!valid_split(*split)) return cudaErrorInvalidValue;
    hs = *split;
  }
  return launch_k(perm_scatter_small_kernel, dim3(T), dim3(1024), 0, s, ids, T, k, E, tile, counts,
                  offsets, tile_prefix, row_of, tok_of_row, Zb, Zp, S, split_stride, ldz, L, A,
                  active, hs, err);
}

cudaError_t launch_scatter_rows(const uint16_t* Zb, const float* Zp, int S, long long split_stride,
                                int ldz, int T, int L, int k, const int32_t* row_of, uint16_t* A,
                                cudaStream_t s) {
  const int threads = L / 8 < 256 ? ((L / 8 + 31) / 32) * 32 : 256;
  return launch_k(scatter_rows_kernel, dim3(T), dim3(threads), 0, s, Zb, Zp, S, split_stride, ldz,
                  L, k, row_of, A);
}

// ---- columns of split-K partials summed into an fp32 matrix ------------------
// out[t, c] = sum_s P[s * sstride + t * ldp + col0 + c] (s ascending) for
// c < n, written with row stride ldo.  The router logits of the GEMM that
// shares its launch with the down-projection (their columns follow the
// latent ones in each partial row).
__global__ void __launch_bounds__(256)
sum_splits_cols_kernel(const float* __restrict__ P, int S, long long sstride, int T, long long ldp,
                       int col0, int n, long long ldo, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)T * n;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / n;
    const int c = (int)(i - t * n);
    const float* p = P + t * ldp + col0 + c;
    float acc = 0.0f;
    for (int sp = 0; sp < S; ++sp) acc += __ldg(p + sp * sstride);
    out[t * ldo + c] = acc;
  }
}

cudaError_t launch_sum_splits_cols(const float* P, int S, long long sstride, int T, long long ldp,
                                   int col0, int n, long long ldo, float* out, cudaStream_t s) {
  const long long total = (long long)T * n;
  const long long blocks = (total + 255) / 256;
  const int grid = (int)(blocks < 4096 ? blocks : 4096);
  return launch_k(sum_splits_cols_kernel, dim3(grid > 0 ? grid : 1), dim3(256), 0, s, P, S,
                  sstride, T, ldp, col0, n, ldo, out);
}

cudaError_t launch_combine_norm(const uint16_t* Y, const float* w, const int32_t* row_of, int T,
                                int k, int L, const uint16_t* gamma, float eps, uint16_t* N,
                                cudaStream_t s) {
  const int nv = L / 8;
  int threads = nv < 256 ? ((nv + 31) / 32) * 32 : 256;
  const int per = (nv + threads - 1) / threads;   // vectors per thread, <= 4 (L <= 8192)
  if (per <= 1)
    return launch_k(combine_norm_kernel<1>, dim3(T), dim3(threads), 0, s, Y, w, row_of, k, L,
                    gamma, eps, N);
  if (per == 2)
    return launch_k(combine_norm_kernel<2>, dim3(T), dim3(threads), 0, s, Y, w, row_of, k, L,
                    gamma, eps, N);
  return launch_k(combine_norm_kernel<4>, dim3(T), dim3(threads), 0, s, Y, w, row_of, k, L, gamma,
                  eps, N);
}

cudaError_t launch_reduce_splits(const float* P, int S, long long sstride, const float* Q, int S2,
                                 long long qstride, const uint16_t* add, long long n,
                                 uint16_t* out, cudaStream_t s) {
  const long long n8 = n / 8;
  return launch_k(reduce_splits_kernel, dim3(grid_for(n8, 256)), dim3(256), 0, s, P, S, sstride, Q,
                  S2, qstride, add, n8, out);
}

cudaError_t launch_reduce_situ(const float* P, int S, long long sstride, int T, int d, float beta,
                               float lbeta, uint16_t* out, cudaStream_t s) {
  const long long n8 = (long long)T * (d / 8);
  return launch_k(reduce_situ_kernel, dim3(grid_for(n8, 256)), dim3(256), 0, s, P, S, sstride, T, d,
                  make_situ_params(beta, lbeta), out);
}

}  // namespace lmoe
