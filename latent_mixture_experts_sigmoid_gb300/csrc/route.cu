// Single-group sigmoid top-k routing (DeepSeekV3 style).
//
// vLLM PR #50088, commit 1: with n_group == 1 and topk_group == 1, grouped
// top-k is plain top-k over all experts; kernels are dispatched from a
// compile-time (num_experts) tier list.  Here: a block of 4 warps per token
// for more than 128 experts and at most 512 tokens (latency: the decode
// sizes), and otherwise a warp per token, persistent, with the token rows
// staged in shared memory (throughput: the large batches).
// Commit 4: sigmoid scores of FP32 logits, e_score_correction_bias added for
// the selection only, weights from the unbiased scores, renormalised, times
// routed_scaling_factor.
//
// The selection key must be reproducible to the bit (the expert ids are
// compared exactly), so the sigmoid that decides it is a fixed sequence of
// IEEE fp32 operations (exact_sigmoid below).  Evaluating that sequence for
// all E experts would make the kernel issue-bound, so selection takes two
// passes:
//   A. a cheap key for every expert (in the block kernel ka = 1/(1 +
//      __expf(-x)) + b, packed with the expert index into one u32, key
//      truncated to 22 bits, index below; the warp kernel's tanh key is
//      described at that kernel), and a bound A: the k-th largest of a small
//      set of per-lane maxima of those keys (so at least k experts reach A),
//      found by a parallel rank count in shared memory (block kernel) or a
//      sort across the warp (warp kernel);
//   B. every expert whose cheap key lies within a proven error bound below A
//      is a candidate; candidates (a few more than k) get the exact
//      key, and each one's output slot is the number of candidates with a
//      larger exact key (ties go to the lower index).  More than 32
//      candidates (a row of tied logits) fall back to an exact selection over
//      all experts.
// Why the candidate set always holds the exact top-k: let |ka - key| <= D for
// every expert and let A be the truncated key of a packed value that at least
// k experts reach.  Those k have ka >= A, so at least k have key >= A - D;
// hence the k-th largest exact key K satisfies K >= A - D, and every member of
// the exact top-k has ka >= key - D >= K - D >= A - 2D.  D is bounded from the documented
// error of __expf (2 + floor(1.173|x|) ulp, |x| <= 87) and __fdividef (2 ulp):
// |s_fast - s| <= s(1-s) * 1.24e-5 + 3 ulp <= 3.5e-6, plus the exact
// sigmoid's own error (<= 3 ulp) and the rounding of the two bias additions
// (<= 2^-23 |key|).  The block kernel uses 2D = 1e-5 + 2^-20 * max(|A|, 1),
// about 2.5x that bound.
#include <atomic>

#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

// ---- the exact fp32 sigmoid ------------------------------------------------
// y = clamp(-x, -87, 88); n = rint(y*log2e); r = (y - n*ln2_hi) - n*ln2_lo;
// p = degree-7 Taylor polynomial of e^r (Horner, separate multiply and add);
// e^y = p * 2^n; s = 1 / (1 + e^y).  Every operation is an explicitly rounded
// intrinsic, so the compiler cannot contract or reorder it.
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.63p-1f;          // 355/512
constexpr float kLn2Lo = -0x1.bd0106p-13f;    // ln2 - 355/512, rounded
constexpr float kInvFact2 = 0x1p-1f;
constexpr float kInvFact3 = 0x1.555556p-3f;
constexpr float kInvFact4 = 0x1.555556p-5f;
constexpr float kInvFact5 = 0x1.111112p-7f;
constexpr float kInvFact6 = 0x1.6c16c2p-10f;
constexpr float kInvFact7 = 0x1.a01a02p-13f;

__device__ __forceinline__ float horner_step(float p, float r, float c) {
  return __fadd_rn(__fmul_rn(p, r), c);
}

__device__ __forceinline__ float exact_sigmoid(float x) {
  const float y = fminf(fmaxf(-x, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(y, kLog2e));
  float r = __fsub_rn(y, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = kInvFact7;
  p = horner_step(p, r, kInvFact6);
  p = horner_step(p, r, kInvFact5);
  p = horner_step(p, r, kInvFact4);
  p = horner_step(p, r, kInvFact3);
  p = horner_step(p, r, kInvFact2);
  p = horner_step(p, r, 1.0f);   // 1/1!
  p = horner_step(p, r, 1.0f);   // 1/0!
  const float two_n = __int_as_float(((int)n + 127) << 23);
  const float e = __fmul_rn(p, two_n);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}


// Monotone map float -> u32 (larger float -> larger integer; -0 < +0).
__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_orderable(uint32_t o) {
  const uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}

constexpr uint32_t kIdxBits = 10;  // E <= 1024
constexpr uint32_t kIdxMask = (1u << kIdxBits) - 1u;
constexpr unsigned FULL = 0xFFFFFFFFu;


// Exact key packed with the index: larger key first, then lower index first.
__device__ __forceinline__ unsigned long long pack_exact(float key, int e) {
  key = __fadd_rn(key, 0.0f);  // -0 -> +0
  return ((unsigned long long)orderable(key) << 32) |
         (unsigned long long)(0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ int expert_of(unsigned long long P) {
  return (int)(0xFFFFFFFFu - (uint32_t)P);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
  const uint32_t hi = __reduce_max_sync(FULL, (uint32_t)(v >> 32));
  const uint32_t lo = __reduce_max_sync(FULL, ((uint32_t)(v >> 32) == hi) ? (uint32_t)v : 0u);
  return ((unsigned long long)hi << 32) | lo;
}


// Threshold of pass B from the (truncated) cheap key of the k-th pick.
__device__ __forceinline__ float candidate_threshold(uint32_t a_k) {
  const float trunc_k = from_orderable(a_k & ~kIdxMask);
  return trunc_k - (1.0e-5f + 0x1p-20f * fmaxf(fabsf(trunc_k), 1.0f));
}

// ---- pass B exact stage for one warp -----------------------------------------
// `cand[0..total)` are the candidate experts (total <= 32).  Every candidate
// gets its exact key; its output position is the number of candidates with a
// larger key plus the number with an equal key and a lower index, so no sort
// network is needed.  Writes the top-k ids and weights of token t.  `row` is
// the token's logits (global or shared memory); `skey` is a 32-entry, 16-byte
// aligned scratch of this warp.
__device__ __forceinline__ void exact_order_and_write(const float* __restrict__ row,
                                                      const float* sbias, const int* cand,
                                                      int total, int k, int renorm, float rsf,
                                                      long long t, int lane, uint32_t* skey,
                                                      int32_t* __restrict__ ids,
                                                      float* __restrict__ weights) {
  uint32_t P = 0u;   // no finite key maps to 0
  float s = 0.0f;
  int e = 0;
  if (lane < total) {
    e = cand[lane];
    s = exact_sigmoid(row[e]);
    P = orderable(__fadd_rn(__fadd_rn(s, sbias ? sbias[e] : 0.0f), 0.0f));  // -0 -> +0
  }
  skey[lane] = P;
  __syncwarp();
  // entries of lanes >= total are 0 and count for nothing
  int rank = 0;
  const int jn = (total + 3) & ~3;
  for (int j = 0; j < jn; j += 4) {
    const uint4 a = *reinterpret_cast<const uint4*>(skey + j);
    rank += (a.x > P) + (a.y > P) + (a.z > P) + (a.w > P);
  }
  // equal keys (rare): the lower expert index goes first
  uint32_t same = __match_any_sync(FULL, P) & ~(1u << lane);
  if (lane < total) {
    while (same) {
      const int j = __ffs(same) - 1;
      same &= same - 1u;
      rank += cand[j] < e;
    }
  }
  const bool sel = lane < total && rank < k;
  float sum = sel ? s : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
  if (sel) {
    const float wv = renorm ? __fmul_rn(__fdiv_rn(s, sum), rsf) : __fmul_rn(s, rsf);
    ids[t * k + rank] = e;
    weights[t * k + rank] = wv;
  }
  __syncwarp();
}

// Weights and outputs of an exact selection already held as lane r = r-th pick.
__device__ __forceinline__ void write_selected(const float* __restrict__ row,
                                               unsigned long long P, int k, int renorm, float rsf,
                                               long long t, int lane, int32_t* __restrict__ ids,
                                               float* __restrict__ weights) {
  const float s = (lane < k) ? exact_sigmoid(row[expert_of(P)]) : 0.0f;
  float sum = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
  if (lane < k) {
    const float wv = renorm ? __fmul_rn(__fdiv_rn(s, sum), rsf) : __fmul_rn(s, rsf);
    ids[t * k + lane] = expert_of(P);
    weights[t * k + lane] = wv;
  }
}

// Largest exact packed key below `lastP` among this lane's experts.
template <int EPL>
__device__ __forceinline__ unsigned long long lane_best_exact(const float* __restrict__ row,
                                                              const float* sbias, int E, int base,
                                                              int stride, int lane,
                                                              unsigned long long lastP) {
  unsigned long long best = 0ull;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = base + lane + stride * i;
    if (e < E) {
      const unsigned long long p =
          pack_exact(__fadd_rn(exact_sigmoid(__ldg(row + e)), sbias ? sbias[e] : 0.0f), e);
      if (p < lastP && p > best) best = p;
    }
  }
  return best;
}

// ---- warp per token --------------------------------------------------------------
// One warp per token, tokens visited with a stride of all warps of the grid.
// Rows are staged in shared memory by cp.async in a ring of NSLOT rows per
// warp, so that NSLOT - 1 rows are in flight while one is processed (a warp
// handles only a few tokens, and one row in flight per warp leaves the copy
// latency exposed); padding slots hold the logit 0 and the bias -inf, so their
// cheap key is -inf, below every threshold (the threshold is clamped to a
// finite value).  Lane l owns the
// experts e = 128*c + 4*l + j (chunk c < C, j < 4): one 16-byte copy and one
// 16-byte shared load per chunk when E is a multiple of 4.
//
// Pass A uses a cheaper key than the block kernel, in a doubled scale:
//   ka2 = tanh(x/2) + 2b   (= 2 sigmoid(x) + 2b - 1 up to the error of tanh;
// the constant shift changes no comparison) with the hardware tanh (one MUFU
// operation per expert) and one fused multiply-add.  tanh.approx.f32 is
// documented with a maximum error near 2^-11; the window below allows 2^-9
// per key (four times that), and an exhaustive run over every finite fp32
// input on GB300 measured at most 2^-16.9 absolute.  Other error terms: the
// rounding of the fused add (2^-24 |ka2|) and the exact key's own error
// doubled (3 ulp of sigmoid plus the rounding of the bias add), all below
// 2^-20 max(|ka2|, 1).  So with D2 = 2^-9 + 2^-21 max(|A2|, 1) the
// candidate argument of the file header holds in the doubled scale.
//
// The bound A2 is first the k-th largest of the 32 lane maxima (a bitonic sort
// across the warp); in the rare case that leaves more than 32 candidates it is
// refined to the k-th largest of 64 group maxima (j < 2 and j >= 2 of every
// lane), and only then does the exact fallback run.
// Seven warps a block and four blocks an SM: 28 resident warps, the most that
// the two-row rings (7 KB a warp) and 72 registers a thread allow together.
constexpr int kWarpsPerBlock = 7;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Per-lane direction bits of the 15 compare-exchange steps of a 32-wide
// ascending bitonic sort: bit s set = keep the smaller value at step s.
__device__ __forceinline__ uint32_t sort32_directions(int lane) {
  uint32_t m = 0;
  int s = 0;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1, ++s)
      if (((lane & stride) == 0) == ((lane & size) == 0)) m |= 1u << s;
  return m;
}

// Ascending bitonic sort of one value per lane across the warp.
__device__ __forceinline__ float warp_sort32(float v, uint32_t dirs) {
  int s = 0;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1, ++s) {
      const float p = __shfl_xor_sync(FULL, v, stride);
      v = ((dirs >> s) & 1u) ? fminf(v, p) : fmaxf(v, p);
    }
  }
  return v;
}

// Ascending bitonic sort of the 64 values (v0, v1) of a warp, element index 2*lane + g.
__device__ __forceinline__ void warp_sort64(float& v0, float& v1, int lane) {
  const int i2 = 2 * lane;
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 1; stride >>= 1) {
      const float p0 = __shfl_xor_sync(FULL, v0, stride >> 1);
      const float p1 = __shfl_xor_sync(FULL, v1, stride >> 1);
      // keep the smaller value where (lower half) == (ascending block)
      const bool kmin = ((i2 & stride) == 0) == ((i2 & size) == 0);
      v0 = kmin ? fminf(v0, p0) : fmaxf(v0, p0);
      v1 = kmin ? fminf(v1, p1) : fmaxf(v1, p1);
    }
    // stride 1: the lane's own pair
    const float lo = fminf(v0, v1), hi = fmaxf(v0, v1);
    const bool asc = (i2 & size) == 0;
    v0 = asc ? lo : hi;
    v1 = asc ? hi : lo;
  }
}

// The 16th largest of one value per lane: each half of the warp sorted (the
// lower ascending, the upper descending, the first four stages of the 32-wide
// network), the larger of each cross pair kept in the upper half (these are the
// 16 largest), and their minimum.
__device__ __forceinline__ float warp_kth16(float v, uint32_t dirs, int lane) {
  int s = 0;
#pragma unroll
  for (int size = 2; size <= 16; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1, ++s) {
      const float p = __shfl_xor_sync(FULL, v, stride);
      v = ((dirs >> s) & 1u) ? fminf(v, p) : fmaxf(v, p);
    }
  }
  const float p = __shfl_xor_sync(FULL, v, 16);
  const uint32_t o = __reduce_max_sync(FULL, (lane & 16) ? ~orderable(fmaxf(v, p)) : 0u);
  return from_orderable(~o);
}

__device__ __forceinline__ float candidate_threshold2(float a2) {
  return a2 - (0x1p-8f + 0x1p-20f * fmaxf(fabsf(a2), 1.0f));
}

// Largest exact packed key below `lastP` among this lane's experts (chunk layout).
template <int C>
__device__ __forceinline__ unsigned long long lane_best_exact_chunk(const float* row,
                                                                    const float* sbias, int E,
                                                                    int lane,
                                                                    unsigned long long lastP) {
  unsigned long long best = 0ull;
#pragma unroll 1
  for (int i = 0; i < 4 * C; ++i) {
    const int e = 128 * (i >> 2) + 4 * lane + (i & 3);
    if (e < E) {
      const unsigned long long p = pack_exact(__fadd_rn(exact_sigmoid(row[e]), sbias[e]), e);
      if (p < lastP && p > best) best = p;
    }
  }
  return best;
}

// Start the copy of token tt's row into `dst` (nothing for tt >= T), then close the group.
template <int C, bool VEC>
__device__ __forceinline__ void stage_row(float* dst, const float* __restrict__ logits,
                                          long long tt, int T, int E, long long ld, int lane) {
  if (tt < T) {
    const float* rr = logits + tt * ld;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int e0 = 128 * c + 4 * lane;
      if (VEC) {
        if (e0 < E) cp_async16(dst + e0, rr + e0);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j < E) cp_async4(dst + e0 + j, rr + e0 + j);
      }
    }
  }
  cp_async_commit();
}

// ring depth and the blocks per SM the register budget is sized for
constexpr int kRouteSlots = 2;
constexpr int kRouteMinBlocks = 4;   // (three for 8 chunks: their rings take 8 KB a warp)

template <int C, int NSLOT>
constexpr size_t warp_kernel_smem() {
  return (size_t)kWarpsPerBlock * NSLOT * 128 * C * sizeof(float);
}

template <int C, bool VEC, int NSLOT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, C >= 8 ? 3 : kRouteMinBlocks)
route_warp_kernel(const float* __restrict__ logits, long long ld, const float* __restrict__ bias,
                  int T, int E, int k, int renorm, float rsf, int32_t* __restrict__ ids,
                  float* __restrict__ weights) {
  constexpr int EW = 128 * C;
  extern __shared__ __align__(16) float srow_all[];   // [warp][slot][EW]
  __shared__ __align__(16) float sbias[EW];
  __shared__ int scand[kWarpsPerBlock][32];
  __shared__ __align__(16) uint32_t skey[kWarpsPerBlock][32];
  pdl_trigger();
  if (E < EW) {
    // padding slots (never written by the copies) hold 0
    for (int i = threadIdx.x; i < kWarpsPerBlock * NSLOT * EW / 4; i += blockDim.x)
      reinterpret_cast<float4*>(srow_all)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  // the bias is a model parameter: read while the preceding kernel drains
  for (int e = threadIdx.x; e < EW; e += blockDim.x)
    sbias[e] = e < E ? (bias ? __ldg(bias + e) : 0.0f) : -INFINITY;
  pdl_wait();
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  float* const ring = srow_all + (size_t)warp * NSLOT * EW;
  const long long step = (long long)gridDim.x * kWarpsPerBlock;
  const long long t0 = (long long)blockIdx.x * kWarpsPerBlock + warp;
  const f32x2 half2 = f2_splat(0.5f), two2 = f2_splat(2.0f);
  const uint32_t dirs = sort32_directions(lane);
#pragma unroll
  for (int p = 0; p < NSLOT - 1; ++p)
    stage_row<C, VEC>(ring + p * EW, logits, t0 + p * step, T, E, ld, lane);
  int slot = 0, fill = NSLOT - 1;
  for (long long t = t0; t < T; t += step) {
    stage_row<C, VEC>(ring + fill * EW, logits, t + (NSLOT - 1) * step, T, E, ld, lane);
    cp_async_wait<NSLOT - 1>();
    __syncwarp();
    const float* row = ring + slot * EW;
    if (++slot == NSLOT) slot = 0;
    if (++fill == NSLOT) fill = 0;
    // pass A: doubled cheap keys as pairs (elements 4c, 4c+1 | 4c+2, 4c+3), two
    // group maxima per lane
    f32x2 kp[2 * C];
    float g0 = -INFINITY, g1 = -INFINITY;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int e0 = 128 * c + 4 * lane;
      const float4 x = *reinterpret_cast<const float4*>(row + e0);
      const float4 b = *reinterpret_cast<const float4*>(sbias + e0);
      const f32x2 h01 = f2_mul(f2_make(__float_as_uint(x.x), __float_as_uint(x.y)), half2);
      const f32x2 h23 = f2_mul(f2_make(__float_as_uint(x.z), __float_as_uint(x.w)), half2);
      kp[2 * c] = f2_fma(f2_make(__float_as_uint(b.x), __float_as_uint(b.y)), two2,
                         f2_make(__float_as_uint(tanh_fast(f2_lo(h01))),
                                 __float_as_uint(tanh_fast(f2_hi(h01)))));
      kp[2 * c + 1] = f2_fma(f2_make(__float_as_uint(b.z), __float_as_uint(b.w)), two2,
                             f2_make(__float_as_uint(tanh_fast(f2_lo(h23))),
                                     __float_as_uint(tanh_fast(f2_hi(h23)))));
      g0 = fmaxf(g0, fmaxf(f2_lo(kp[2 * c]), f2_hi(kp[2 * c])));
      g1 = fmaxf(g1, fmaxf(f2_lo(kp[2 * c + 1]), f2_hi(kp[2 * c + 1])));
    }
    const float gm = fmaxf(g0, g1);
    float thr = candidate_threshold2(k == 16 ? warp_kth16(gm, dirs, lane)
                                             : __shfl_sync(FULL, warp_sort32(gm, dirs), 32 - k));
    thr = fmaxf(thr, -0x1p127f);   // finite: padding keys (-inf) stay below it
    // candidate bits: the sign of (key - thr) of every element, shifted in from
    // the last element down, so that bit i ends up clear for a candidate
    uint32_t below = 0u;
    {
      const f32x2 nthr = f2_splat(-thr);
#pragma unroll
      for (int j = 2 * C - 1; j >= 0; --j) {
        const f32x2 d = f2_add(kp[j], nthr);
        below = __funnelshift_l((uint32_t)(d >> 32), below, 1);
        below = __funnelshift_l((uint32_t)d, below, 1);
      }
    }
    uint32_t cmask = ~below & (4 * C >= 32 ? 0xFFFFFFFFu : (1u << (4 * C)) - 1u);
    int total = (int)__reduce_add_sync(FULL, (uint32_t)__popc(cmask));
    if (total > 32) {
      // refine the bound with the 64 group maxima
      warp_sort64(g0, g1, lane);
      const int kpos = 64 - k;
      thr = fmaxf(candidate_threshold2(__shfl_sync(FULL, (kpos & 1) ? g1 : g0, kpos >> 1)),
                  -0x1p127f);
      cmask = 0;
#pragma unroll
      for (int i = 0; i < 4 * C; ++i) {
        const float v = (i & 1) ? f2_hi(kp[i >> 1]) : f2_lo(kp[i >> 1]);
        if (v >= thr) cmask |= 1u << i;
      }
      total = (int)__reduce_add_sync(FULL, (uint32_t)__popc(cmask));
    }
    // fewer than k candidates only where keys overflow to -inf: the exact fallback
    if (total <= 32 && total >= k) {
      const int ccount = __popc(cmask);
      int incl = ccount;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = incl - ccount;
      while (cmask) {
        const int i = __ffs(cmask) - 1;
        cmask &= cmask - 1u;
        scand[warp][pos++] = 128 * (i >> 2) + 4 * lane + (i & 3);
      }
      __syncwarp();
      exact_order_and_write(row, sbias, scand[warp], total, k, renorm, rsf, t, lane, skey[warp],
                            ids, weights);
    } else {
      // fallback (rows of tied logits): exact selection over all experts, one pick per round
      unsigned long long lastP = ~0ull, P = 0ull;
      for (int r = 0; r < k; ++r) {
        const unsigned long long m =
            warp_max_u64(lane_best_exact_chunk<C>(row, sbias, E, lane, lastP));
        if (lane == r) P = m;
        lastP = m;
      }
      write_selected(row, P, k, renorm, rsf, t, lane, ids, weights);
    }
    __syncwarp();
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- block per token ---------------------------------------------------------
// W warps per token (E > 32*W); warp w owns experts e = 32*w + lane + 32*W*i.  Instead of
// merging sorted lists round by round, the block takes as its pass-B bound the
// k-th largest of the W*32 lane maxima of the cheap keys: at least k experts
// reach it, which is all the candidate argument above needs, and when the
// top-k sit in distinct lanes it equals the k-th largest cheap key.  It is
// found in parallel: every thread counts the lane maxima above its own.
template <int EPL, int W>
__global__ void __launch_bounds__(W * 32)
route_block_kernel(const float* __restrict__ logits, long long ld, const float* __restrict__ bias,
                   int T, int E, int k, int renorm, float rsf, int32_t* __restrict__ ids,
                   float* __restrict__ weights) {
  __shared__ __align__(16) uint32_t smax[W * 32];
  __shared__ int scnt[W];
  __shared__ int scand[32];
  __shared__ uint32_t sak;
  __shared__ unsigned long long spick[W];
  __shared__ __align__(16) uint32_t skey[32];
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int base = 32 * warp, stride = 32 * W;
  // per-lane constants for every token of this block: bias and packed index
  float lb[EPL];
  uint32_t lidx[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = base + lane + stride * i;
    lb[i] = (e < E && bias) ? __ldg(bias + e) : 0.0f;
    lidx[i] = kIdxMask - (uint32_t)e;
  }

  // this lane's logits of the block's next token are loaded one token ahead
  float xn[EPL];
  auto load_row = [&](long long tt) {
    const float* rr = logits + tt * ld;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = base + lane + stride * i;
      xn[i] = (tt < T && e < E) ? __ldg(rr + e) : 0.0f;
    }
  };
  load_row(blockIdx.x);
  for (long long t = blockIdx.x; t < T; t += gridDim.x) {
    const float* row = logits + t * ld;
    float xv[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) xv[i] = xn[i];
    load_row(t + gridDim.x);
    // pass A: cheap keys and this lane's maximum (every lane owns >= 1 expert: E > 32*W).
    // No clamp is needed: __expf saturates to 0 or inf beyond |x| ~ 88 and the
    // key then differs from the exact one by less than 1e-38.
    float ka[EPL];
    uint32_t cmax = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = base + lane + stride * i;
      ka[i] = -INFINITY;
      if (e < E) {
        ka[i] = __fdividef(1.0f, 1.0f + __expf(-xv[i])) + lb[i];
        cmax = max(cmax, (orderable(ka[i]) & ~kIdxMask) | lidx[i]);
      }
    }
    smax[threadIdx.x] = cmax;
    __syncthreads();
    // rank of this lane maximum among all W*32 (packed values are distinct)
    int above = 0;
#pragma unroll
    for (int j = 0; j < W * 32; j += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(smax + j);
      above += (v.x > cmax) + (v.y > cmax) + (v.z > cmax) + (v.w > cmax);
    }
    if (above == k - 1) sak = cmax;
    __syncthreads();
    const float thr = candidate_threshold(sak);
    uint32_t cmask = 0;
    int ccount = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (ka[i] >= thr) { cmask |= 1u << i; ++ccount; }
    int incl = ccount;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) scnt[warp] = incl;
    __syncthreads();
    int total = 0, before = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      if (w < warp) before += scnt[w];
      total += scnt[w];
    }
    if (total <= 32) {
      int pos = before + incl - ccount;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (cmask & (1u << i)) scand[pos++] = base + lane + stride * i;
      __syncthreads();
      if (warp == 0)
        exact_order_and_write(row, bias, scand, total, k, renorm, rsf, t, lane, skey, ids,
                              weights);
    } else {
      // fallback: exact selection over all experts, one pick per round
      unsigned long long lastP = ~0ull, P = 0ull;
      for (int r = 0; r < k; ++r) {
        const unsigned long long m =
            warp_max_u64(lane_best_exact<EPL>(row, bias, E, base, stride, lane, lastP));
        if (lane == 0) spick[warp] = m;
        __syncthreads();
        unsigned long long best = 0ull;
#pragma unroll
        for (int w = 0; w < W; ++w) best = spick[w] > best ? spick[w] : best;
        __syncthreads();
        if (lane == r) P = best;
        lastP = best;
      }
      if (warp == 0) write_selected(row, P, k, renorm, rsf, t, lane, ids, weights);
    }
    __syncthreads();
  }
}

template <int C, bool VEC>
cudaError_t launch_warp_tier(const float* logits, long long ld, const float* bias, int T, int E,
                             int k, int renorm, float rsf, int32_t* ids, float* w, cudaStream_t s) {
  constexpr size_t smem = warp_kernel_smem<C, kRouteSlots>();
  // resident blocks per SM, per device (the shared-memory attribute is set on
  // each device once, before its first launch)
  static std::atomic<int> per_sm_of[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int per_sm = per_sm_of[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int n = 0;
    if (cudaFuncSetAttribute(route_warp_kernel<C, VEC, kRouteSlots>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return cudaGetLastError();
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, route_warp_kernel<C, VEC, kRouteSlots>,
                                                      kWarpsPerBlock * 32, smem) != cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
    per_sm_of[dev].store(n, std::memory_order_relaxed);
  }
  const long long need = ((long long)T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const long long cap = (long long)num_sms() * per_sm;
  const int blocks = (int)(need < cap ? need : cap);
  return launch_k(route_warp_kernel<C, VEC, kRouteSlots>, dim3(blocks), dim3(kWarpsPerBlock * 32),
                  smem, s, logits, ld, bias, T, E, k, renorm, rsf, ids, w);
}

template <int C>
cudaError_t launch_warp_chunks(const float* logits, long long ld, const float* bias, int T, int E,
                               int k, int renorm, float rsf, int32_t* ids, float* w,
                               cudaStream_t s) {
  // 16-byte row loads need every row to start on a 16-byte boundary
  if (E % 4 == 0 && ld % 4 == 0)
    return launch_warp_tier<C, true>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
  return launch_warp_tier<C, false>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
}

template <int EPL, int W>
cudaError_t launch_block_tier(const float* logits, long long ld, const float* bias, int T, int E,
                              int k, int renorm, float rsf, int32_t* ids, float* w,
                              cudaStream_t s) {
  // persistent: as many blocks as fit on the GPU at once loop over the tokens
  // (bias loaded once per block, next token's logits prefetched)
  static std::atomic<int> per_sm_of[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int per_sm = per_sm_of[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, route_block_kernel<EPL, W>, W * 32, 0) !=
            cudaSuccess || n < 1)
      n = 4;
    per_sm = n;
    per_sm_of[dev].store(n, std::memory_order_relaxed);
  }
  const long long cap = (long long)num_sms() * per_sm;
  const int grid = (int)(T < cap ? T : cap);
  return launch_k(route_block_kernel<EPL, W>, dim3(grid), dim3(W * 32), 0, s, logits, ld, bias, T,
                  E, k, renorm, rsf, ids, w);
}

}  // namespace

// Dispatch.  E > 128 and few tokens: a block of 4 warps per token (latency);
// otherwise a warp per token, C = ceil(E / 128) chunks of four experts per lane.
constexpr int kBlockMaxT = 512;

cudaError_t launch_route(const float* logits, long long ld, const float* bias, int T, int E, int k,
                         int renorm, float rsf, int32_t* ids, float* w, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (E > 128 && T <= kBlockMaxT) {
    if (E <= 256) return launch_block_tier<2, 4>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
    if (E <= 512) return launch_block_tier<4, 4>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
    if (E <= 896) return launch_block_tier<7, 4>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
    return launch_block_tier<8, 4>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
  }
  if (E <= 128) return launch_warp_chunks<1>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
  if (E <= 256) return launch_warp_chunks<2>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
  if (E <= 512) return launch_warp_chunks<4>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
  if (E <= 896) return launch_warp_chunks<7>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
  return launch_warp_chunks<8>(logits, ld, bias, T, E, k, renorm, rsf, ids, w, s);
}

}  // namespace lmoe
