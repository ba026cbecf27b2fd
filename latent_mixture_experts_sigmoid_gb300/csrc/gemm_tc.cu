// bf16 GEMMs of the latent-MoE layer on the 5th-generation tensor cores.
//
//   out[tok, f] = sum_c X[tok, c] * W[g*M_feat + f, c]   (+ add[tok, f])
//
// X holds token rows (K-major), W weight rows (K-major, PyTorch Linear
// layout).  One kernel serves every contraction of the layer:
//   * the latent down-projection and up-projection (dense; the up-projection
//     adds the shared-expert output in its epilogue, the beta-add of the
//     ``addmm_`` in the vLLM latent_moe_runner page, _shard_up_proj_tail);
//   * the grouped expert GEMM1 / GEMM2 over the expert-major row blocks
//     (group g owns token rows grp_offset[g] .. +grp_count[g]);
//   * the shared expert's two GEMMs.
//
// Design (sm_103a): a persistent, warp-specialised kernel.
//   warp 0      TMA producer: 64-wide K blocks of both operands, 128-byte
//               swizzle, into a ring of shared-memory stages (mbarrier
//               full/empty pairs);
//   warp 1      allocates TMEM and one elected thread issues tcgen05.mma
//               (kind::f16, bf16 in, fp32 accumulate, M = 128) into one of
//               two TMEM accumulators, committing stage releases and
//               accumulator-ready signals through tcgen05.commit;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator; with tokens on M the
//               rows are rounded to bf16 (after SituGLU or the bf16 addend
//               where asked) into a swizzled shared-memory staging buffer and
//               leave by a TMA bulk tensor store (a block of 32 valid rows)
//               or 4 rows x 128 bytes per 16-byte store instruction (a ragged
//               block); otherwise fp32 partials or bf16 values go straight out.
//   warp 6      (the weights-on-M GEMM1 + SituGLU instance only) a second MMA
//               issuer: the up halves, beside warp 1's gate halves.
// GEMMs with tokens on M and 256-row weight tiles run in clusters of two CTAs.
// A pair of units shares an operand: token tiles 2t and 2t+1 of a group
// against the same weight tile (each CTA loads one 128-row half of the weight
// tile with a TMA multicast into both CTAs' shared memory), or, for the last
// token tile of a group with an odd tile count, that token tile against weight
// tiles 2f and 2f+1 (CTA 0 multicasts the token tile).  A group of t token
// tiles and nfeat weight tiles thus gives exactly t * nfeat / 2 pair units.
// Each CTA's MMA commit releases the stage in both CTAs.
// The MMA's M side (128 rows) is either the tokens (large token counts) or
// the weight rows ("swap AB", up to 128 tokens: N = 16..128); the N side is
// the other operand.  Small dense problems split K across CTAs and write fp32
// partials that a reduction kernel sums in a fixed order.  The unit walk
// (decode_unit) also compiles for the host: lmoe_gemm_unit_walk lists it.
//
// Every wait on an mbarrier is bounded (clock64 deadline).  A wait that gives
// up records a code in the device error word, raises a CTA-wide abort flag,
// and the CTA drains its own in-flight copies and MMAs (again bounded),
// frees its TMEM and returns (CTA pairs meet at a cluster barrier first, so
// that neither leaves while the other may still write into it).
#include <cuda.h>

#include <mutex>
#include <vector>

#include "lmoe_internal.cuh"
#include "gemm_tc.cuh"

namespace lmoe {

__device__ int g_device_error = 0;

void* tensor_map_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
  });
  return fn;
}

namespace {

// K elements per ring stage: 64 (128-byte rows, 128-byte swizzle) or 32
// (64-byte rows, 64-byte swizzle: the same bytes in flight split into twice as
// many, half as large stages, so that less of the ring is held by the MMA
// currently reading it)
#ifndef LMOE_BK
#define LMOE_BK 64
#endif
constexpr int BK = LMOE_BK;
static_assert(BK == 64 || BK == 32, "stages are 64 or 32 K elements wide");
constexpr int kK16 = BK / 16;          // MMAs (K = 16 each) per stage and accumulator
constexpr int kMaxStages = 12 * 64 / BK;
constexpr int BM = 128;                // MMA M
constexpr int kThreads = 192;          // 6 warps (7 in the swap form, below)
// the swap form adds a seventh warp: the second MMA issuer (the up halves)
constexpr int kThreadsSwap = 224;
constexpr long long kWaitCycles = 1ll << 32;   // ~2 s at 2 GHz

// error codes written to g_device_error
enum : int { kErrProducer = 1, kErrMmaFull = 2, kErrMmaTmem = 3, kErrEpilogue = 4,
             kErrDrain = 5, kErrDone = 6 };
static_assert(kErrExpertId > kErrDone, "error codes are distinct");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed; false on deadline or abort.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      atomicCAS(&g_device_error, 0, code);
      *abort_flag = 1;
      return false;
    }
  }
}

// Fast path inline (the phase is usually complete already), bounded loop out of line.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int code) {
  return mbar_try_wait(bar, parity) || wait_bounded(bar, parity, abort_flag, code);
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// The same box into the same shared-memory offset of every CTA in `mask`,
// completing bytes on each CTA's barrier at `bar`'s offset.
__device__ __forceinline__ void tma_load_2d_mc(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                               int c0, int c1, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "h"(mask)
      : "memory");
}

// Bulk tensor store of a shared-memory box (laid out as the map's swizzle
// expects) to the global tensor at {c0, c1}; completion is tracked by bulk
// async-groups of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// every bulk store of this thread has finished reading its shared memory
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every bulk store of this thread has completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// order this thread's generic-proxy shared-memory writes before async-proxy reads
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, rows of BK * 2 bytes
// swizzled over that width (128-byte swizzle for 128-byte rows, 64-byte
// swizzle for 64-byte rows), 8-row groups 8 * BK * 2 bytes apart (stride
// byte offset), version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused with swizzling)
  d |= (uint64_t)((8 * BK * 2) >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)(BK == 64 ? 2 : 4) << 61;    // 128-byte / 64-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Arrive on the barrier at `bar`'s offset in every CTA of `mask` once the
// MMAs this thread issued so far have completed.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct Unit {
  int feat_tile;
  int kb0, kb1;
  int split;
  int tok_row0;   // first token row of the tile (in X / out rows)
  int nvalid;     // valid token rows in the tile
  int w_row0;     // first weight row of the tile
  int shareA;     // multicast: 1 = the pair shares the token tile, 0 = the weight tile
};

// Grouped GEMMs keep the per-group tables (tile prefix, token count, first
// row, and in pairs the prefix of pair units) in shared memory, copied once
// per CTA; a unit's group is found by a binary search there (the last g whose
// prefix is <= the unit's tile or pair index).
struct GroupTables {
  const int* prefix;   // [G+1]
  const int* count;    // [G]
  const int* first;    // [G]
  const int* pairs;    // [G+1] prefix of tiles * nfeat / 2 (CTA pairs only)
};

// Ints of shared memory the grouped tables take.
__host__ __device__ constexpr int group_table_ints(int G) { return 4 * G + 2; }

// Largest i in [0, n) with a[i] <= v (a non-decreasing, a[0] <= v).
__host__ __device__ __forceinline__ int last_leq(const int* a, int n, int v) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Work units of one CTA: with multicast a unit is a pair of token tiles (one
// per CTA of the cluster), so both CTAs walk the same unit sequence.
template <bool kPairs>
__host__ __device__ __forceinline__ int total_units(const GemmParams& p, const GroupTables& gt_tab,
                                                    int tok_tile, int nfeat) {
  if (kPairs && p.tile_prefix) return gt_tab.pairs[p.num_groups];
  const int tiles = p.tile_prefix ? gt_tab.prefix[p.num_groups]
                                  : (p.T_dense + tok_tile - 1) / tok_tile;
  // multicast pairs two units (tiles * nfeat is even: the launcher checks)
  return kPairs ? tiles * nfeat / 2 : tiles * nfeat * p.splits;
}

// Dense GEMMs with tokens on M walk their tiles in bands of kBand feature
// tiles: inside a band the feature tile changes fastest, then the token tile,
// so the 152 concurrent tiles share a band of weight tiles and a run of token
// tiles that both stay in L2 (for K = 7168: 8 x 3.7 MB + 19 x 1.8 MB).
constexpr int kBand = 8;

template <bool kPairs>
__host__ __device__ __forceinline__ Unit decode_unit(const GemmParams& p, const GroupTables& gt_tab,
                                                     int u, int tok_tile, int feat_tile, int nfeat,
                                                     int nkb, int rank) {
  Unit x;
  x.shareA = 0;
  x.split = u % p.splits;
  const int v = u / p.splits;
  int g = 0, t_in_g, count = p.T_dense, first = 0;
  if (kPairs) {
    // pair unit v of group g: first floor(t/2) * nfeat pairs of token tiles
    // (2tp + rank, same feature tile; dense GEMMs in bands of kBand feature
    // tiles as below), then for an odd t the last token tile against feature
    // tiles 2j + rank
    int t, j = v;
    if (p.tile_prefix) {
      g = last_leq(gt_tab.pairs, p.num_groups, v);
      j = v - gt_tab.pairs[g];
      t = gt_tab.prefix[g + 1] - gt_tab.prefix[g];
      count = gt_tab.count[g];
      first = gt_tab.first[g];
    } else {
      t = (p.T_dense + tok_tile - 1) / tok_tile;
    }
    const int nb = (t / 2) * nfeat;
    if (j < nb) {
      if (p.tile_prefix) {
        t_in_g = 2 * (j / nfeat) + rank;
        x.feat_tile = j % nfeat;
      } else {
        const int nt = t / 2;
        const int nbands = (nfeat + kBand - 1) / kBand;
        const int b = min(j / (nt * kBand), nbands - 1);
        const int rem = j - b * nt * kBand;
        const int fb = (b == nbands - 1) ? nfeat - kBand * (nbands - 1) : kBand;
        t_in_g = 2 * (rem / fb) + rank;
        x.feat_tile = b * kBand + rem % fb;
      }
    } else {
      x.shareA = 1;
      t_in_g = t - 1;
      x.feat_tile = 2 * (j - nb) + rank;
    }
  } else if (p.tile_prefix) {
    x.feat_tile = v % nfeat;
    const int gt = v / nfeat;
    g = last_leq(gt_tab.prefix, p.num_groups, gt);
    t_in_g = gt - gt_tab.prefix[g];
    count = gt_tab.count[g];
    first = gt_tab.first[g];
  } else if (p.tok_on_m) {
    const int ntok = (p.T_dense + tok_tile - 1) / tok_tile;
    const int nbands = (nfeat + kBand - 1) / kBand;
    const int b = min(v / (ntok * kBand), nbands - 1);
    const int rem = v - b * ntok * kBand;
    const int fb = (b == nbands - 1) ? nfeat - kBand * (nbands - 1) : kBand;
    t_in_g = rem / fb;
    x.feat_tile = b * kBand + rem % fb;
  } else {
    x.feat_tile = v % nfeat;
    t_in_g = v / nfeat;
  }
  x.nvalid = min(tok_tile, count - t_in_g * tok_tile);
  x.tok_row0 = first + t_in_g * tok_tile;
  x.w_row0 = g * p.M_feat + x.feat_tile * (p.fuse_situ ? BM : feat_tile);
  x.kb0 = (int)((long long)x.split * nkb / p.splits);
  x.kb1 = (int)((long long)(x.split + 1) * nkb / p.splits);
  return x;
}

// Forms of the kernel beyond the CTA pairs (one instance each: compiled into
// the regular form, even unused, their code measurably slowed it):
//   kFormSwap   weights on M, tokens on N, no pairs; every unit's weight tile
//               is two 128-row halves, the gate and up rows of the same 128
//               features, each multiplied into its own accumulator, so that
//               the epilogue applies SituGLU (p.fuse_situ is set).  Each half
//               has an MMA issuer of its own (warp 1: gate, warp 6: up): with
//               16 tokens on N an MMA is cheap to execute but not to issue
//               (about 1 us per decode step, bit-identical);
//   kFormStack  weights on M; weight rows from p.w2_row0 on come from a second
//               matrix (its own tensor map), stacked after the first.
enum : int { kFormRegular = 0, kFormSwap = 1, kFormStack = 2 };

// kPairs: the CTA-pair form (launched in clusters of two; p.mcast is set).
template <bool kPairs, int kForm>
__global__ void __launch_bounds__(kForm == kFormSwap ? kThreadsSwap : kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmO,
               const GemmParams p) {
  constexpr bool kSwap = kForm == kFormSwap;
  constexpr bool kStack = kForm == kFormStack;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int S = p.stages;
  const int bn = p.bn;
  const uint32_t a_bytes = BM * BK * 2;
  // weight rows per stage on the M side: one 128-row box, or the two halves
  const uint32_t w_bytes = (kSwap ? 2u : 1u) * a_bytes;
  const uint32_t stage_bytes =
      (p.tok_on_m ? a_bytes : w_bytes) + (uint32_t)bn * BK * 2;
  // TMEM columns between the two accumulators (a swap-form unit keeps its
  // gate and up accumulators side by side)
  const uint32_t acc_stride = kSwap ? 2u * (uint32_t)bn : (uint32_t)bn;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], done
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // grouped: prefix | count | first | pairs
  int* tab = reinterpret_cast<int*>(tmem_holder + 4);
  GroupTables tabs{tab, tab + p.num_groups + 1, tab + 2 * p.num_groups + 1,
                   tab + 3 * p.num_groups + 1};
  // epilogue staging: 4 warps x [32 rows][32 fp32], 16-byte chunks XOR-swizzled
  // by row: the 128-byte swizzle of a [32 rows][64 bf16] TMA box, so each
  // warp's buffer starts on a 1024-byte boundary
  float* stage_out = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(tab + (p.tile_prefix ? group_table_ints(p.num_groups) : 0)) +
       1023) &
      ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t done_bar = bar0 + 8u * (2 * S + 4);

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), (kPairs || kSwap) ? 2 : 1);   // both CTAs' / both issuers' MMAs release
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), kSwap ? 2 : 1);
      mbar_init(tempty_bar(a), 4 * 32);
    }
    mbar_init(done_bar, kSwap ? 2 : 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (p.tile_prefix) {
    // the tables are produced by the previous kernels: wait for them first
    pdl_wait();
    const int G = p.num_groups;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) tab[i] = __ldg(p.tile_prefix + i);
    for (int i = threadIdx.x; i < G; i += blockDim.x) {
      tab[G + 1 + i] = __ldg(p.grp_count + i);
      tab[2 * G + 1 + i] = __ldg(p.grp_offset + i);
    }
    if (kPairs) {
      // prefix of pair units per group (tiles * nfeat / 2), by warp 0 (G <= 1024: a run per lane)
      __syncthreads();
      if (warp == 0) {
        const int nf = p.fuse_situ ? (p.M_feat / 2) / BM : p.M_feat / bn;
        const int per = (G + 31) / 32;
        const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
        int sum = 0;
        for (int g = g0; g < g1; ++g) sum += (tab[g + 1] - tab[g]) * nf / 2;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += v;
        }
        int run = incl - sum;
        int* pairs = tab + 3 * G + 1;
        for (int g = g0; g < g1; ++g) {
          pairs[g] = run;
          run += (tab[g + 1] - tab[g]) * nf / 2;
        }
        if (lane == 31) pairs[G] = incl;
      }
    }
  }
  tc_fence_before();
  // with multicast the partner CTA's barriers must be initialised before any
  // copy or commit reaches them: a cluster-wide barrier (it also syncs this CTA)
  if (kPairs) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // CTA-to-unit walk: with multicast both CTAs of a cluster take the same units
  const int rank = kPairs ? (int)cluster_rank() : 0;
  const int cl0 = kPairs ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ncl = kPairs ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  const int tok_tile = p.tok_on_m ? BM : bn;
  const int feat_tile = p.tok_on_m ? bn : BM;
  const int nfeat = p.fuse_situ ? (p.M_feat / 2) / BM : p.M_feat / feat_tile;
  const int nkb = p.K / BK;
  const bool dense = p.tile_prefix == nullptr;
  // the weight operand is B when tokens are on M, A otherwise
  const CUtensorMap* mapW = p.tok_on_m ? &tmB : &tmA;
  const CUtensorMap* mapX = p.tok_on_m ? &tmA : &tmB;
  const uint32_t offW = p.tok_on_m ? a_bytes : 0u;
  const uint32_t offX = p.tok_on_m ? 0u : w_bytes;
  // the weight tile: one box, or (fused SituGLU) 128 gate rows and the 128 up
  // rows of the same features, stacked into one 256-row operand.  In the
  // stacked form rows from p.w2_row0 on come from the second weight matrix.
  auto load_w = [&](uint32_t dst, uint32_t bar, int kb, int row) {
    if (p.fuse_situ) {
      tma_load_2d(mapW, dst, bar, kb * BK, row);
      tma_load_2d(mapW, dst + BM * BK * 2, bar, kb * BK, row + p.M_feat / 2);
    } else if (kStack && row >= p.w2_row0) {
      tma_load_2d(&tmW2, dst, bar, kb * BK, row - p.w2_row0);
    } else {
      tma_load_2d(mapW, dst, bar, kb * BK, row);
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      // Dense GEMMs know their units without reading device data, so the
      // weight tiles of the first ring of stages are requested before the
      // wait for the previous kernel (weights are constant).
      uint32_t pre = 0;
      if (dense && !kPairs) {
        const int U0 = total_units<kPairs>(p, tabs, tok_tile, nfeat);
        for (int u = cl0; u < U0 && pre < (uint32_t)S; u += ncl) {
          const Unit x = decode_unit<kPairs>(p, tabs, u, tok_tile, feat_tile, nfeat, nkb, rank);
          for (int kb = x.kb0; kb < x.kb1 && pre < (uint32_t)S; ++kb, ++pre) {
            const uint32_t sa = smem_u32(smem + (size_t)pre * stage_bytes);
            mbar_arrive_expect_tx(full_bar((int)pre), stage_bytes);
            load_w(sa + offW, full_bar((int)pre), kb, x.w_row0);
          }
        }
      }
      pdl_wait();
      const int U = total_units<kPairs>(p, tabs, tok_tile, nfeat);
      // ring position kept incrementally: stage s, its smem address, parity
      uint32_t it = 0, s = 0, ph = 0;
      uint32_t sa = smem_u32(smem);
      const uint32_t sa0 = sa;
      bool ok = true;
      for (int u = cl0; u < U && ok; u += ncl) {
        const Unit x = decode_unit<kPairs>(p, tabs, u, tok_tile, feat_tile, nfeat, nkb, rank);
        for (int kb = x.kb0; kb < x.kb1; ++kb, ++it) {
          if (kPairs) {
            if (!wait_phase(empty_bar((int)s), ph ^ 1u, abort_flag, kErrProducer)) { ok = false; break; }
            mbar_arrive_expect_tx(full_bar((int)s), stage_bytes);
            // the weight tile in two 128-row boxes: gate and up rows (fused
            // SituGLU) or rows w_row0 and w_row0 + 128
            const int wstep = p.fuse_situ ? p.M_feat / 2 : BM;
            if (!x.shareA) {
              // this CTA's half of the shared weight tile goes to both CTAs,
              // the token tile to this one only
              tma_load_2d_mc(mapW, sa + offW + (uint32_t)rank * (BM * BK * 2), full_bar((int)s),
                             kb * BK, x.w_row0 + rank * wstep, (uint16_t)3u);
              tma_load_2d(mapX, sa + offX, full_bar((int)s), kb * BK, x.tok_row0);
            } else {
              // shared token tile (CTA 0 multicasts it), own weight tile
              if (rank == 0)
                tma_load_2d_mc(mapX, sa + offX, full_bar((int)s), kb * BK, x.tok_row0, (uint16_t)3u);
              tma_load_2d(mapW, sa + offW, full_bar((int)s), kb * BK, x.w_row0);
              tma_load_2d(mapW, sa + offW + BM * BK * 2, full_bar((int)s), kb * BK, x.w_row0 + wstep);
            }
          } else {
            if (it >= pre) {
              if (!wait_phase(empty_bar((int)s), ph ^ 1u, abort_flag, kErrProducer)) { ok = false; break; }
              mbar_arrive_expect_tx(full_bar((int)s), stage_bytes);
              load_w(sa + offW, full_bar((int)s), kb, x.w_row0);
            }
            tma_load_2d(mapX, sa + offX, full_bar((int)s), kb * BK, x.tok_row0);
          }
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; sa = sa0; } else { sa += stage_bytes; }
        }
      }
      // stages armed before the wait but never reached (abort) still get their
      // token tile so that every armed phase can complete
      for (; it < pre; ++it) {
        const int s = (int)it;
        tma_load_2d(mapX, smem_u32(smem + (size_t)s * stage_bytes) + offX, full_bar(s), 0, 0);
      }
      // drain: every copy this thread issued has landed before the CTA exits
      const uint32_t first = it > (uint32_t)S ? it - (uint32_t)S : 0u;
      for (uint32_t j = first; j < it; ++j) {
        volatile int never = 0;
        const uint32_t bar = full_bar((int)(j % (uint32_t)S));
        const uint32_t par = (j / (uint32_t)S) & 1u;
        if (!wait_bounded(bar, par, &never, kErrDrain)) break;
      }
    }
  } else if (warp == 1 || (kSwap && warp == 6)) {
    if (lane == 0) {
      // ---------------- MMA issuer(s) ----------------
      // (swap form: warp 1 the gate halves, warp 6 the up halves)
      const int half = warp == 6 ? 1 : 0;
      pdl_wait();
      const int U = total_units<kPairs>(p, tabs, tok_tile, nfeat);
      const uint32_t idesc = idesc_bf16(BM, bn);
      // descriptors of stage 0 (A side = the M operand, B side = the N
      // operand); stage s adds s*stage_bytes, each K=16 step adds 32 bytes (+2
      // in the 16-byte address field, which never carries out)
      const uint64_t dx0 = sdesc(smem_u32(smem) + offX);
      const uint64_t dw0 = sdesc(smem_u32(smem) + offW);
      const uint64_t da0 = p.tok_on_m ? dx0 : dw0;
      const uint64_t db0 = p.tok_on_m ? dw0 : dx0;
      const uint64_t dstep = stage_bytes >> 4;
      uint32_t uit = 0, s = 0, ph = 0;
      uint64_t da = da0, db = db0;
      bool ok = true;
      for (int u = cl0; u < U && ok; u += ncl, ++uit) {
        const Unit x = decode_unit<kPairs>(p, tabs, u, tok_tile, feat_tile, nfeat, nkb, rank);
        const int acc = (int)(uit & 1u);
        if (!wait_phase(tempty_bar(acc), ((uit >> 1) & 1u) ^ 1u, abort_flag, kErrMmaTmem)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * acc_stride;
        uint32_t accumulate = 0u;
        for (int kb = x.kb0; kb < x.kb1; ++kb) {
          if (!wait_phase(full_bar((int)s), ph, abort_flag, kErrMmaFull)) { ok = false; break; }
          tc_fence_after();
          if constexpr (kSwap) {
            // the stage's two 128-row weight halves on M (A side), the unit's
            // tokens on N, each half into its own accumulator
            constexpr uint64_t kHalf = (BM * BK * 2) >> 4;
#pragma unroll
            for (int j = 0; j < kK16; ++j)
              mma_bf16(d_tmem + (uint32_t)(half * bn), da + (uint64_t)half * kHalf + 2 * j,
                       db + 2 * j, idesc, j ? 1u : accumulate);
          } else {
#pragma unroll
            for (int j = 0; j < kK16; ++j)
              mma_bf16(d_tmem, da + 2 * j, db + 2 * j, idesc, j ? 1u : accumulate);
          }
          accumulate = 1u;
          if (kPairs) mma_commit_mc(empty_bar((int)s), (uint16_t)3u);
          else mma_commit(empty_bar((int)s));
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; da = da0; db = db0; }
          else { da += dstep; db += dstep; }
        }
        if (ok) mma_commit(tfull_bar(acc));
      }
      // every MMA this thread issued has completed before TMEM is freed
      mma_commit(done_bar);
      volatile int never = 0;
      wait_bounded(done_bar, 0u, &never, kErrDone);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;             // accumulator row of this thread
    pdl_wait();
    const int U = total_units<kPairs>(p, tabs, tok_tile, nfeat);
    uint32_t uit = 0;
    for (int u = cl0; u < U; u += ncl, ++uit) {
      const Unit x = decode_unit<kPairs>(p, tabs, u, tok_tile, feat_tile, nfeat, nkb, rank);
      const int acc = (int)(uit & 1u);
      if (!wait_bounded(tfull_bar(acc), (uit >> 1) & 1u, abort_flag, kErrEpilogue)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * acc_stride;
      if constexpr (kSwap) {
        // row r of the gate half and of the up half (output feature fcol0 + r),
        // columns = the unit's tokens; both rounded to bf16 first, as the
        // stored GEMM output would be, then SituGLU
        const int fcol0 = x.feat_tile * BM;
        uint16_t* o = reinterpret_cast<uint16_t*>(p.out);
        for (int c0 = 0; c0 < bn; c0 += 16) {
          uint32_t g[16], v[16];
          tmem_ld16(tbase + (uint32_t)c0, g);
          tmem_ld16(tbase + (uint32_t)(bn + c0), v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const int t = c0 + j;
            const uint32_t gb = pack_bf16x2(__uint_as_float(g[j]), __uint_as_float(g[j + 1]));
            const uint32_t ub = pack_bf16x2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
            const uint32_t a = situ2(gb, ub, p.sp);
            const long long row = (long long)(x.tok_row0 + t);
            if (t < x.nvalid) o[row * p.ldo + fcol0 + r] = (uint16_t)a;
            if (t + 1 < x.nvalid) o[(row + 1) * p.ldo + fcol0 + r] = (uint16_t)(a >> 16);
          }
        }
      } else if (p.tok_on_m && !p.out_fp32) {
        // row r = token, columns = features.  Per 64-column chunk each thread
        // rounds its row to bf16 (after SituGLU when fused, after adding the
        // bf16 addend in fp32 when there is one) into its warp's staging
        // buffer [32 rows][64 bf16].  When all 32 rows of the warp's block are
        // valid, one lane stores the buffer with a TMA bulk tensor store;
        // otherwise (a ragged block: the rows past it belong to the next
        // group) the warp writes 4 rows x 128 bytes per 16-byte store
        // instruction, valid rows only.
        uint32_t* st = reinterpret_cast<uint32_t*>(stage_out) + (size_t)q * 32 * 32;
        const bool bulk = p.tma_store && q * 32 + 31 < x.nvalid;
        const int width = p.fuse_situ ? BM : bn;           // output columns of this tile
        const int fcol0 = x.feat_tile * width;
        const int ldo = p.fuse_situ ? p.M_feat / 2 : p.ldo;
        const bool row_ok = r < x.nvalid;
        const uint16_t* arow =
            p.add ? p.add + (long long)(x.tok_row0 + (row_ok ? r : 0)) * ldo + fcol0 : nullptr;
        if (p.add && row_ok)   // pull this thread's addend row into L2 while the tile drains
          for (int b = 0; b < width * 2; b += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(arow) + b));
        for (int c0 = 0; c0 < width; c0 += 64) {
          // the staging buffer is free once the previous bulk store read it
          if (p.tma_store) {
            if (lane == 0) bulk_wait_read();
            __syncwarp();
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // the addend's 32 columns, loaded before the accumulator
            uint4 ad[4] = {};
            if (p.add && row_ok) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ad[i] = __ldg(reinterpret_cast<const uint4*>(arow + c0 + 32 * h) + i);
            }
            float f[32];
            {
              uint32_t v[16];
              tmem_ld16(tbase + (uint32_t)(c0 + 32 * h), v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]);
              tmem_ld16(tbase + (uint32_t)(c0 + 32 * h + 16), v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) f[16 + j] = __uint_as_float(v[j]);
            }
            uint32_t pk[16];
            if (p.fuse_situ) {
              // gate = f, up = the same features 128 columns further; both
              // rounded to bf16 first, as the stored GEMM output would be
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[16];
                tmem_ld16(tbase + (uint32_t)(BM + c0 + 32 * h + 16 * hh), v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                  const uint32_t gb = pack_bf16x2(f[16 * hh + j], f[16 * hh + j + 1]);
                  const uint32_t ub = pack_bf16x2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                  const f32x2 o = situ2_f32(gb, ub, p.sp);
                  pk[8 * hh + j / 2] = pack_bf16x2(f2_lo(o), f2_hi(o));
                }
              }
            } else {
              if (p.add) {
                const uint32_t aw[16] = {ad[0].x, ad[0].y, ad[0].z, ad[0].w, ad[1].x, ad[1].y,
                                         ad[1].z, ad[1].w, ad[2].x, ad[2].y, ad[2].z, ad[2].w,
                                         ad[3].x, ad[3].y, ad[3].z, ad[3].w};
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  f[2 * j] += bf16_lo(aw[j]);
                  f[2 * j + 1] += bf16_hi(aw[j]);
                }
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(f[2 * j], f[2 * j + 1]);
            }
            // 16-byte chunk 4h + c of row `lane`, XOR-swizzled by row
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(st + lane * 32 + (((4 * h + c) ^ (lane & 7)) * 4)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
          if (bulk) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmO, smem_u32(st), fcol0 + c0, x.tok_row0 + q * 32);
              bulk_commit();
            }
            continue;
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = i * 4 + (lane >> 3);            // row within this warp's 32
            const int c = lane & 7;                        // 8-column chunk
            const uint4 a = *reinterpret_cast<const uint4*>(st + rr * 32 + ((c ^ (rr & 7)) * 4));
            const int row_in_tile = q * 32 + rr;
            if (row_in_tile < x.nvalid) {
              const long long off = (long long)(x.tok_row0 + row_in_tile) * ldo + fcol0 + c0 + c * 8;
              *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + off) = a;
            }
          }
          __syncwarp();
        }
      } else if (p.tok_on_m) {
        // fp32 split partials, row r = token
        const bool valid = r < x.nvalid;
        const long long orow = (long long)(x.tok_row0 + r);
        const int fcol0 = x.feat_tile * bn;
        for (int c0 = 0; c0 < bn; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + (uint32_t)c0, v);
          tmem_wait_ld();
          if (!valid) continue;
          float* o = reinterpret_cast<float*>(p.out) + (long long)x.split * p.split_stride +
                     orow * p.ldo + fcol0 + c0;
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<uint4*>(o + j) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      } else {
        // row r = feature, columns = tokens
        const int fcol = x.feat_tile * BM + r;
        for (int c0 = 0; c0 < bn; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + (uint32_t)c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            if (t < x.nvalid) {
              const long long orow = (long long)(x.tok_row0 + t);
              float f = __uint_as_float(v[j]);
              if (p.out_fp32) {
                reinterpret_cast<float*>(p.out)[(long long)x.split * p.split_stride +
                                                 orow * p.ldo + fcol] = f;
              } else {
                if (p.add) f += __uint_as_float((uint32_t)p.add[orow * p.ldo + fcol] << 16);
                reinterpret_cast<uint16_t*>(p.out)[orow * p.ldo + fcol] = to_bf16(f);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
    }
    // this warp's bulk stores have completed before the CTA exits
    if (p.tma_store && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(p.tmem_cols)
                 : "memory");
  }
  // no CTA leaves while its partner may still multicast into it or commit to it
  if (kPairs) cluster_sync();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() { return reinterpret_cast<EncodeTiledFn>(tensor_map_encoder()); }

bool make_map(CUtensorMap* m, const void* base, long long rows, int K, int box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Bytes of one ring stage: the M-side operand (one 128-row box; two for the
// swap form with weight halves) and bn rows of the N-side operand, 64 K wide.
int stage_bytes_for(int bn, int tok_on_m, int swap) {
  return (tok_on_m ? 1 : (swap ? 2 : 1)) * BM * BK * 2 + bn * BK * 2;
}

int stages_for(int stage) {
  const int budget = 200 * 1024;
  int s = budget / stage;
  return s > kMaxStages ? kMaxStages : (s < 2 ? 2 : s);
}

// Clusters of two gemm_tc_kernel CTAs that fit on the device at once with
// `smem` bytes each, cached per size (queried once per size and device).
int max_pairs_resident(size_t smem) {
  struct Entry { int dev; size_t smem; int pairs; };
  static Entry cache[16];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].dev == dev && cache[i].smem == smem) return cache[i].pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pairs = 0;
  if (cudaOccupancyMaxActiveClusters(&pairs, gemm_tc_kernel<true, kFormRegular>, &cfg) !=
      cudaSuccess)
    pairs = 0;
  if (n < 16) cache[n++] = Entry{dev, smem, pairs};
  return pairs;
}

// ring of stages, barriers, TMEM holder/abort flag, group tables, and (tokens
// on M only) the epilogue staging buffers; at most 227 KB
size_t smem_for(int stage, int stages, int groups, int tok_on_m) {
  return 1024 + stages * stage + (2 * stages + 5) * 8 + 16 +
         (groups ? (size_t)group_table_ints(groups) * 4 : 0) + 1024 +
         (tok_on_m ? 4 * 32 * 32 * 4 : 0);
}

// Tensor map of a bf16 output [rows, cols] (row stride ldo) for bulk stores of
// [32 rows][64 columns] boxes with the 128-byte swizzle.
bool make_out_map(CUtensorMap* m, const void* base, long long rows, int cols, int ldo) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ldo * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const GemmDesc& g, cudaStream_t stream) {
  GemmParams p{};
  p.tok_on_m = g.tok_on_m;
  p.M_feat = g.M_feat;
  p.K = g.K;
  p.bn = g.bn;
  p.num_groups = g.G;
  p.grp_count = g.grp_count;
  p.grp_offset = g.grp_offset;
  p.tile_prefix = g.tile_prefix;
  p.T_dense = g.T_dense;
  p.splits = g.splits;
  p.out = g.out;
  p.ldo = g.ldo;
  p.split_stride = g.split_stride;
  p.out_fp32 = g.out_fp32;
  p.add = g.add;
  p.fuse_situ = g.fuse_situ;
  // weights on M with SituGLU fused: the swap-form instance (gate and up
  // halves as two MMAs per stage); it writes bf16 and does not split K
  const int swap = !g.tok_on_m && g.fuse_situ;
  if (swap && (g.splits != 1 || g.out_fp32 || g.add || g.bn > 128 || g.W2))
    return cudaErrorInvalidValue;
  const int stage = stage_bytes_for(g.bn, g.tok_on_m, swap);
  p.stages = stages_for(stage);
  // CTA pairs with a multicast operand: tokens on M, 256-row weight tiles, and
  // an even count of weight tiles (or, dense, of token tiles)
  {
    const int nfeat = g.fuse_situ ? (g.M_feat / 2) / BM : g.M_feat / 256;
    const int ntok = (g.T_dense + BM - 1) / BM;
    p.mcast = g.tok_on_m && g.bn == 256 && g.splits == 1 &&
              (nfeat % 2 == 0 || (!g.grp_count && ntok % 2 == 0));
  }
  p.sp = make_situ_params(g.beta > 0.0f ? g.beta : 1.0f, g.linear_beta);
  // a second weight matrix stacked after the first: weights on M, one
  // 128-row box per unit, and the first one's rows a whole number of units
  p.w2_row0 = g.W2 ? g.w2_row0 : 0;
  if (g.W2 && (g.tok_on_m || g.fuse_situ || g.w2_row0 <= 0 || g.w2_row0 % BM))
    return cudaErrorInvalidValue;
  uint32_t cols = 32;
  while (cols < (uint32_t)((swap ? 4 : 2) * g.bn)) cols <<= 1;
  if (cols > 512) return cudaErrorInvalidValue;
  p.tmem_cols = cols;

  CUtensorMap mw, mx, mw2;
  const int w_box = (g.fuse_situ || p.mcast) ? BM : (g.tok_on_m ? g.bn : BM);
  const int x_box = g.tok_on_m ? BM : g.bn;
  // the weight map covers the rows that exist (fewer than G * M_feat when the
  // last feature tile is partial: its missing rows read as zeros)
  const long long w_rows = g.W2 ? (long long)g.w2_row0
                                : (g.w_rows > 0 ? g.w_rows : (long long)g.G * g.M_feat);
  if (!make_map(&mw, g.W, w_rows, g.K, w_box)) return cudaErrorInvalidValue;
  if (!make_map(&mx, g.X, g.x_rows, g.K, x_box)) return cudaErrorInvalidValue;
  if (g.W2) {
    if (!make_map(&mw2, g.W2, g.w2_rows, g.K, BM)) return cudaErrorInvalidValue;
  } else {
    mw2 = mw;
  }
  // bf16 output with tokens on M: full 32-row blocks leave by bulk tensor stores
  CUtensorMap mo = mw;
#ifndef LMOE_TMA_STORE
#define LMOE_TMA_STORE 1
#endif
  p.tma_store = 0;
  if (LMOE_TMA_STORE && g.tok_on_m && !g.out_fp32) {
    const int cols = g.fuse_situ ? g.M_feat / 2 : g.M_feat;
    const long long out_rows = g.grp_count ? g.x_rows : (long long)g.T_dense;
    if (!make_out_map(&mo, g.out, out_rows, cols, g.ldo))
      return cudaErrorInvalidValue;
    p.tma_store = 1;
  }

  const size_t smem = smem_for(stage, p.stages, g.grp_count ? g.G : 0, g.tok_on_m);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto* kern = p.mcast ? gemm_tc_kernel<true, kFormRegular>
                       : swap ? gemm_tc_kernel<false, kFormSwap>
                              : g.W2 ? gemm_tc_kernel<false, kFormStack>
                                     : gemm_tc_kernel<false, kFormRegular>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (p.mcast) {
    // as many CTA pairs as can be resident at once (pairs share a GPC)
    const int pairs = max_pairs_resident(smem);
    if (pairs < 1) return cudaErrorInvalidConfiguration;
    int np = pairs;
    if (g.max_units > 0 && g.max_units < np) np = g.max_units;
    return launch_k_cluster(gemm_tc_kernel<true, kFormRegular>, dim3(2 * np), dim3(kThreads), smem,
                            stream, 2, mx, mw, mw2, mo, p);
  }
  int grid = num_sms();
  if (g.max_units > 0 && g.max_units < grid) grid = g.max_units;
  if (grid < 1) grid = 1;
  if (g.tok_on_m)
    return launch_k(kern, dim3(grid), dim3(kThreads), smem, stream, mx, mw, mw2, mo, p);
  return launch_k(kern, dim3(grid), dim3(swap ? kThreadsSwap : kThreads), smem, stream, mw, mx, mw2, mo,
                  p);
}

int* device_error_word() {
  static int* cache[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

int read_device_error(int clear) {
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return LMOE_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return LMOE_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return LMOE_ERR_CUDA;
  }
  return v;
}

}  // namespace lmoe

extern "C" int lmoe_gemm_unit_walk(int G, const int* count, int nfeat, int paired, int* out,
                                   int max_units) {
  using namespace lmoe;
  if (G < 1 || G > 1024 || !count || nfeat < 1 || (paired != 0 && paired != 1) ||
      (paired && nfeat % 2) || max_units < 0)
    return LMOE_ERR_DIM;
  // the tables the kernel builds in its prologue, built here in order
  std::vector<int> tab(group_table_ints(G));
  int* prefix = tab.data();
  int* cnt = prefix + G + 1;
  int* first = cnt + G;
  int* pairs = first + G;
  prefix[0] = pairs[0] = 0;
  long long row = 0;
  for (int g = 0; g < G; ++g) {
    if (count[g] < 0) return LMOE_ERR_DIM;
    const int t = (count[g] + BM - 1) / BM;
    cnt[g] = count[g];
    first[g] = (int)row;
    row += count[g];
    prefix[g + 1] = prefix[g] + t;
    pairs[g + 1] = pairs[g] + t * nfeat / 2;
  }
  if (row > (1LL << 30)) return LMOE_ERR_DIM;
  GemmParams p{};
  p.tok_on_m = 1;
  p.bn = 256;
  p.M_feat = 256 * nfeat;
  p.num_groups = G;
  p.tile_prefix = prefix;   // marks the grouped walk; the walk reads the tables only
  p.splits = 1;
  const GroupTables tabs{prefix, cnt, first, pairs};
  const int U = paired ? total_units<true>(p, tabs, BM, nfeat)
                       : total_units<false>(p, tabs, BM, nfeat);
  if (!out) return U;
  const int nr = 1 + paired;
  for (int u = 0; u < U && u < max_units; ++u)
    for (int r = 0; r < nr; ++r) {
      const Unit x = paired ? decode_unit<true>(p, tabs, u, BM, 256, nfeat, 1, r)
                            : decode_unit<false>(p, tabs, u, BM, 256, nfeat, 1, r);
      int* o = out + ((size_t)u * nr + r) * 5;
      o[0] = x.tok_row0;
      o[1] = x.nvalid;
      o[2] = x.w_row0;
      o[3] = x.feat_tile;
      o[4] = x.shareA;
    }
  return U;
}
