// Block-scaled (MXFP4) routed-expert weights: their dequantization to bf16 and
// the decode-size expert kernels that read the 4-bit weights directly.
//
// Format (vLLM PR #50088, commits 4-5, and TensorRT-LLM PR #20541 run this
// layer's routed experts on the TRTLLM-Gen MXFP4 backend; the layout is the
// OCP microscaling one): a weight matrix [rows, K] is 4-bit E2M1 codes, two per
// byte (element 2i in the low nibble of byte i), and one E8M0 power-of-two
// scale per 32 consecutive elements of a row:
//   w[r, c] = E2M1(code[r, c]) * 2^(scale[r, c / 32] - 127).
// E2M1 pairs become f16x2 by the hardware conversion (exact: every E2M1 value
// is an f16 value), then fp32.
//
// Decode expert kernels.  At T <= 128 an expert holds a few (token, slot)
// rows, so its GEMMs are matrix-vector products bound by the weight bytes:
// 4.25 bits a weight instead of 16.  One block takes one active expert (the
// permutation lists them) and a strip of output columns.  Each warp loads the
// codes and scales of its columns into registers first, then the expert's
// rows of the input are staged in shared memory as fp32 (two tokens a pass, in
// a piece-major order that makes the lanes' 16-byte reads conflict-free).
// A lane owns whole 32-element scale blocks of a row: it sums the block's 32
// products in fp32, multiplies the sum by the block's power of two (exact) and
// adds it to its accumulator; the lanes of a row then reduce by shuffles.
// GEMM1 holds the gate row c and the up row d + c of each column and applies
// SituGLU to the two bf16-rounded sums, so act is written directly
// (vLLM PR #50088, commit 5: SituGLU acts on the dequantized gate/up).
#include <cuda.h>

#include "lmoe_internal.cuh"
#include "mxfp4.cuh"

namespace lmoe {
namespace {

__device__ __forceinline__ void f16x2_to_f32(uint32_t h, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
}

// 8 E2M1 codes of a 32-bit word (element 0 in the low nibble) -> fp32
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float (&v)[8]) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
  f16x2_to_f32(h0, v[0], v[1]);
  f16x2_to_f32(h1, v[2], v[3]);
  f16x2_to_f32(h2, v[4], v[5]);
  f16x2_to_f32(h3, v[6], v[7]);
}

// two fp32 -> f16x2, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// E8M0 scale exponent -> 2^(s - 127) in fp32 (s = 0: the subnormal 2^-127;
// s = 255: NaN)
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  const uint32_t bits = s == 0u ? 0x00400000u : (s == 255u ? 0x7FC00000u : s << 23);
  return __uint_as_float(bits);
}

// ---- dequantization: out[r, :] = bf16(w[r, :]) --------------------------------
// The codes and the output are one flat sequence of words: word q is 8 codes
// (4 bytes, element 0 in the low nibble) and 8 bf16 outputs (16 bytes), with
// the scale byte scales[q / 4] (rows are whole 32-element blocks).  A warp
// takes a unit of up to kDqUnitWords consecutive words of one group (the rows
// of one expert, or everything); its lanes take words lane, lane + 32, ..., with
// kDqInFlight of them loaded before any is converted, so that a warp's loads
// are 128-byte lines and its stores 512-byte runs.  With `counts`, the units
// of a group g with counts[g] == 0 (an expert no token was routed to) are
// skipped as a whole.  With `src_group`, output group g is read from the
// codes and scales of group src_group[g] (a compact copy of some experts).
// One launch takes up to two such jobs (the units of the first, then the
// second's).
constexpr int kDqUnitWords = 1024;
constexpr int kDqInFlight = 8;

__device__ __forceinline__ uint4 dequant_word(uint32_t w, uint32_t s) {
  const float sc = e8m0_to_f32(s);
  float v[8];
  e2m1x8_to_f32(w, v);
  return make_uint4(pack_bf16x2(v[0] * sc, v[1] * sc), pack_bf16x2(v[2] * sc, v[3] * sc),
                    pack_bf16x2(v[4] * sc, v[5] * sc), pack_bf16x2(v[6] * sc, v[7] * sc));
}

struct DqJob {
  const uint32_t* codes;
  const uint8_t* scales;
  uint4* out;
  long long words, words_per_group;
  const int32_t* counts;
  const int32_t* src_group;
};

__host__ __device__ __forceinline__ long long dq_units(const DqJob& j) {
  if (j.words <= 0) return 0;
  return (j.words + j.words_per_group - 1) / j.words_per_group *
         ((j.words_per_group + kDqUnitWords - 1) / kDqUnitWords);
}

__global__ void __launch_bounds__(256) dequant_kernel(const DqJob j0, const DqJob j1) {
  pdl_trigger();
  pdl_wait();   // out may still be read by the previous forward's GEMMs
  const long long units0 = dq_units(j0), units = units0 + dq_units(j1);
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (long long uu = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); uu < units;
       uu += nwarps) {
    const bool second = uu >= units0;   // (warp-uniform)
    const long long u = second ? uu - units0 : uu;
    const uint32_t* __restrict__ codes = second ? j1.codes : j0.codes;
    const uint8_t* __restrict__ scales = second ? j1.scales : j0.scales;
    uint4* __restrict__ out = second ? j1.out : j0.out;
    const long long words = second ? j1.words : j0.words;
    const long long words_per_group = second ? j1.words_per_group : j0.words_per_group;
    const int32_t* __restrict__ counts = second ? j1.counts : j0.counts;
    const int32_t* __restrict__ src_group = second ? j1.src_group : j0.src_group;
    const long long units_per_group = (words_per_group + kDqUnitWords - 1) / kDqUnitWords;
    const long long g = u / units_per_group;
    if (counts && counts[g] == 0) continue;   // (warp-uniform)
    // source word = output word + shift (a group is whole rows: a multiple of
    // 4 words, so the scale byte of a word is still its source index / 4)
    const long long shift = src_group ? ((long long)__ldg(src_group + g) - g) * words_per_group : 0;
    const long long q0 = g * words_per_group + (u - g * units_per_group) * kDqUnitWords;
    const long long q1 = min(q0 + kDqUnitWords, min((g + 1) * words_per_group, words));
    const uint32_t* cs = codes + shift;
    const uint8_t* ss = scales + shift / 4;
    long long q = q0 + lane;
    for (; q + 32 * (kDqInFlight - 1) < q1; q += 32 * kDqInFlight) {
      uint32_t w[kDqInFlight], sv[kDqInFlight];
#pragma unroll
      for (int i = 0; i < kDqInFlight; ++i) {
        w[i] = __ldg(cs + q + 32 * i);
        sv[i] = __ldg(ss + ((q + 32 * i) >> 2));
      }
#pragma unroll
      for (int i = 0; i < kDqInFlight; ++i) out[q + 32 * i] = dequant_word(w[i], sv[i]);
    }
    for (; q < q1; q += 32) out[q] = dequant_word(__ldg(cs + q), __ldg(ss + (q >> 2)));
  }
}

// ---- decode expert kernel -------------------------------------------------------
// Persistent: one block per SM; a ring of S (4 or 8) stages, one consumer warp
// per stage slot, so that a stage is computed and written by a single warp and
// S stages are in flight and in compute at once.
//   producer (one lane of the last warp): walks this block's work items
//     (active expert, strip of C output columns, pass of up to nts tokens);
//     per item it fills the next slot with the strip's codes (2D TMA boxes of
//     8 rows x sw bytes with the widest swizzle the row length allows, so that
//     the rows a warp reads at one column hit distinct banks), its scales and
//     the item's bf16 input rows (bulk copies), completing on the slot's
//     `full` mbarrier;
//   converters (4 warps; warp c serves the slots c, c+4): once a slot has
//     landed, convert the item's bf16 input rows (copied with the codes) to
//     f16 in place, each token scaled by a power of two, then arrive on
//     `ready`;
//   consumers (warp w serves slot w): the item's rows form 16-row tiles
//     (GEMM1: 8 gate rows over the same 8 up rows, so that a lane holds both
//     halves of its outputs); per 32-element scale block a lane widens its 8
//     codes of two rows to f16 (exact) and issues two mma.sync m16n8k16 (f16
//     in, fp32 accumulate) against the f16 inputs of up to 8 tokens, then adds
//     the result times the block's power of two to its accumulators.  The K
//     order inside a block is permuted alike for the codes and the inputs (a
//     lane's 4 code bytes are one 32-bit word of the row), which leaves the sums
//     unchanged.  The warp then writes its outputs (SituGLU on the bf16 gate and
//     up for GEMM1) and releases the slot.  No partial sums cross warps: the
//     results do not depend on timing.
// Every wait is bounded (about 2 s); on expiry the kernel records kErrFp4Wait
// and returns, after the producer has waited (bounded) for its copies in flight.
constexpr int kSlotWarps = 8;        // the most slots; two consumer warps a slot
constexpr int kConsumerWarps = 2 * kSlotWarps;
constexpr int kConverterWarps = 4;
constexpr int kProducerWarp = kConsumerWarps + kConverterWarps;
constexpr int kGemvThreads = (kProducerWarp + 1) * 32;
constexpr int kMaxNts = 8;           // tokens a stage: the MMA's N
constexpr int kMaxTiles = 4;         // 16-row tiles an item
constexpr long long kFp4WaitCycles = 1ll << 32;
constexpr int kErrFp4Wait = 8;       // device error code (after the GEMM's 1-6 and 7)
constexpr int kSmemBudget = 220 * 1024;
constexpr uint32_t kHdrOff = 384;    // after four mbarrier arrays and the abort flag

struct GemvArgs {
  const uint8_t* codes;     // [E, kRows * ncols, K/2] (also through the tensor map)
  const uint8_t* scales;    // [E, kRows * ncols, K/32]
  const uint16_t* x;        // expert-major input rows [rows, K] bf16
  uint16_t* out;            // [rows, ncols] bf16
  const int32_t* counts;    // [E]
  const int32_t* offsets;   // [E+1]
  const int32_t* active;    // active expert of each slot
  const int32_t* n_active;  // number of active experts
  int* err;                 // device error word
  int K, ncols, C, tiles, nchunk, nts, stages, max_slots;
  int sw;                   // swizzle span of the code boxes: 128, 64 or 32 bytes
  // byte offsets inside a stage (codes at 0, then scale bytes, input rows:
  // bf16 as copied, f16 once converted in place, the second consumer warp's
  // sums), and of the ring and slot table in the block's memory
  uint32_t codes_bytes, strip_scales, xh_off, part_off, stage_bytes, ring_off, table_off;
  SituParams situ;
};

struct StageHdr {
  int e, nt, row, c0;
  int exotic;               // a scale exponent of the item is 0 or 255 (set by the converter)
  float inv[kMaxNts];       // 2^-k of each token's f16 input rows (set by a converter)
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
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
// The same, suspending the thread (up to about 0.1 ms) until the phase
// completes: waiting warps then take no issue slots from the working ones.
__device__ __forceinline__ bool bar_try_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}
// true once the phase of `parity` has completed; false when the abort flag is
// set or the deadline passes (which sets it and records the error)
__device__ __noinline__ bool bar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* err) {
  const long long t0 = clock64();
  while (!bar_try_sleep(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kFp4WaitCycles) {
      atomicCAS(err, 0, kErrFp4Wait);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}
// Warps that go on to warp-synchronous instructions (shuffles, mma.sync) take
// the outcome for the whole warp (__all_sync): a wait that runs out in one lane
// then never leaves the other lanes at a collective the first one skipped.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* err) {
  return bar_try(bar, parity) || bar_wait_slow(bar, parity, abort_flag, err);
}
// global -> shared bulk copy completing on `bar` (addresses 16-byte aligned,
// bytes a multiple of 16), with an L2 cache policy
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// 3D TMA box {all sw-byte columns, C rows, every segment} of the codes
__device__ __forceinline__ void tma_box3(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                         int row, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(row), "r"(0), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// the four bytes of w (two E2M1 codes each, low nibble first) -> four f16x2
__device__ __forceinline__ void e2m1x4_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// 8 bf16 (a uint4) times a power of two -> 8 f16
__device__ __forceinline__ uint4 to_f16x8(const uint4 w, float up) {
  uint4 o;
  o.x = pack_f16x2(bf16_lo(w.x) * up, bf16_hi(w.x) * up);
  o.y = pack_f16x2(bf16_lo(w.y) * up, bf16_hi(w.y) * up);
  o.z = pack_f16x2(bf16_lo(w.z) * up, bf16_hi(w.z) * up);
  o.w = pack_f16x2(bf16_lo(w.w) * up, bf16_hi(w.w) * up);
  return o;
}

// kQ consecutive scale exponents of one row from jb (one 32-bit load for 4
// aligned ones, else 16-bit or byte loads)
template <int kQ>
__device__ __forceinline__ void load_scales(const uint8_t* row, int jb, uint32_t (&sv)[kQ]) {
  if (kQ == 4 && ((reinterpret_cast<uintptr_t>(row + jb) & 3) == 0)) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + jb);
#pragma unroll
    for (int q = 0; q < kQ; ++q) sv[q] = (w >> (8 * q)) & 255u;
  } else if (kQ % 2 == 0 && ((reinterpret_cast<uintptr_t>(row + jb) & 1) == 0)) {
#pragma unroll
    for (int q = 0; q < kQ; q += 2) {
      const uint32_t w = *reinterpret_cast<const uint16_t*>(row + jb + q);
      sv[q] = w & 255u;
      sv[(q + 1) % kQ] = w >> 8;
    }
  } else {
#pragma unroll
    for (int q = 0; q < kQ; ++q) sv[q] = row[jb + q];
  }
}

// One item on one warp.  Tile t of the item holds, for GEMM1 (kRows = 2),
// the gate rows c0 + 8t .. + 7 over the up rows of the same columns, for
// GEMM2 the rows c0 + 16t .. + 15; lane (g, tq) accumulates rows g and g + 8
// for tokens 2tq and 2tq + 1.
// Per-lane geometry of an item: rows g and g+8 of each 16-row tile.  Tile t
// of the item holds, for GEMM1 (kRows = 2), the gate rows c0 + 8t .. + 7 over
// the up rows of the same columns, for GEMM2 the rows c0 + 16t .. + 15; lane
// (g, tq) accumulates rows g and g + 8 for tokens 2tq and 2tq + 1.
template <int kRows, int kTiles>
struct ItemLane {
  const uint8_t* st;
  const uint16_t* xrow;
  const uint8_t* sc0[kTiles];
  const uint8_t* sc1[kTiles];
  uint32_t off0[kTiles], off1[kTiles];   // rows g, g+8 of each tile at segment 0
  uint32_t xsw, swz_mask, seg_bytes;
  int blk_shift;
  bool has_x;

  __device__ __forceinline__ ItemLane(const GemvArgs& a, const uint8_t* st_, int nt, int lane) {
    const int K = a.K, nblk = K >> 5, half_k = K >> 1;
    const int g = lane >> 2, tq = lane & 3;
    const int sw = a.sw, nseg = half_k / sw;
    st = st_;
    blk_shift = sw == 128 ? 3 : (sw == 64 ? 2 : 1);
    swz_mask = (1u << blk_shift) - 1u;
    // a strip of C rows is [segment][row][sw bytes]; kRows strips back to back
    seg_bytes = (uint32_t)(a.C * sw);
    const uint32_t strip_bytes = seg_bytes * (uint32_t)nseg;
    xsw = ((uint32_t)(g * sw) >> 7) & swz_mask;        // row g's swizzle (and g+8's)
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (kRows == 2) {
        off0[t] = (uint32_t)((8 * t + g) * sw + 4 * tq);   // gate strip
        off1[t] = strip_bytes + off0[t];                   // up strip
      } else {
        off0[t] = (uint32_t)((16 * t + g) * sw + 4 * tq);
        off1[t] = off0[t] + 8u * sw;
      }
    }
    xrow = reinterpret_cast<const uint16_t*>(st + a.xh_off) + g * K + 8 * tq;
    has_x = g < nt;
    // scale rows of the lane's two rows in each tile
    const uint8_t* scb = st + a.codes_bytes;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (kRows == 2) {
        sc0[t] = scb + (8 * t + g) * nblk;                       // gate strip row
        sc1[t] = scb + a.strip_scales + (8 * t + g) * nblk;      // up strip row
      } else {
        sc0[t] = scb + (16 * t + g) * nblk;
        sc1[t] = sc0[t] + 8 * nblk;
      }
    }
  }

  // kQ consecutive blocks from jb: for each tile, the blocks' MMAs interleaved.
  // kExact: scale exponents 0 and 255 may occur (2^-127 and NaN); otherwise
  // 2^(s-127) is just s in the fp32 exponent field.
  template <int kQ, bool kExact>
  __device__ __forceinline__ void blocks(int jb, float (&acc)[kTiles][4]) const {
    uint4 xv[kQ];
    uint32_t seg_off[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      xv[q] = make_uint4(0u, 0u, 0u, 0u);
      if (has_x) xv[q] = *reinterpret_cast<const uint4*>(xrow + 32 * (jb + q));
      seg_off[q] = (uint32_t)((jb + q) >> blk_shift) * seg_bytes +
                   (((uint32_t)(jb + q) & swz_mask) ^ xsw) * 16u;
    }
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      uint32_t p[kQ][2][4];   // [block][row g / g+8] f16x2 of code bytes 0..3
      uint32_t e0[kQ], e1[kQ];
      load_scales<kQ>(sc0[t], jb, e0);
      load_scales<kQ>(sc1[t], jb, e1);
      float s0[kQ], s1[kQ];
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        e2m1x4_to_f16x2(*reinterpret_cast<const uint32_t*>(st + off0[t] + seg_off[q]), p[q][0]);
        e2m1x4_to_f16x2(*reinterpret_cast<const uint32_t*>(st + off1[t] + seg_off[q]), p[q][1]);
        s0[q] = kExact ? e8m0_to_f32(e0[q]) : __uint_as_float(e0[q] << 23);
        s1[q] = kExact ? e8m0_to_f32(e1[q]) : __uint_as_float(e1[q] << 23);
      }
      float d[kQ][4];
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.0f;
        const uint32_t a0[4] = {p[q][0][0], p[q][1][0], p[q][0][1], p[q][1][1]};
        mma_f16(d[q], a0, xv[q].x, xv[q].y);
      }
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const uint32_t a1[4] = {p[q][0][2], p[q][1][2], p[q][0][3], p[q][1][3]};
        mma_f16(d[q], a1, xv[q].z, xv[q].w);
      }
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        acc[t][0] = fmaf(d[q][0], s0[q], acc[t][0]);
        acc[t][1] = fmaf(d[q][1], s0[q], acc[t][1]);
        acc[t][2] = fmaf(d[q][2], s1[q], acc[t][2]);
        acc[t][3] = fmaf(d[q][3], s1[q], acc[t][3]);
      }
    }
  }
};

// The lane's sums over the scale blocks [jb_lo, jb_hi) of the item.
template <int kRows, int kTiles, bool kExact>
__device__ __forceinline__ void accumulate_range(const ItemLane<kRows, kTiles>& L, int jb_lo,
                                                 int jb_hi, float (&acc)[kTiles][4]) {
  // blocks interleaved a step: 4 with one tile, 2 with more (registers)
  constexpr int kQ = kTiles == 1 ? 4 : 2;
  int jb = jb_lo;
  for (; jb + kQ <= jb_hi; jb += kQ) L.template blocks<kQ, kExact>(jb, acc);
  for (; jb < jb_hi; ++jb) L.template blocks<1, kExact>(jb, acc);
}
template <int kRows, int kTiles>
__device__ __forceinline__ void accumulate_blocks(const GemvArgs& a, const uint8_t* st,
                                                  const StageHdr& h, int lane, int jb_lo,
                                                  int jb_hi, float (&acc)[kTiles][4]) {
  const ItemLane<kRows, kTiles> L(a, st, h.nt, lane);
#pragma unroll
  for (int t = 0; t < kTiles; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
  if (h.exotic) accumulate_range<kRows, kTiles, true>(L, jb_lo, jb_hi, acc);
  else accumulate_range<kRows, kTiles, false>(L, jb_lo, jb_hi, acc);
}

// The item's outputs from the lane's sums: tokens 2tq, 2tq+1 below nt (undo
// the power-of-two input scaling, exact, then round).
template <int kRows, int kTiles>
__device__ __forceinline__ void write_item(const GemvArgs& a, const StageHdr& h, int lane,
                                           const float (&acc)[kTiles][4]) {
  const int g = lane >> 2, tq = lane & 3;
  const int nt = h.nt, ncols = a.ncols;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int n = 2 * tq + q;
      if (n >= nt) continue;
      const float inv = h.inv[n];
      uint16_t* orow = a.out + (long long)(h.row + n) * ncols + h.c0;
      if (kRows == 2) {
        // act = bf16(SituGLU(bf16(gate), bf16(up))), column c0 + 8t + g
        const uint32_t g2 = to_bf16(acc[t][q] * inv);
        const uint32_t u2 = to_bf16(acc[t][2 + q] * inv);
        orow[8 * t + g] = (uint16_t)(situ2(g2, u2, a.situ) & 0xFFFFu);
      } else {
        orow[16 * t + g] = to_bf16(acc[t][q] * inv);
        orow[16 * t + g + 8] = to_bf16(acc[t][2 + q] * inv);
      }
    }
  }
}

template <int kRows, int kTiles>
__global__ void __launch_bounds__(kGemvThreads, 1)
    fp4_expert_kernel(const __grid_constant__ CUtensorMap tm_codes, GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* ready = full + kSlotWarps;
  uint64_t* empty = ready + kSlotWarps;
  uint64_t* half_done = empty + kSlotWarps;   // the second half's sums are stored
  volatile int* abort_flag = reinterpret_cast<volatile int*>(half_done + kSlotWarps);
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem + kHdrOff);
  uint8_t* ring = smem + a.ring_off;
  int32_t* tab = reinterpret_cast<int32_t*>(smem + a.table_off);   // e, n, row0 per slot
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;   // 4 or 8
  const int K = a.K, ncols = a.ncols, C = a.C;
  const int nblk = K >> 5, k8 = K >> 3;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      bar_init(smem_addr(full + i), 1);
      bar_init(smem_addr(ready + i), 1);
      bar_init(smem_addr(empty + i), 1);
      bar_init(smem_addr(half_done + i), 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_trigger();
  pdl_wait();
  const int n_active = min(a.n_active[0], a.max_slots);
  // the slot table (expert, rows, first row of every active expert)
  for (int i = threadIdx.x; i < n_active; i += blockDim.x) {
    const int e = a.active[i];
    tab[3 * i] = e;
    tab[3 * i + 1] = a.counts[e];
    tab[3 * i + 2] = a.offsets[e];
  }
  __syncthreads();
  if (warp == kProducerWarp) {
    if (lane == 0) {
      uint64_t stream_pol, keep_pol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream_pol));
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep_pol));
      const int total = n_active * a.nchunk;
      const long long rows_w = (long long)kRows * ncols;
      int s = 0;
      uint32_t ph = 0;
      int filled = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
        const int slot = it / a.nchunk, chunk = it - slot * a.nchunk;
        const int e = tab[3 * slot], n = tab[3 * slot + 1], row0 = tab[3 * slot + 2];
        const int c0 = chunk * C;
        for (int t0 = 0; t0 < n; t0 += a.nts) {
          if (!bar_wait(smem_addr(empty + s), ph ^ 1u, abort_flag, a.err)) { ok = false; break; }
          StageHdr& h = hdr[s];
          h.e = e;
          h.nt = min(a.nts, n - t0);
          h.row = row0 + t0;
          h.c0 = c0;
          const uint32_t bar = smem_addr(full + s);
          const uint32_t xbytes = (uint32_t)h.nt * K * 2;
          bar_arrive_tx(bar, a.codes_bytes + kRows * a.strip_scales + xbytes);
          uint8_t* st = ring + (size_t)s * a.stage_bytes;
          // codes: one 3D box per strip (C rows x every segment), landing as
          // [segment][row][sw bytes]
          const long long ebase = (long long)e * rows_w;
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            tma_box3(&tm_codes, smem_addr(st + r * (a.codes_bytes / kRows)), bar,
                     (int)(ebase + (long long)r * ncols + c0), stream_pol);
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            bulk_g2s(smem_addr(st + a.codes_bytes + r * a.strip_scales),
                     a.scales + (ebase + (long long)r * ncols + c0) * nblk, a.strip_scales, bar,
                     stream_pol);
          bulk_g2s(smem_addr(st + a.xh_off), a.x + (long long)(row0 + t0) * K, xbytes, bar,
                   keep_pol);
          ++filled;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      // end markers: one stage with no copies for every slot
      for (int i = 0; ok && i < S; ++i) {
        if (!bar_wait(smem_addr(empty + s), ph ^ 1u, abort_flag, a.err)) break;
        hdr[s].e = -1;
        bar_arrive(smem_addr(full + s));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      // copies still in flight (only after an abort): wait for them to land
      if (*abort_flag) {
        int ss = s;
        uint32_t pp = ph;
        for (int i = 0; i < min(filled, S); ++i) {
          if (--ss < 0) { ss = S - 1; pp ^= 1u; }
          const long long t0 = clock64();
          while (!bar_try(smem_addr(full + ss), pp) && clock64() - t0 < kFp4WaitCycles) {
          }
        }
      }
    }
    return;
  }
  if (warp >= kConsumerWarps) {
    // converter c serves the slots c, c + 4: once a slot has landed, the
    // item's input rows to f16, in place.
    // Token t is scaled by 2^k_t so that its largest magnitude lies in
    // [2^14, 2^15) (k_t = 0 for an all-zero or non-finite row, k_t <= 126);
    // every element within 2^30 of that largest one is then exact in f16,
    // smaller ones round to the f16 subnormal grid.
    // (with 8 slots each converter serves two, taking them in turn)
    const int cw = warp - kConsumerWarps;
    const bool two = S > kConverterWarps;
    uint32_t ph0 = 0u, ph1 = 0u;   // phases of slots cw and cw + 4
    bool live0 = true, live1 = two;
    bool turn = false;             // false: slot cw, true: slot cw + 4
    while (live0 || live1) {
      if (turn ? !live1 : !live0) { turn = !turn; continue; }
      const int s = turn ? cw + kConverterWarps : cw;
      if (!__all_sync(0xffffffffu, bar_wait(smem_addr(full + s), turn ? ph1 : ph0, abort_flag, a.err)))
        break;
      StageHdr& h = hdr[s];
      const int e = h.e;
      if (e >= 0) {
        uint4* xb = reinterpret_cast<uint4*>(ring + (size_t)s * a.stage_bytes + a.xh_off);
        for (int t = 0; t < h.nt; ++t) {
          uint4* xr = xb + t * k8;
          uint32_t mx = 0;   // largest |x| as fp32 bits (ordered like the magnitudes)
#pragma unroll 4
          for (int p = lane; p < k8; p += 32) {
            const uint4 w = xr[p];
            mx = max(mx, max((w.x << 16) & 0x7FFFFFFFu, w.x & 0x7FFF0000u));
            mx = max(mx, max((w.y << 16) & 0x7FFFFFFFu, w.y & 0x7FFF0000u));
            mx = max(mx, max((w.z << 16) & 0x7FFFFFFFu, w.z & 0x7FFF0000u));
            mx = max(mx, max((w.w << 16) & 0x7FFFFFFFu, w.w & 0x7FFF0000u));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const int ex = (int)(mx >> 23);   // biased exponent of the largest |x|
          const int k = (mx == 0u || ex == 255) ? 0 : min(141 - ex, 126);
          const float up = __uint_as_float((uint32_t)(k + 127) << 23);
          if (lane == 0) h.inv[t] = __uint_as_float((uint32_t)(127 - k) << 23);
          // in place: a lane rewrites the 16 bytes it read
#pragma unroll 4
          for (int p = lane; p < k8; p += 32) xr[p] = to_f16x8(xr[p], up);
        }
        // is a scale exponent of the item 0 or 255?  (4 bytes a step; the
        // scale strips are a multiple of 16 bytes)
        const uint32_t* sw4 = reinterpret_cast<const uint32_t*>(
            ring + (size_t)s * a.stage_bytes + a.codes_bytes);
        bool exotic = false;
        for (int i = lane; i < (int)(kRows * a.strip_scales / 4); i += 32) {
          const uint32_t w = sw4[i];
          // a zero byte of w, or of ~w (a 255 byte)
          const uint32_t z0 = (w - 0x01010101u) & ~w & 0x80808080u;
          const uint32_t z1 = (~w - 0x01010101u) & w & 0x80808080u;
          exotic |= (z0 | z1) != 0u;
        }
        exotic = __any_sync(0xffffffffu, exotic);
        if (lane == 0) h.exotic = exotic ? 1 : 0;
        // these generic-proxy writes precede the next TMA fill of the slot
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();   // orders every lane's writes before lane 0's release
      if (lane == 0) bar_arrive(smem_addr(ready + s));
      if (turn) {
        ph1 ^= 1u;
        if (e < 0) live1 = false;
      } else {
        ph0 ^= 1u;
        if (e < 0) live0 = false;
      }
      if (two) turn = !turn;
    }
    return;
  }
  // ---- consumers: warps w and w + 8 serve slot w, each half of the blocks ----
  const int s = warp & (kSlotWarps - 1), half = warp >> 3;
  if (s >= S) return;
  uint32_t ph = 0;
  const uint8_t* st = ring + (size_t)s * a.stage_bytes;
  float* part = reinterpret_cast<float*>(ring + (size_t)s * a.stage_bytes + a.part_off);
  const int jb_mid = nblk / 2;
  while (true) {
    if (!__all_sync(0xffffffffu, bar_wait(smem_addr(ready + s), ph, abort_flag, a.err))) break;
    const StageHdr& h = hdr[s];
    if (h.e < 0) break;
    float acc[kTiles][4];
    if (half) {
      accumulate_blocks<kRows, kTiles>(a, st, h, lane, jb_mid, nblk, acc);
#pragma unroll
      for (int t = 0; t < kTiles; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) part[(t * 4 + i) * 32 + lane] = acc[t][i];
      __syncwarp();   // orders every lane's writes before lane 0's release
      if (lane == 0) bar_arrive(smem_addr(half_done + s));
    } else {
      accumulate_blocks<kRows, kTiles>(a, st, h, lane, 0, jb_mid, acc);
      if (!__all_sync(0xffffffffu, bar_wait(smem_addr(half_done + s), ph, abort_flag, a.err))) break;
      // the two halves in a fixed order: the first half's blocks, then the second's
#pragma unroll
      for (int t = 0; t < kTiles; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] += part[(t * 4 + i) * 32 + lane];
      write_item<kRows, kTiles>(a, h, lane, acc);
      __syncwarp();
      if (lane == 0) bar_arrive(smem_addr(empty + s));
    }
    ph ^= 1u;
  }
}

// Geometry of one launch: columns an item C (GEMM1: 8 per tile, GEMM2: 16 per
// tile; tiles <= 4, codes at most 32 KB where possible), swizzle span, tokens
// a stage (up to 8), ring depth 8 (else 4), shared-memory layout.
bool plan_gemv(GemvArgs& a, int kRows, int max_slots, size_t* smem) {
  const int K = a.K;
  a.max_slots = max_slots;
  const int row_bytes = K / 2, nblk = K / 32;
  a.sw = row_bytes % 128 == 0 ? 128 : (row_bytes % 64 == 0 ? 64 : 32);
  if (row_bytes % a.sw || K > 4096) return false;
  const int cols_tile = kRows == 2 ? 8 : 16;
  a.table_off = (kHdrOff + kSlotWarps * (uint32_t)sizeof(StageHdr) + 127) & ~127u;
  const uint32_t table_bytes = (uint32_t)(3 * 4 * max_slots + 127) & ~127u;
  a.ring_off = (a.table_off + table_bytes + 1023) & ~1023u;
  for (int want : {8, 4}) {
    for (int tiles = kMaxTiles; tiles >= 1; tiles >>= 1) {
      const int C = tiles * cols_tile;
      if (a.ncols % C || (C * nblk) % 16) continue;
      if (tiles > 1 && 16LL * tiles * row_bytes > 32 * 1024) continue;
      for (int nts = kMaxNts; nts >= 1; nts >>= 1) {
        a.C = C;
        a.tiles = tiles;
        a.nchunk = a.ncols / C;
        a.codes_bytes = (uint32_t)(16 * tiles * row_bytes);
        a.strip_scales = (uint32_t)(C * nblk);
        a.nts = nts;
        a.xh_off = (a.codes_bytes + kRows * a.strip_scales + 127) & ~127u;
        a.part_off = a.xh_off + nts * K * 2;
        a.stage_bytes = (a.part_off + tiles * 4 * 32 * 4 + 1023) & ~1023u;
        if ((long long)kSmemBudget - a.ring_off >= (long long)want * a.stage_bytes) {
          a.stages = want;
          *smem = a.ring_off + (size_t)want * a.stage_bytes;
          return true;
        }
      }
    }
  }
  return false;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// codes [rows, K/2] bytes viewed as a 3D tensor {sw bytes, rows, K/2 / sw
// segments} (the segment dimension strides by sw bytes), boxes of
// {sw, box_rows, every segment}
bool make_codes_map(CUtensorMap* m, const uint8_t* codes, long long rows, int K, int sw,
                    int box_rows) {
  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!enc) return false;
  const int nseg = K / 2 / sw;
  cuuint64_t dims[3] = {(cuuint64_t)sw, (cuuint64_t)rows, (cuuint64_t)nseg};
  cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)sw};
  cuuint32_t box[3] = {(cuuint32_t)sw, (cuuint32_t)box_rows, (cuuint32_t)nseg};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle mode = sw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : (sw == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B);
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(codes), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, mode, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kRows, int kTiles>
cudaError_t launch_tiles(const CUtensorMap& tm, const GemvArgs& a, size_t smem, cudaStream_t s) {
  auto kern = fp4_expert_kernel<kRows, kTiles>;
  // (set on every launch: the attribute belongs to the current device)
  const cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_k(kern, dim3((unsigned)num_sms()), dim3(kGemvThreads), smem, s, tm, a);
}

template <int kRows>
cudaError_t launch_expert_kernel(GemvArgs& a, int slots, int E, cudaStream_t s) {
  size_t smem = 0;
  if (!plan_gemv(a, kRows, slots, &smem)) return cudaErrorInvalidValue;
  CUtensorMap tm;
  if (!make_codes_map(&tm, a.codes, (long long)E * kRows * a.ncols, a.K, a.sw, a.C))
    return cudaErrorInvalidValue;
  switch (a.tiles) {
    case 1: return launch_tiles<kRows, 1>(tm, a, smem, s);
    case 2: return launch_tiles<kRows, 2>(tm, a, smem, s);
    default: return launch_tiles<kRows, 4>(tm, a, smem, s);
  }
}

}  // namespace

namespace {
DqJob dq_job(const uint8_t* codes, const uint8_t* scales, uint16_t* out, long long rows, int K,
             const int32_t* counts, int rows_per_expert, const int32_t* src_group) {
  DqJob j{};
  if (rows <= 0) return j;
  const long long words_per_row = K / 8;
  j.codes = reinterpret_cast<const uint32_t*>(codes);
  j.scales = scales;
  j.out = reinterpret_cast<uint4*>(out);
  j.words = rows * words_per_row;
  j.words_per_group =
      counts ? (long long)(rows_per_expert > 0 ? rows_per_expert : 1) * words_per_row : j.words;
  j.counts = counts;
  j.src_group = src_group;
  return j;
}

cudaError_t launch_dq(const DqJob& j0, const DqJob& j1, cudaStream_t s) {
  const long long units = dq_units(j0) + dq_units(j1);
  if (units == 0) return cudaSuccess;
  long long grid = (units + 7) / 8;
  const long long cap = (long long)num_sms() * 8;
  if (grid > cap) grid = cap;
  return launch_k(dequant_kernel, dim3((unsigned)grid), dim3(256), 0, s, j0, j1);
}
}  // namespace

cudaError_t launch_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, uint16_t* out,
                                 long long rows, int K, cudaStream_t s, const int32_t* counts,
                                 int rows_per_expert, const int32_t* src_group) {
  return launch_dq(dq_job(codes, scales, out, rows, K, counts, rows_per_expert, src_group),
                   DqJob{}, s);
}

cudaError_t launch_dequant_mxfp4_pair(const uint8_t* codes0, const uint8_t* scales0,
                                      uint16_t* out0, long long rows0, int K0,
                                      const uint8_t* codes1, const uint8_t* scales1,
                                      uint16_t* out1, long long rows1, int K1, cudaStream_t s,
                                      const int32_t* counts, int rows_per_expert0,
                                      int rows_per_expert1, const int32_t* src_group) {
  return launch_dq(
      dq_job(codes0, scales0, out0, rows0, K0, counts, rows_per_expert0, src_group),
      dq_job(codes1, scales1, out1, rows1, K1, counts, rows_per_expert1, src_group), s);
}

cudaError_t launch_fp4_expert_gemv(const uint8_t* codes, const uint8_t* scales, const uint16_t* x,
                                   uint16_t* out, const int32_t* counts, const int32_t* offsets,
                                   const int32_t* active, const int32_t* n_active, int slots,
                                   int E, int K, int ncols, int situ, float beta, float lbeta,
                                   int* err, cudaStream_t s) {
  if (slots <= 0) return cudaSuccess;
  GemvArgs a{};
  a.codes = codes;
  a.scales = scales;
  a.x = x;
  a.out = out;
  a.counts = counts;
  a.offsets = offsets;
  a.active = active;
  a.n_active = n_active;
  a.err = err;
  a.K = K;
  a.ncols = ncols;
  a.situ = make_situ_params(beta, lbeta);
  return situ ? launch_expert_kernel<2>(a, slots, E, s) : launch_expert_kernel<1>(a, slots, E, s);
}

}  // namespace lmoe
