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

// E8M0 scale exponent -> 2^(s - 127) in fp32 (s = 0: the subnormal 2^-127;
// s = 255: NaN)
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  const uint32_t bits = s == 0u ? 0x00400000u : (s == 255u ? 0x7FC00000u : s << 23);
  return __uint_as_float(bits);
}

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int q) {
  return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// ---- dequantization: out[r, :] = bf16(w[r, :]) --------------------------------
// One warp per row at a time; a lane converts 8 codes (one 32-bit word) into 8
// bf16 values (one 16-byte store) per step.
__global__ void __launch_bounds__(256)
dequant_kernel(const uint32_t* __restrict__ codes, const uint8_t* __restrict__ scales,
               uint4* __restrict__ out, long long rows, int words_per_row, int nblk) {
  pdl_trigger();
  pdl_wait();   // out may still be read by the previous forward's GEMMs
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const uint32_t* cr = codes + r * words_per_row;
    const uint8_t* sr = scales + r * nblk;
    uint4* orow = out + r * words_per_row;
#pragma unroll 4
    for (int g = lane; g < words_per_row; g += 32) {
      const float sc = e8m0_to_f32(__ldg(sr + (g >> 2)));
      float v[8];
      e2m1x8_to_f32(__ldg(cr + g), v);
      orow[g] = make_uint4(pack_bf16x2(v[0] * sc, v[1] * sc), pack_bf16x2(v[2] * sc, v[3] * sc),
                           pack_bf16x2(v[4] * sc, v[5] * sc), pack_bf16x2(v[6] * sc, v[7] * sc));
    }
  }
}

// ---- decode expert GEMV ---------------------------------------------------------
constexpr int kGemvWarps = 8;
constexpr int kGemvNT = 2;   // tokens per pass over the staged input

struct GemvArgs {
  const uint8_t* codes;     // [E, kRows * ncols, K/2]
  const uint8_t* scales;    // [E, kRows * ncols, K/32]
  const uint16_t* x;        // expert-major input rows [rows, K] bf16
  uint16_t* out;            // [rows, ncols] bf16
  const int32_t* counts;    // [E]
  const int32_t* offsets;   // [E+1]
  const int32_t* active;    // active expert of each slot
  const int32_t* n_active;  // number of active experts
  int K, nblk, ncols, lr_log2;
  SituParams situ;
};

// kRows = 2: gate row c and up row ncols + c, SituGLU of the two sums;
// kRows = 1: one row per output column.  kBPL: scale blocks a lane owns in a
// row (K/32 blocks over the 2^lr_log2 lanes of the row); kU: columns a warp
// takes per row group.
template <int kRows, int kBPL, int kU>
__global__ void __launch_bounds__(kGemvWarps * 32, 2) fp4_gemv_kernel(GemvArgs a) {
  extern __shared__ float4 xs[];   // [kGemvNT][K/4], piece-major within a token
  pdl_trigger();
  pdl_wait();
  const int slot = blockIdx.y;
  if (slot >= a.n_active[0]) return;
  const int e = a.active[slot];
  const int n = a.counts[e], row0 = a.offsets[e];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LR = 1 << a.lr_log2, RS = 32 >> a.lr_log2;
  const int grp = lane >> a.lr_log2, li = lane & (LR - 1);
  const int K = a.K, nblk = a.nblk, ncols = a.ncols;
  const long long ebase = (long long)e * kRows * ncols;
  const int c_warp = (blockIdx.x * kGemvWarps + warp) * kU * RS;
  // this lane's codes and scales, for every column, row and block it owns
  uint4 cw[kU][kRows][kBPL];
  uint32_t sv[kU][kRows][kBPL];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int c = c_warp + u * RS + grp;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const long long wrow = ebase + (long long)r * ncols + c;
#pragma unroll
      for (int i = 0; i < kBPL; ++i) {
        const int j = li + (i << a.lr_log2);
        if (c < ncols && j < nblk) {
          cw[u][r][i] = ld_stream(a.codes + wrow * (K >> 1) + j * 16);
          sv[u][r][i] = __ldg(a.scales + wrow * nblk + j);
        } else {
          cw[u][r][i] = make_uint4(0u, 0u, 0u, 0u);
          sv[u][r][i] = 127u;
        }
      }
    }
  }
  const int q4 = K >> 2;   // float4 per staged token
  for (int t0 = 0; t0 < n; t0 += kGemvNT) {
    const int nt = min(kGemvNT, n - t0);
    __syncthreads();   // the previous pass is done reading xs
    const int g8 = K >> 3;
    for (int idx = threadIdx.x; idx < nt * g8; idx += blockDim.x) {
      const int t = idx / g8, m = idx - t * g8;
      const uint4 v =
          __ldg(reinterpret_cast<const uint4*>(a.x + (long long)(row0 + t0 + t) * K) + m);
      const int j = m >> 2, q = m & 3;
      xs[t * q4 + (2 * q) * nblk + j] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y),
                                                    bf16_hi(v.y));
      xs[t * q4 + (2 * q + 1) * nblk + j] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w),
                                                        bf16_hi(v.w));
    }
    __syncthreads();
    float acc[kU][kRows][kGemvNT];
#pragma unroll
    for (int u = 0; u < kU; ++u)
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kGemvNT; ++t) acc[u][r][t] = 0.0f;
#pragma unroll
    for (int i = 0; i < kBPL; ++i) {
      const int j = li + (i << a.lr_log2);
      if (j < nblk) {
        float bs[kU][kRows][kGemvNT];
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int t = 0; t < kGemvNT; ++t) bs[u][r][t] = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float xv[kGemvNT][8];
#pragma unroll
          for (int t = 0; t < kGemvNT; ++t) {
            if (t < nt) {
              const float4 p0 = xs[t * q4 + (2 * q) * nblk + j];
              const float4 p1 = xs[t * q4 + (2 * q + 1) * nblk + j];
              xv[t][0] = p0.x; xv[t][1] = p0.y; xv[t][2] = p0.z; xv[t][3] = p0.w;
              xv[t][4] = p1.x; xv[t][5] = p1.y; xv[t][6] = p1.z; xv[t][7] = p1.w;
            } else {
#pragma unroll
              for (int s = 0; s < 8; ++s) xv[t][s] = 0.0f;
            }
          }
#pragma unroll
          for (int u = 0; u < kU; ++u)
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
              float w[8];
              e2m1x8_to_f32(word(cw[u][r][i], q), w);
#pragma unroll
              for (int t = 0; t < kGemvNT; ++t) {
                if (t >= nt) continue;   // (warp-uniform)
#pragma unroll
                for (int s = 0; s < 8; ++s) bs[u][r][t] = fmaf(w[s], xv[t][s], bs[u][r][t]);
              }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const float sc = e8m0_to_f32(sv[u][r][i]);
#pragma unroll
            for (int t = 0; t < kGemvNT; ++t) acc[u][r][t] = fmaf(bs[u][r][t], sc, acc[u][r][t]);
          }
      }
    }
    // sum over the lanes of each row (xor offsets below LR stay in the group)
#pragma unroll
    for (int u = 0; u < kU; ++u)
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kGemvNT; ++t)
          for (int o = LR >> 1; o > 0; o >>= 1)
            acc[u][r][t] += __shfl_xor_sync(0xffffffffu, acc[u][r][t], o);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c_warp + u * RS + grp;
      if (c >= ncols) continue;
#pragma unroll
      for (int t = 0; t < kGemvNT; ++t) {
        if (t >= nt || (t & (LR - 1)) != li) continue;
        uint16_t o;
        if (kRows == 2) {
          // act = bf16(SituGLU(bf16(gate), bf16(up)))
          const uint32_t g2 = to_bf16(acc[u][0][t]);
          const uint32_t u2 = to_bf16(acc[u][kRows - 1][t]);
          o = (uint16_t)(situ2(g2, u2, a.situ) & 0xFFFFu);
        } else {
          o = to_bf16(acc[u][0][t]);
        }
        a.out[(long long)(row0 + t0 + t) * ncols + c] = o;
      }
    }
  }
}

int ilog2_ceil(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

template <int kRows, int kBPL>
cudaError_t launch_gemv_bpl(const GemvArgs& a, int slots, cudaStream_t s) {
  constexpr int kU = (8 / (kRows * kBPL)) > 1 ? 8 / (kRows * kBPL) : 1;
  auto kern = fp4_gemv_kernel<kRows, kBPL, kU>;
  const size_t smem = (size_t)kGemvNT * a.K * sizeof(float);
  if (smem > 48 * 1024) {
    // (set on every such launch: the attribute belongs to the current device)
    const cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  const int rs = 32 >> a.lr_log2;
  const int cpb = kGemvWarps * kU * rs;
  const dim3 grid((unsigned)ceil_div(a.ncols, cpb), (unsigned)slots);
  return launch_k(kern, grid, dim3(kGemvWarps * 32), smem, s, a);
}

template <int kRows>
cudaError_t launch_gemv_rows(const GemvArgs& a, int slots, cudaStream_t s) {
  const int bpl = (a.nblk + (1 << a.lr_log2) - 1) >> a.lr_log2;
  if (bpl <= 1) return launch_gemv_bpl<kRows, 1>(a, slots, s);
  if (bpl <= 2) return launch_gemv_bpl<kRows, 2>(a, slots, s);
  if (bpl <= 4) return launch_gemv_bpl<kRows, 4>(a, slots, s);
  return launch_gemv_bpl<kRows, 8>(a, slots, s);
}

}  // namespace

cudaError_t launch_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, uint16_t* out,
                                 long long rows, int K, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const long long warps = rows < (1ll << 20) ? rows : (1ll << 20);
  long long blocks = (warps + 7) / 8;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  return launch_k(dequant_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                  reinterpret_cast<const uint32_t*>(codes), scales, reinterpret_cast<uint4*>(out),
                  rows, K / 8, K / 32);
}

cudaError_t launch_fp4_expert_gemv(const uint8_t* codes, const uint8_t* scales, const uint16_t* x,
                                   uint16_t* out, const int32_t* counts, const int32_t* offsets,
                                   const int32_t* active, const int32_t* n_active, int slots,
                                   int K, int ncols, int situ, float beta, float lbeta,
                                   cudaStream_t s) {
  if (slots <= 0) return cudaSuccess;
  GemvArgs a;
  a.codes = codes;
  a.scales = scales;
  a.x = x;
  a.out = out;
  a.counts = counts;
  a.offsets = offsets;
  a.active = active;
  a.n_active = n_active;
  a.K = K;
  a.nblk = K / 32;
  a.ncols = ncols;
  a.lr_log2 = ilog2_ceil(a.nblk < 32 ? a.nblk : 32);
  a.situ = make_situ_params(beta, lbeta);
  return situ ? launch_gemv_rows<2>(a, slots, s) : launch_gemv_rows<1>(a, slots, s);
}

}  // namespace lmoe
