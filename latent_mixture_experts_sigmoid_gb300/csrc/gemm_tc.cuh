// Host interface of the tcgen05 GEMM (internal to liblmoe.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lmoe_internal.cuh"

namespace lmoe {

// Kernel parameters (passed by value).
struct GemmParams {
  int tok_on_m;            // 1: MMA M side = token rows; 0: M side = weight rows
  int M_feat;              // output features = weight rows per group
  int K;                   // reduction length (multiple of 64)
  int bn;                  // MMA N (16..256, multiple of 16)
  int num_groups;          // groups (experts); 1 for a dense GEMM
  const int* grp_count;    // [G] token rows per group (grouped) or NULL
  const int* grp_offset;   // [G] first token row per group (grouped) or NULL
  const int* tile_prefix;  // [G+1] prefix sums of token tiles per group, or NULL (dense)
  int T_dense;             // token rows of a dense GEMM
  int splits;              // split-K factor (each split >= 1 K block)
  void* out;               // bf16 [rows, ldo], or fp32 [splits][rows, ldo]
  int ldo;
  long long split_stride;  // elements between fp32 split partials
  int out_fp32;
  const uint16_t* add;     // bf16 [rows, ldo] added before rounding, or NULL
  int stages;
  uint32_t tmem_cols;
  int fuse_situ;           // W tile = 128 gate rows + the matching 128 up rows; the epilogue
                           // writes bf16(SituGLU(bf16(G))) [rows, M_feat/2].  Tokens on M:
                           // one 256-row B operand; weights on M: the two halves as two
                           // M = 128 MMAs into two accumulators (the kernel's swap-form
                           // instance)
  int mcast;               // 1: launched in clusters of two CTAs (the gemm_tc_kernel<true>
                           // form) that share an operand tile by TMA multicast; dense or
                           // grouped, tokens on M, 256-row weight tiles, no split-K
  int w2_row0;             // > 0: weight rows from w2_row0 on are rows (row - w2_row0) of the
                           // second weight map (weights on M only)
  int tma_store;           // 1: bf16 outputs with tokens on M leave full 32-row blocks by
                           // bulk tensor stores through the output tensor map
  SituParams sp;
};

// One GEMM launch:  out[tok, f] = sum_c X[tok, c] W[g*M_feat + f, c] (+ add).
struct GemmDesc {
  const uint16_t* W;       // [G*M_feat, K] bf16 (or [w_rows, K])
  long long w_rows;        // > 0: W has only this many rows; the rest of the tiles read zeros
  const uint16_t* X;       // [x_rows, K] bf16
  long long x_rows;
  int K, M_feat, G;
  const int* grp_count;    // device, grouped only
  const int* grp_offset;   // device, grouped only
  const int* tile_prefix;  // device, grouped only (token tile = 128 if tok_on_m, else bn)
  int T_dense;
  int tok_on_m, bn, splits;
  void* out;
  int ldo;
  int out_fp32;
  long long split_stride;
  const uint16_t* add;
  int max_units;           // > 0: known upper bound on work units (caps the grid)
  int fuse_situ;           // see GemmParams; tokens on M: bn == 256; weights on M: bn <= 128;
                           // splits == 1
  const uint16_t* W2;      // optional second weight matrix [w2_rows, K] bf16, stacked after
  long long w2_rows;       // the first w2_row0 rows of W (weights on M, w2_row0 % 128 == 0;
  int w2_row0;             // rows of the stack beyond w2_row0 + w2_rows read as zeros)
  float beta, linear_beta;
};

cudaError_t launch_gemm(const GemmDesc& g, cudaStream_t stream);
int read_device_error(int clear);

}  // namespace lmoe
