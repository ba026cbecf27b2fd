// Host interface of the MXFP4 expert-weight kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

// out [rows, K] bf16 = E2M1(codes) * 2^(scales - 127), rounded to bf16.
// codes [rows, K/2] (16-byte aligned), scales [rows, K/32]; K % 32 == 0.
// With counts: the rows_per_expert rows of expert e are left untouched when
// counts[e] == 0 (experts no token was routed to).  With src_group (needs
// counts): output expert j holds the weights of expert src_group[j] (a compact
// copy; rows counts the output rows, the source spans every src_group[j]).
cudaError_t launch_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, uint16_t* out,
                                 long long rows, int K, cudaStream_t s,
                                 const int32_t* counts = nullptr, int rows_per_expert = 0,
                                 const int32_t* src_group = nullptr);

// Two launch_dequant_mxfp4 jobs in one launch (the same counts and src_group).
cudaError_t launch_dequant_mxfp4_pair(const uint8_t* codes0, const uint8_t* scales0,
                                      uint16_t* out0, long long rows0, int K0,
                                      const uint8_t* codes1, const uint8_t* scales1,
                                      uint16_t* out1, long long rows1, int K1, cudaStream_t s,
                                      const int32_t* counts, int rows_per_expert0,
                                      int rows_per_expert1, const int32_t* src_group);

// Decode expert stage on MXFP4 weights (a persistent kernel, one block per
// SM): out[row, c] for the rows offsets[e] .. offsets[e] + counts[e] - 1 of
// each active expert e (active[0 .. *n_active - 1], slots >= *n_active), from
// the bf16 input rows x [rows, K].
//   situ != 0: codes [E, 2 * ncols, K/2]; out = bf16(SituGLU(bf16(x Wg^T),
//              bf16(x Wu^T))) with Wg rows 0..ncols-1, Wu rows ncols..;
//   situ == 0: codes [E, ncols, K/2]; out = bf16(x W^T).
// E experts; K % 64 == 0, K <= 4096, ncols % 16 == 0, codes and scales
// 16-byte aligned.  A bounded wait that runs out records 8 in the device error
// word `err`.
cudaError_t launch_fp4_expert_gemv(const uint8_t* codes, const uint8_t* scales, const uint16_t* x,
                                   uint16_t* out, const int32_t* counts, const int32_t* offsets,
                                   const int32_t* active, const int32_t* n_active, int slots,
                                   int E, int K, int ncols, int situ, float beta, float lbeta,
                                   int* err, cudaStream_t s);

}  // namespace lmoe
