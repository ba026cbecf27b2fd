/*
 * lmoe.h -- C ABI of the GB300 (sm_103a) latent-MoE layer forward.
 *
 * The operations follow three pages:
 *   [vLLM-50088]   vLLM PR #50088, "[MoE] Latent-MoE runner, fused MoE tail,
 *                  SituGLU activation and single-group top-k routing";
 *   [TRTLLM-20541] TensorRT-LLM PR #20541, "Kimi K3 MoE decode: router GEMM and
 *                  routing kernel on a router stream";
 *   [vLLM-runner]  vLLM API page vllm.models.kimi_k3.amd.latent_moe_runner
 *                  (ROCmLatentMoERunner).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; it must
 *     stay valid until the work enqueued on `stream` has finished.  Tensors are
 *     dense and row-major (last index fastest).  Every pointer must be 16-byte
 *     aligned.
 *   - Every tensor pointer must address memory allocated on the CURRENT
 *     device (cudaGetDevice): each call asks the runtime for the attributes of
 *     every pointer it is given (cudaPointerGetAttributes) after the argument
 *     checks and refuses host memory (pinned or pageable), managed memory and
 *     another device's memory with LMOE_ERR_DEVICE, launching nothing.  The
 *     GEMMs of the layer read operand tiles through tensor maps that pairs of
 *     CTAs share on this GPU, so no call may be handed another GPU's memory.
 *     A pointer the runtime cannot describe is refused the same way.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     The calls are asynchronous: the return code covers argument validation
 *     and launch errors only.  No call synchronises the host with the device
 *     and no call allocates device memory; scratch memory is the caller's
 *     workspace.  The enqueued work can be captured in a CUDA graph.
 *   - On a validation error nothing is launched and a negative lmoe_status is
 *     returned.  A zero-sized problem (T == 0, N == 0, E == 0) returns LMOE_OK
 *     and launches nothing.
 *   - Weights (the members of lmoe_weights, the `w` of lmoe_linear and the
 *     e_score_correction_bias of moe_route) are read-only model parameters.
 *     Kernels launch with programmatic dependent launch and may start reading
 *     them before the preceding work on `stream` has finished; work that
 *     writes a weight must be separated from the call by an event or a
 *     synchronisation, not by stream order alone.  Activations (hidden states,
 *     router logits) are read only after the preceding work has finished.
 *   - bf16 values are carried as raw 16-bit patterns (lmoe_bf16).
 *   - Internal waits in the tensor-core kernels are bounded; if one ever gives
 *     up, the kernel records a code in a device error word and returns early
 *     (its outputs are then undefined).  lmoe_device_error() reads that word.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMOE_OK = 0,
  LMOE_ERR_NULL = -1,        /* a required pointer is NULL                     */
  LMOE_ERR_DIM = -2,         /* a size is out of range or not a supported multiple */
  LMOE_ERR_UNSUPPORTED = -3, /* n_group/topk_group other than 1                 */
  LMOE_ERR_BETA = -4,        /* beta <= 0 or not finite                         */
  LMOE_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than required         */
  LMOE_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed               */
  LMOE_ERR_ALIGN = -7,       /* a pointer is not 16-byte aligned                */
  LMOE_ERR_DEVICE = -8       /* a pointer is not device memory of the current   */
                             /* device (host, managed or another GPU's memory)  */
} lmoe_status;

typedef uint16_t lmoe_bf16;

/* ------------------------------------------------------------------------ */
/* Routing: [vLLM-50088] commit 1 (single-group fast path of grouped top-k:   */
/* with n_group == 1 and topk_group == 1 it is plain top-k over all experts) */
/* and commit 4 (DeepSeekV3 routing on FP32 logits).                          */
/*                                                                            */
/*   s[t,e]   = sigmoid(router_logits[t,e])  (fp32, a fixed IEEE operation     */
/*              sequence so that the selection is reproducible to the bit)    */
/*   key[t,e] = s[t,e] + e_score_correction_bias[e]    (selection only)       */
/*   topk_ids[t,:]     = the topk experts of largest key, in descending key    */
/*                       order; equal keys go to the lower expert index        */
/*   topk_weights[t,j] = s[t,ids_j] / sum_j s[t,ids_j] * routed_scaling_factor */
/*                       (without the division when renormalize == 0)          */
/*                                                                            */
/* router_logits [T,E] fp32; e_score_correction_bias [E] fp32 or NULL (zero); */
/* topk_ids [T,topk] int32 and topk_weights [T,topk] fp32 are outputs.         */
/* Limits: 1 <= E <= 1024, 1 <= topk <= min(E, 32), n_group == topk_group == 1 */
/* (else LMOE_ERR_UNSUPPORTED).  NaN logits are not supported.                */
/* ------------------------------------------------------------------------ */
int moe_route(const float* router_logits, const float* e_score_correction_bias,
              int T, int E, int topk, int n_group, int topk_group,
              int renormalize, float routed_scaling_factor,
              int32_t* topk_ids, float* topk_weights, void* stream);

/* ------------------------------------------------------------------------ */
/* SituGLU: [vLLM-50088] commit 2 (formula, dense and masked kernels, fp32   */
/* arithmetic, written straight to the output) and commit 3 (beta required;  */
/* linear_beta <= 0 means unset and up passes through).                       */
/*                                                                            */
/*   gate_out = beta * tanh(gate / beta) * sigmoid(gate)                      */
/*   up_out   = linear_beta * tanh(up / linear_beta)   if linear_beta > 0     */
/*            = up                                      otherwise             */
/*   out      = gate_out * up_out                                             */
/*                                                                            */
/* situ_and_mul: in [N, 2d] bf16 with gate = in[:, :d], up = in[:, d:];      */
/* out [N, d] bf16.  Requires d % 8 == 0.  beta <= 0 -> LMOE_ERR_BETA.        */
/* ------------------------------------------------------------------------ */
int situ_and_mul(const lmoe_bf16* in, lmoe_bf16* out, int64_t N, int d,
                 float beta, float linear_beta, void* stream);

/* masked_situ_and_mul: batched MoE layout.  in [E, T_max, 2d] bf16, out      */
/* [E, T_max, d] bf16, expert_num_tokens [E] int32 on the device.  Row t of   */
/* expert e is computed iff t < expert_num_tokens[e]; every other output row  */
/* is left untouched (its bytes are never written).  Counts outside           */
/* [0, T_max] are clamped to that range on the device.  Requires d % 8 == 0.  */
int masked_situ_and_mul(const lmoe_bf16* in, lmoe_bf16* out,
                        const int32_t* expert_num_tokens, int E, int T_max,
                        int d, float beta, float linear_beta, void* stream);

/* ------------------------------------------------------------------------ */
/* The latent-MoE layer forward on one GPU: [vLLM-runner] _fused_forward and */
/* _shard_up_proj_tail, [vLLM-50088] commits 1-3 and 7, [TRTLLM-20541]       */
/* Commit 2 (decode order).                                                   */
/*                                                                            */
/*   ids, w = moe_route(router_logits)                                        */
/*   Z      = bf16(hidden W_down^T)                          [T, latent]       */
/*   rows   = (token, slot) pairs grouped by expert, tokens ascending         */
/*   per expert e:  G = bf16(Z W13_e^T)                      [n_e, 2*inter]     */
/*                  A = bf16(SituGLU(G))                     [n_e, inter]       */
/*                  Y = bf16(A W2_e^T)                       [n_e, latent]      */
/*   C[t]   = sum_j w[t,j] * Y[row(t,j)]      (fp32, the complete routed sum)  */
/*   N      = bf16(C / sqrt(mean(C^2) + rms_eps) * norm_w)                     */
/*   Sh     = bf16(bf16(SituGLU(bf16(hidden Ws13^T))) Ws2^T)  shared expert    */
/*   out    = bf16(N W_up^T + Sh)                (Sh added in the GEMM epilogue) */
/*                                                                            */
/* Limits: hidden % 128 == 0, latent % 128 == 0, latent <= 8192,            */
/* inter % 64 == 0, shared_inter % 64 == 0 (when the shared expert is        */
/* present), the routing limits above, T >= 0, T * topk <= 2^30 and          */
/* T * topk * max(2 * inter, latent) <= 2^40 (LMOE_ERR_DIM otherwise).        */
/* ------------------------------------------------------------------------ */
typedef struct lmoe_dims {
  int T;                 /* tokens                                           */
  int hidden;            /* H                                                */
  int latent;            /* L                                                */
  int num_experts;       /* E                                                */
  int topk;              /* k                                                */
  int inter;             /* d: per-expert intermediate size                  */
  int shared_inter;      /* ds: shared-expert intermediate size              */
  int n_group;           /* must be 1                                        */
  int topk_group;        /* must be 1                                        */
  int renormalize;       /* 1: w = s / sum(s) * rsf;  0: w = s * rsf          */
  float routed_scaling_factor;
  float beta;            /* SituGLU beta (> 0)                               */
  float linear_beta;     /* SituGLU linear_beta (<= 0: unset)                */
  float rms_eps;         /* RMSNorm epsilon (inside the square root)         */
} lmoe_dims;

typedef struct lmoe_weights {
  const lmoe_bf16* w_down;  /* [L, H]                                        */
  const lmoe_bf16* w13;     /* [E, 2d, L]: rows 0..d-1 gate, d..2d-1 up       */
  const lmoe_bf16* w2;      /* [E, L, d]                                     */
  const lmoe_bf16* ws13;    /* [2ds, H] or NULL (no shared expert)           */
  const lmoe_bf16* ws2;     /* [H, ds] (NULL iff ws13 is NULL)                */
  const lmoe_bf16* norm_w;  /* [L] RMSNorm gamma, or NULL (= ones)           */
  const lmoe_bf16* w_up;    /* [H, L]                                        */
  const float* e_score_correction_bias; /* [E] or NULL (= zeros)             */
} lmoe_weights;

/* Stages of one forward, in launch order (for per-stage timing).            */
enum {
  LMOE_STAGE_ROUTE = 0,        /* routing                                    */
  LMOE_STAGE_DOWN = 1,         /* latent down-projection GEMM                */
  LMOE_STAGE_PERMUTE = 2,      /* counts, offsets, rows                      */
  LMOE_STAGE_SCATTER = 3,      /* routed input into expert-major rows        */
  LMOE_STAGE_GEMM1 = 4,        /* grouped expert GEMM1                       */
  LMOE_STAGE_SITU = 5,         /* SituGLU of the experts                     */
  LMOE_STAGE_GEMM2 = 6,        /* grouped expert GEMM2                       */
  LMOE_STAGE_COMBINE = 7,      /* top-k combine + RMSNorm                    */
  LMOE_STAGE_SHARED1 = 8,      /* shared expert GEMM1 + SituGLU              */
  LMOE_STAGE_SHARED2 = 9,      /* shared expert GEMM2                        */
  LMOE_STAGE_UP = 10,          /* up-projection + shared add                 */
  LMOE_NUM_STAGES = 11
};

/* Optional outputs for inspection (any member may be NULL / 0).              */
typedef struct lmoe_debug {
  int32_t* topk_ids;          /* [T, k]                                      */
  float* topk_weights;        /* [T, k]                                      */
  int32_t* expert_num_tokens; /* [E]                                         */
  int32_t* expert_offsets;    /* [E+1]: expert e owns rows off[e]..off[e+1]-1 */
  int32_t* row_of;            /* [T, k]: permuted row of (token, slot)       */
  void** stage_events;        /* LMOE_NUM_STAGES + 1 cudaEvent_t (host array, */
                              /* created by the caller): event 0 is recorded */
                              /* before the first stage, event i+1 after      */
                              /* stage i, all on `stream`.                    */
} lmoe_debug;

/* Bytes of device workspace latent_moe_forward needs for these dims (0 on   */
/* invalid dims).  Depends on the dims only.                                  */
size_t latent_moe_workspace_bytes(const lmoe_dims* dims);

/* Byte offsets of the layer's intermediate buffers inside the workspace, in */
/* this order (LMOE_WS_COUNT entries), for inspection after a call:           */
/*   0 topk_ids int32 [T,k]    1 topk_weights fp32 [T,k]  2 counts int32 [E]   */
/*   3 offsets int32 [E+1]     4 row_of int32 [T,k]       5 Z bf16 [T,L]       */
/*   6 A bf16 [T*k,L]          7 G bf16 [T*k,2d]          8 act bf16 [T*k,d]   */
/*   9 Y bf16 [T*k,L]         10 N bf16 [T,L]            11 Gs bf16 [T,2ds]    */
/*  12 As bf16 [T,ds]         13 Sh bf16 [T,H]                                 */
/*  14 logits fp32 [T, Ep] with Ep = E rounded up to a multiple of 128 (the   */
/*     router logits of latent_moe_forward_router, columns E..Ep-1 unused)    */
/* Z and Sh hold data only when the call did not split K (T > 128).  G holds */
/* data only if inter % 128 != 0 (otherwise SituGLU runs in GEMM1's          */
/* epilogue); at T > 128, Gs only if shared_inter % 128 != 0 (otherwise it   */
/* runs in the shared GEMM1's epilogue).                                      */
/* Returns LMOE_OK or a validation error.                                     */
enum { LMOE_WS_COUNT = 15 };
int latent_moe_workspace_offsets(const lmoe_dims* dims, size_t* offsets);

/* Number of kernel launches latent_moe_forward makes for these dims (0 on   */
/* invalid dims), without the optional debug copies.  Uses the current       */
/* device's SM count.                                                         */
int latent_moe_launch_count(const lmoe_dims* dims, int has_shared_expert);

/* hidden [T, H] bf16, router_logits [T, E] fp32, out [T, H] bf16; workspace  */
/* at least latent_moe_workspace_bytes(dims) bytes, 256-byte aligned, not     */
/* shared with a concurrent call.  dbg may be NULL.  The shared expert runs  */
/* on a library-owned second stream kept for this (device, `stream`) pair,    */
/* forked from `stream` and joined back to it by events (also inside a       */
/* stream capture), so all of the call's work is ordered after earlier work  */
/* on `stream` and before later.  Calls on different streams share no        */
/* second stream: host threads may call concurrently, each on its own stream */
/* and workspace, and one of them may be capturing (capture in thread-local  */
/* or relaxed mode: during a global-mode capture the runtime may refuse      */
/* calls it deems unsafe in every other thread).  The second                 */
/* stream of a caller stream is created by its first call (also inside a     */
/* capture; up to 64 caller streams per device); a call without one runs     */
/* every stage on `stream` (same results).  With dbg->stage_events every      */
/* stage runs on `stream`, one after another.                                 */
int latent_moe_forward(const lmoe_dims* dims, const lmoe_weights* weights,
                       const lmoe_bf16* hidden, const float* router_logits,
                       lmoe_bf16* out, void* workspace, size_t workspace_bytes,
                       const lmoe_debug* dbg, void* stream);

/* The layer forward on a routing done ahead of it (pre-routing: the         */
/* TensorRT-LLM PR #20541 launches the routing of a decode step early on its */
/* own stream and the MoE layer consumes its result after an event join).    */
/* topk_ids [T, k] int32 and topk_weights [T, k] fp32 as moe_route writes    */
/* them (same dims; the weights already renormalised and scaled) replace     */
/* router_logits; the layer skips its routing kernel and otherwise runs as    */
/* latent_moe_forward (same arguments, workspace and errors; one launch      */
/* fewer than latent_moe_launch_count).  The routing must be complete on the */
/* GPU before the call's work starts (same stream, or an event the caller    */
/* waits on).  The ids of a token must be distinct, as moe_route writes     */
/* them.  An id outside [0, E) is read as expert 0 and the device error word */
/* records 7 (the output is then wrong, but no memory outside the call's     */
/* buffers is touched).                                                       */
int latent_moe_forward_routed(const lmoe_dims* dims, const lmoe_weights* weights,
                              const lmoe_bf16* hidden, const int32_t* topk_ids,
                              const float* topk_weights, lmoe_bf16* out, void* workspace,
                              size_t workspace_bytes, const lmoe_debug* dbg, void* stream);

/* ------------------------------------------------------------------------ */
/* Router GEMM ([TRTLLM-20541] Commit 2: the router GEMM produces the logits */
/* the routing kernel reads; "fused router+down projection" is the           */
/* configuration that computes it in one pass with the latent down           */
/* projection; [vLLM-50088] commit 4: DeepSeekV3 routing takes FP32 logits): */
/*                                                                            */
/*   logits[t, e] = sum_h hidden[t, h] * w_router[e, h]   (fp32 accumulation, */
/*                                                         stored fp32)       */
/*                                                                            */
/* hidden [T, H] bf16, w_router [E, H] bf16 (PyTorch Linear layout, no bias), */
/* logits [T, E] fp32 output.  Requires 1 <= E <= 1024, H % 64 == 0, T >= 0. */
/* The workspace (at least lmoe_router_logits_workspace_bytes(T, E, H)       */
/* bytes, 256-byte aligned) holds split-K partials at T <= 128 and padded    */
/* rows when E % 128 != 0.                                                    */
/* ------------------------------------------------------------------------ */
size_t lmoe_router_logits_workspace_bytes(int T, int E, int H);
int lmoe_router_logits(const lmoe_bf16* hidden, const lmoe_bf16* w_router, float* logits, int T,
                       int E, int H, void* workspace, size_t workspace_bytes, void* stream);

/* The layer forward with its router GEMM: latent_moe_forward on the logits  */
/* hidden W_router^T (fp32, as lmoe_router_logits computes them) instead of   */
/* logits passed in.  w_router [num_experts, hidden] bf16.  At T <= 128 the  */
/* router rows are stacked after the down-projection's rows in one split-K   */
/* GEMM launch over the hidden states (the fused router + down projection;   */
/* a small kernel sums the logit partials for the routing); above, the       */
/* router GEMM is its own launch ahead of the routing (on the second stream, */
/* beside the down-projection).  Same workspace, limits and errors as         */
/* latent_moe_forward; the logits are left in the workspace (entry 14).      */
int latent_moe_forward_router(const lmoe_dims* dims, const lmoe_weights* weights,
                              const lmoe_bf16* w_router, const lmoe_bf16* hidden, lmoe_bf16* out,
                              void* workspace, size_t workspace_bytes, const lmoe_debug* dbg,
                              void* stream);

/* Kernel launches of latent_moe_forward_router for these dims (0 on invalid */
/* dims), as latent_moe_launch_count counts them.                             */
int latent_moe_launch_count_router(const lmoe_dims* dims, int has_shared_expert);

/* ------------------------------------------------------------------------ */
/* Block-scaled (MXFP4) routed experts ([vLLM-50088] commits 4-5: the        */
/* TRTLLM-Gen MXFP4 MoE backend runs this layer's routed experts, SituGLU    */
/* acting on the dequantized gate/up; [TRTLLM-20541]: Kimi K3 decode with    */
/* the MXFP4 MoE).  Each expert matrix [rows, K] is stored as               */
/*   codes  uint8 [rows, K/2]:  two 4-bit E2M1 values per byte, element 2i  */
/*          in the low nibble of byte i, element 2i+1 in the high nibble     */
/*          (E2M1: bit 3 sign, bits 2-1 exponent with bias 1, bit 0         */
/*          mantissa; exponent 0 is subnormal: 0 or 0.5)                    */
/*   scales uint8 [rows, K/32]: one power of two per 32 consecutive elements */
/*          of a row, 2^(s - 127) (E8M0; 255 is NaN)                        */
/* and weight[r, c] = E2M1(code[r, c]) * 2^(scale[r, c/32] - 127).  The      */
/* activations stay bf16 (W4A16): the expert GEMMs compute with the exact   */
/* dequantized weights.  Scale exponents 2..252 keep every weight a bf16     */
/* value; outside that range the prefill path rounds the weight to bf16.     */
/* ------------------------------------------------------------------------ */
typedef struct lmoe_mxfp4_experts {
  const uint8_t* w13_codes;   /* [E, 2d, L/2] (rows as lmoe_weights.w13)     */
  const uint8_t* w13_scales;  /* [E, 2d, L/32]                               */
  const uint8_t* w2_codes;    /* [E, L, d/2]                                 */
  const uint8_t* w2_scales;   /* [E, L, d/32]                                */
} lmoe_mxfp4_experts;

/* out [rows, K] bf16 = the dequantized weights (rounded to bf16, exact for */
/* scale exponents 2..252).  K % 32 == 0, rows >= 0; codes and out 16-byte  */
/* aligned device pointers of the current device.                           */
int lmoe_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, lmoe_bf16* out,
                       int64_t rows, int K, void* stream);

/* Workspace bytes of latent_moe_forward_mxfp4 (0 on invalid dims): the      */
/* workspace of latent_moe_forward, plus at T > 16 (inter % 128 == 0) room   */
/* for H = min(E, T*topk / 17) experts' weights dequantized to bf16          */
/* (H * 3 * inter * latent * 2 bytes) and their tables, or with             */
/* inter % 128 != 0 at T > 128 room for every expert's (H = E).              */
size_t latent_moe_workspace_bytes_mxfp4(const lmoe_dims* dims);

/* The layer forward with MXFP4 routed experts: latent_moe_forward with      */
/* weights->w13 and weights->w2 unused (may be NULL) and the experts' GEMMs  */
/* on `experts` instead.  The two expert stages read the 4-bit weights      */
/* directly (one kernel per stage over the active experts, GEMM1's gate/up  */
/* and SituGLU in one kernel), except that the experts that received more    */
/* than 16 tokens, when at least 4 did (the device picks them from the       */
/* routing; inter % 128 == 0), are dequantized into the workspace each call  */
/* and run on the bf16 tensor-core path.  With inter % 128 != 0 above 128    */
/* tokens every expert that received tokens takes that path.  (A caller that */
/* runs large batches repeatedly on the same weights can also dequantize     */
/* once with lmoe_dequant_mxfp4 and call latent_moe_forward.)                */
/* Limits: those of latent_moe_forward and latent <= 4096, inter <= 4096.    */
/* The four expert pointers are required (LMOE_ERR_NULL), codes and scales   */
/* 16-byte aligned (LMOE_ERR_ALIGN), device memory of the current device     */
/* (LMOE_ERR_DEVICE).  In the 4-bit kernels the expert inputs enter         */
/* as f16 scaled per token by a power of two (exact for every element within */
/* 2^30 of the token's largest; smaller ones round to the f16 subnormal grid)*/
/* and the products are summed in fp32 on the tensor cores.                  */
/* The workspace layout (latent_moe_workspace_offsets) is the same.          */
int latent_moe_forward_mxfp4(const lmoe_dims* dims, const lmoe_weights* weights,
                             const lmoe_mxfp4_experts* experts, const lmoe_bf16* hidden,
                             const float* router_logits, lmoe_bf16* out, void* workspace,
                             size_t workspace_bytes, const lmoe_debug* dbg, void* stream);

/* Kernel launches of latent_moe_forward_mxfp4 (0 on invalid dims).         */
int latent_moe_launch_count_mxfp4(const lmoe_dims* dims, int has_shared_expert);

/* The layer forward without a caller workspace.  The pages have no          */
/* counterpart to this entry point; it exists for callers that cannot         */
/* allocate device memory: a plugin that an inference runtime calls with only */
/* its input and output buffers (the runtime owns every allocation), host     */
/* code with no allocator of its own, or a latency path where cudaMalloc is   */
/* not allowed because it may synchronise the device.                         */
/* Same computation, arguments and errors as latent_moe_forward, except that  */
/* the scratch is a 32 MiB array held by the library in device memory (every */
/* GPU that loads the library keeps it until the process exits).  Calls whose */
/* latent_moe_workspace_bytes exceeds 32 MiB return LMOE_ERR_WORKSPACE and    */
/* launch nothing (the 896-expert, hidden-7168 layer fits up to T = 15).      */
/* Every call looks up the array's address on the current device            */
/* (cudaGetSymbolAddress; not cached, so it stays valid across a device      */
/* reset).  With lazy module loading the first lookup on a device loads the  */
/* library's module there, which reserves the 32 MiB and may synchronise the */
/* device: make that first call (or any other call of the library) on each    */
/* device before a latency-critical path and before any stream capture.       */
/* No call allocates.  Every call on a device shares the one array, which   */
/* keeps the previous call's contents (nothing in it has to start at zero:   */
/* each call writes every scratch value it reads), so calls that may overlap */
/* on the GPU (different streams, or host threads) race; serialise them on   */
/* one stream.                                                                */
int latent_moe_forward_noalloc(const lmoe_dims* dims, const lmoe_weights* weights,
                               const lmoe_bf16* hidden, const float* router_logits,
                               lmoe_bf16* out, const lmoe_debug* dbg, void* stream);

/* ------------------------------------------------------------------------ */
/* Dense linear layer on the same tensor-core GEMM engine (the up-projection */
/* with its shared-output add, [vLLM-runner] _shard_up_proj_tail:             */
/* hidden_shard.addmm_(latent, up_proj_shard.t())):                           */
/*   out[t, n] = bf16( sum_c x[t, c] * w[n, c]  (+ add[t, n]) )                */
/* x [T, K] bf16, w [N, K] bf16 (PyTorch Linear layout), add [T, N] bf16 or  */
/* NULL, out [T, N] bf16.  fp32 accumulation, one rounding.  Requires          */
/* K % 64 == 0, N % 128 == 0, T >= 0.  No workspace (no split K).             */
/* ------------------------------------------------------------------------ */
int lmoe_linear(const lmoe_bf16* x, const lmoe_bf16* w, const lmoe_bf16* add, lmoe_bf16* out,
                int T, int N, int K, void* stream);

/* ------------------------------------------------------------------------ */
/* Utilities                                                                  */
/* ------------------------------------------------------------------------ */
/* Static description of a status code (never NULL).                         */
const char* lmoe_status_string(int status);

/* Reads (and with clear != 0 resets) the device error word of the current    */
/* device: 0 = nothing went wrong; 1-6 = a bounded wait of the tensor-core    */
/* GEMM gave up; 7 = latent_moe_forward_routed met an expert id outside      */
/* [0, E).  The first code written stays until cleared.  Synchronises the    */
/* device.                                                                    */
/* Returns the word, or LMOE_ERR_CUDA if it cannot be read.                   */
int lmoe_device_error(int clear);

/* ABI version of this header (major * 100 + minor).                          */
int lmoe_abi_version(void);

/* Work-unit walk of the grouped expert GEMM with tokens on M (the prefill    */
/* form), for inspection and tests; host only, launches nothing.  G groups   */
/* (experts) of count[g] >= 0 token rows, stored consecutively in group order */
/* (group g starts at the sum of the earlier counts); token tiles of 128 rows */
/* and nfeat feature tiles of 256 weight rows per group (M_feat = 256*nfeat). */
/* paired = 1: the CTA-pair form (two CTAs share one operand tile; nfeat    */
/* even), paired = 0: one CTA per unit.  Writes, for unit u in walk order and */
/* CTA rank r < 1 + paired, five ints at out[(u * (1 + paired) + r) * 5]:    */
/* first token row, valid token rows, first weight row, feature tile, and 1  */
/* if the pair shares its token tile (0 if it shares the weight tile).  A     */
/* persistent launch of n CTAs (or pairs) gives unit u to CTA (pair) u % n.  */
/* Writes at most max_units units (nothing if out is NULL); returns the unit  */
/* count, or LMOE_ERR_DIM for G outside 1..1024, a negative count, nfeat < 1  */
/* or odd with paired = 1, or more than 2^30 rows.                            */
int lmoe_gemm_unit_walk(int G, const int* count, int nfeat, int paired, int* out, int max_units);

#ifdef __cplusplus
}
#endif

#endif /* LMOE_H */
