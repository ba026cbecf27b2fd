// The C ABI of liblmoe.so (declared in include/lmoe.h): argument validation,
// the workspace layout and the schedule of kernels of one layer forward.
//
// Layer schedule (no host synchronisation, no allocation), following the data
// flow of the vLLM latent_moe_runner page (ROCmLatentMoERunner._fused_forward
// and _shard_up_proj_tail) on one device, with the stream layout of
// TensorRT-LLM PR #20541, Commit 2: the shared expert (steps 9-11) runs on a
// second stream forked from and joined back to the caller's by events, and at
// large T so do steps 1 and 3, beside the down-projection.  The pre-routed
// entry point (that PR's Commit 1) skips step 1.
//   1 route             ids, w                        (routing kernel)
//   2 down-projection   Z = X W_down^T                (tcgen05 GEMM)
//   3 permute           counts, offsets, row_of       (bitmap counting sort)
//   4 scatter           A[row_of[t,j]] = bf16(Z[t])
//   5 GEMM1 (grouped)   G = A W13_e^T                 (tcgen05 GEMM)
//   6 SituGLU           act = SituGLU(G)              (in GEMM1's epilogue at
//                                                      large T)
//   7 GEMM2 (grouped)   Y = act W2_e^T                (tcgen05 GEMM)
//   8 combine + norm    N = RMSNorm(sum_j w Y) * gamma
//   9 shared GEMM1      Gs = X Ws13^T                 (tcgen05 GEMM)
//  10 SituGLU           As = SituGLU(Gs)
//  11 shared GEMM2      Sh = As Ws2^T                 (tcgen05 GEMM)
//  12 up-projection     out = N W_up^T + Sh           (tcgen05 GEMM, Sh added
//                                                      in the epilogue)
// Two regimes.  Small T (<= 128 tokens, decode): every GEMM puts the weight
// rows on the MMA's M side and the tokens on N (16..128), dense GEMMs split K
// so that all SMs stream weights, and the split partials are summed in a fixed
// order by the consumer (the scatter of step 4, fused with the permutation of
// step 3, the SituGLU of step 10, and the final reduction that also adds Sh).
// Large T (prefill): tokens on M, 128 x (128|256) tiles (CTA pairs sharing
// operand tiles), no split, bf16 stored straight from the epilogue.
#include <math.h>
#include <string.h>

#include <atomic>
#include <initializer_list>
#include <memory>
#include <mutex>
#include <vector>

#include "gemm_tc.cuh"
#include "lmoe_internal.cuh"
#include "moe_data.cuh"
#include "mxfp4.cuh"

namespace lmoe {

int num_sms() {
  static std::atomic<int> cache[64];   // 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kNumSmsDefault;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kNumSmsDefault;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

constexpr int kDecodeMaxT = 128;
// MXFP4 experts: an expert with more than this many tokens (more than two
// 8-token passes of the 4-bit kernels, which run in one block per column
// strip and re-read its codes) is widened to bf16 into a compact workspace
// copy and runs on the tensor-core GEMMs instead; the others stay on the
// 4-bit kernels.  The split is made on the device from the permutation's
// counts.  (Measured on the 896-expert layer: 16 against 32 and 64 tokens,
// with skewed and with spread-out routing.)
constexpr int kFp4HeavyTokens = 16;
// ... when at least this many experts are that heavy (a few heavy experts give
// the GEMMs too few units to hide their latency: then all stay on the 4-bit
// kernels)
constexpr int kFp4MinHeavy = 4;
constexpr int kMaxSplits = 32;

bool finite_pos(float x) { return isfinite(x) && x > 0.0f; }

int round_up(int x, int m) { return (x + m - 1) / m * m; }

struct DenseCfg {
  int tok_on_m, bn, splits;
};

// Split count minimising the modelled makespan in K blocks (one unit of
// per-tile overhead), for `tiles` output tiles of `nkb` K blocks each.
int choose_splits(int tiles, int nkb, int nsm) {
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= kMaxSplits && s <= nkb; ++s) {
    const long long waves = ((long long)tiles * s + nsm - 1) / nsm;
    const long long cost = waves * ((nkb + s - 1) / s + 1);
    if (best_cost < 0 || cost < best_cost) { best = s; best_cost = cost; }
  }
  return best;
}

DenseCfg dense_cfg(int T, int M_feat, int K, int nsm) {
  DenseCfg c;
  if (T <= kDecodeMaxT) {
    c.tok_on_m = 0;
    c.bn = round_up(T, 16);
    const int tiles = M_feat / 128;
    c.splits = choose_splits(tiles, K / 64, nsm);
  } else {
    c.tok_on_m = 1;
    c.bn = (M_feat % 256 == 0) ? 256 : 128;
    c.splits = 1;
  }
  return c;
}

// Workspace carving (256-byte aligned pieces).
struct Carver {
  size_t off = 0;
  char* base = nullptr;
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

struct Ws {
  int32_t* ids; float* w;
  int32_t* counts; int32_t* offsets; int32_t* tile_prefix; int32_t* row_of; int32_t* tok_of_row;
  void* perm_scratch;
  uint16_t *Z, *A, *G, *act, *Y, *N, *Gs, *As, *Sh;
  float *logits;   // router logits [T, round_up(E, 128)] of the router-GEMM forward
  float *Pa, *Pb;
  int32_t* active;          // active experts in expert order (decode permutation)
  uint16_t *Wd13, *Wd2;     // MXFP4 experts dequantized to bf16 (MXFP4 forward: every
                            // expert at T > 128, the heavy slots at decode sizes)
  // MXFP4 forward at decode sizes with heavy slots: the light experts' list
  // and count, the heavy slots' group tables
  int32_t *light, *n_light, *h_expert, *h_count, *h_offset, *h_prefix;
};

// Heavy-expert slots of the MXFP4 forward: an upper bound on the experts with
// more than kFp4HeavyTokens of the T*k (token, slot) pairs (0 when no expert
// can have that many, or GEMM1 cannot fuse SituGLU).
int fp4_heavy_slots(const lmoe_dims& d) {
  if (d.T <= kFp4HeavyTokens || d.inter % 128) return 0;
  const long long h = (long long)d.T * d.topk / (kFp4HeavyTokens + 1);
  return (int)(h < d.num_experts ? h : d.num_experts);
}

// The MXFP4 forward runs the 4-bit expert kernels for its light experts: at
// decode sizes, and above them wherever the heavy experts can be split off
// (GEMM1 fuses SituGLU); otherwise (inter % 128 != 0 above decode sizes) it
// widens every expert with tokens to bf16 and runs the tensor-core GEMMs
// (measured on the 896-expert layer, the split path is the faster one at
// every T from 17 to 4096, with and without skewed routing).
bool fp4_direct(const lmoe_dims& d) {
  return d.T <= kDecodeMaxT || fp4_heavy_slots(d) > 0;
}

// Router logits rows are padded to whole 128-row weight tiles of the router GEMM.
size_t padded_experts(int E) { return (size_t)round_up(E, 128); }

size_t carve(const lmoe_dims& d, char* base, Ws* ws, bool mxfp4 = false) {
  Carver c;
  c.base = base;
  const size_t T = d.T, k = d.topk, E = d.num_experts, L = d.latent, H = d.hidden;
  const size_t dI = d.inter, ds = d.shared_inter > 0 ? d.shared_inter : 0;
  Ws w{};
  w.ids = c.take<int32_t>(T * k);
  w.w = c.take<float>(T * k);
  w.counts = c.take<int32_t>(E);
  w.offsets = c.take<int32_t>(E + 1);
  w.tile_prefix = c.take<int32_t>(E + 1);
  w.row_of = c.take<int32_t>(T * k);
  w.tok_of_row = c.take<int32_t>(T * k);
  w.perm_scratch = c.take<char>(permute_scratch_bytes(d.T, d.num_experts));
  w.Z = c.take<uint16_t>(T * L);
  w.A = c.take<uint16_t>(T * k * L);
  w.G = c.take<uint16_t>(T * k * 2 * dI);
  w.act = c.take<uint16_t>(T * k * dI);
  w.Y = c.take<uint16_t>(T * k * L);
  w.N = c.take<uint16_t>(T * L);
  w.Gs = c.take<uint16_t>(T * 2 * ds);
  w.As = c.take<uint16_t>(T * ds);
  w.Sh = c.take<uint16_t>(T * H);
  const size_t Ep = padded_experts(d.num_experts);
  w.logits = c.take<float>(T * Ep);
  if (d.T <= kDecodeMaxT) {
    // split-K partials: the down-projection (with the router rows after the
    // latent ones in the router-GEMM forward) and the up-projection
    const size_t ma = (L + Ep > H) ? L + Ep : H;
    const size_t mb = (2 * ds > H) ? 2 * ds : H;
    w.Pa = c.take<float>((size_t)kMaxSplits * T * ma);
    w.Pb = c.take<float>((size_t)kMaxSplits * T * mb);
  } else {
    w.Pa = w.Pb = nullptr;
  }
  w.active = c.take<int32_t>(E);
  w.light = w.n_light = w.h_expert = w.h_count = w.h_offset = w.h_prefix = nullptr;
  const size_t Hs = mxfp4 ? (size_t)fp4_heavy_slots(d) : 0;
  if (mxfp4 && !fp4_direct(d)) {
    w.Wd13 = c.take<uint16_t>(E * 2 * dI * L);
    w.Wd2 = c.take<uint16_t>(E * L * dI);
  } else if (Hs > 0) {
    w.Wd13 = c.take<uint16_t>(Hs * 2 * dI * L);
    w.Wd2 = c.take<uint16_t>(Hs * L * dI);
    w.light = c.take<int32_t>(E);
    w.n_light = c.take<int32_t>(1);
    w.h_expert = c.take<int32_t>(Hs);
    w.h_count = c.take<int32_t>(Hs);
    w.h_offset = c.take<int32_t>(Hs);
    w.h_prefix = c.take<int32_t>(Hs + 1);
  } else {
    w.Wd13 = w.Wd2 = nullptr;
  }
  if (ws) *ws = w;
  return (c.off + 255) & ~size_t(255);
}

int validate_dims(const lmoe_dims* d) {
  if (!d) return LMOE_ERR_NULL;
  if (d->T < 0) return LMOE_ERR_DIM;
  if (d->n_group != 1 || d->topk_group != 1) return LMOE_ERR_UNSUPPORTED;
  if (d->num_experts < 1 || d->num_experts > 1024) return LMOE_ERR_DIM;
  if (d->topk < 1 || d->topk > d->num_experts || d->topk > 32) return LMOE_ERR_DIM;
  if (d->hidden <= 0 || d->hidden % 128 || d->latent <= 0 || d->latent % 128 ||
      d->latent > 8192 || d->inter <= 0 || d->inter % 64)
    return LMOE_ERR_DIM;
  if (d->shared_inter < 0 || d->shared_inter % 64) return LMOE_ERR_DIM;
  if (!finite_pos(d->beta)) return LMOE_ERR_BETA;
  if (!isfinite(d->linear_beta) || !isfinite(d->routed_scaling_factor) || !isfinite(d->rms_eps) ||
      d->rms_eps < 0.0f)
    return LMOE_ERR_DIM;
  // expert-major rows are indexed with 32-bit integers, elements with 64-bit
  if ((long long)d->T * d->topk > (1ll << 30) ||
      (long long)d->T * d->topk * (long long)(2 * d->inter > d->latent ? 2 * d->inter : d->latent) >
          (1ll << 40))
    return LMOE_ERR_DIM;
  return LMOE_OK;
}

cudaError_t gemm_dense(const uint16_t* W, int M_feat, const uint16_t* X, int T, int K,
                       const DenseCfg& c, void* out, int out_fp32, long long split_stride,
                       const uint16_t* add, cudaStream_t s, int fuse_situ = 0, float beta = 1.0f,
                       float linear_beta = 0.0f, long long w_rows = 0,
                       const uint16_t* W2 = nullptr, long long w2_rows = 0, int w2_row0 = 0) {
  GemmDesc g{};
  g.W = W;
  g.w_rows = w_rows;
  g.W2 = W2;
  g.w2_rows = w2_rows;
  g.w2_row0 = w2_row0;
  g.X = X;
  g.x_rows = T;
  g.K = K;
  g.M_feat = M_feat;
  g.G = 1;
  g.T_dense = T;
  g.tok_on_m = c.tok_on_m;
  g.bn = c.bn;
  g.splits = c.splits;
  g.out = out;
  g.ldo = fuse_situ ? M_feat / 2 : M_feat;
  g.out_fp32 = out_fp32;
  g.split_stride = split_stride;
  g.add = add;
  g.fuse_situ = fuse_situ;
  g.beta = beta;
  g.linear_beta = linear_beta;
  const int tok_tile = c.tok_on_m ? 128 : c.bn;
  const int feat_tile = c.tok_on_m ? c.bn : 128;
  g.max_units = ((T + tok_tile - 1) / tok_tile) * (M_feat / feat_tile) * c.splits;
  return launch_gemm(g, s);
}

cudaError_t gemm_grouped(const uint16_t* W, int E, int M_feat, const uint16_t* X, long long rows,
                         int K, int tok_on_m, int bn, const Ws& ws, int tile, void* out,
                         cudaStream_t s, int fuse_situ = 0, float beta = 1.0f,
                         float linear_beta = 0.0f) {
  GemmDesc g{};
  g.W = W;
  g.X = X;
  g.x_rows = rows;
  g.K = K;
  g.M_feat = M_feat;
  g.G = E;
  g.grp_count = ws.counts;
  g.grp_offset = ws.offsets;
  g.tile_prefix = ws.tile_prefix;
  g.tok_on_m = tok_on_m;
  g.bn = bn;
  g.splits = 1;
  g.out = out;
  g.ldo = fuse_situ ? M_feat / 2 : M_feat;
  g.fuse_situ = fuse_situ;
  g.beta = beta;
  g.linear_beta = linear_beta;
  const int feat_tile = fuse_situ ? 256 : (tok_on_m ? bn : 128);
  const long long nonempty = rows < E ? rows : E;
  g.max_units = (int)(((rows + tile - 1) / tile + nonempty) * (M_feat / feat_tile));
  return launch_gemm(g, s);
}

struct Plan {
  int T;
  bool decode;
  bool router;       // the forward computes its router logits (router GEMM)
  int Ep;            // experts padded to whole 128-row router tiles
  bool fuse_g1;      // GEMM1 with SituGLU in its epilogue (inter % 128 == 0)
  bool fuse_s1;      // shared GEMM1 likewise (tokens on M, no split-K, shared_inter % 128 == 0)
  int tile;          // token tile of the grouped GEMMs
  int g1_bn, g2_bn;  // MMA N of the grouped GEMMs
  bool fp4_direct;   // the MXFP4 forward runs the 4-bit expert kernels
  int fp4_heavy;     // heavy-expert slots of the MXFP4 forward
  DenseCfg down, s1, s2, up;
  DenseCfg rtr;      // the router GEMM: at decode stacked after the down-projection's rows
                     // (one launch), otherwise its own launch
};

Plan make_plan(const lmoe_dims& d, int nsm, bool router = false) {
  Plan p;
  p.T = d.T;
  p.decode = d.T <= kDecodeMaxT;
  p.router = router;
  p.Ep = (int)padded_experts(d.num_experts);
  p.tile = p.decode ? round_up(d.T, 16) : 128;
  p.fp4_direct = fp4_direct(d);
  p.fp4_heavy = fp4_heavy_slots(d);
  p.g1_bn = p.decode ? p.tile : ((2 * d.inter) % 256 == 0 ? 256 : 128);
  // tokens on M: a 256-row B operand of 128 gate + 128 up rows; weights on M
  // (decode): the two halves as two MMAs of N = tile tokens
  p.fuse_g1 = d.inter % 128 == 0;
  if (p.fuse_g1 && !p.decode) p.g1_bn = 256;
  p.g2_bn = p.decode ? p.tile : (d.latent % 256 == 0 ? 256 : 128);
  p.down = dense_cfg(d.T, router && p.decode ? d.latent + p.Ep : d.latent, d.hidden, nsm);
  p.rtr = dense_cfg(d.T, p.Ep, d.hidden, nsm);
  p.s1 = dense_cfg(d.T, 2 * d.shared_inter, d.hidden, nsm);
  p.fuse_s1 = p.s1.tok_on_m && p.s1.splits == 1 && p.s1.bn == 256 && d.shared_inter % 128 == 0;
  p.s2 = dense_cfg(d.T, d.hidden, d.shared_inter, nsm);
  p.up = dense_cfg(d.T, d.hidden, d.latent, nsm);
  return p;
}

int plan_launches(const Plan& p, bool shared, bool mxfp4 = false) {
  // one permutation kernel for T <= 256; at decode sizes it also does the scatter
  const int perm = p.T <= 256 ? 1 : 3;
  // GEMM1 (+ SituGLU unless fused), GEMM2; MXFP4 experts: one kernel per
  // stage on the 4-bit weights, with heavy slots also the heavy experts'
  // dequantization, GEMM1 + SituGLU and GEMM2 (split off in the permutation);
  // without the 4-bit kernels, one dequantization kernel first
  int experts = p.fuse_g1 ? 2 : 3;
  if (mxfp4) experts = p.fp4_direct ? 2 + (p.fp4_heavy > 0 ? 3 : 0) : experts + 1;
  // route, down, permute, scatter (fused into the permutation at decode sizes),
  // experts, combine
  int n = 1 + 1 + perm + (p.decode ? 0 : 1) + experts + 1;
  if (shared) n += p.fuse_s1 ? 2 : 3;   // shared GEMM1 (+ SituGLU unless fused), shared GEMM2
  n += 1;                               // up-projection GEMM
  const bool sh_part = shared && p.s2.splits > 1;
  if (p.up.splits > 1 || sh_part) n += 1;   // fixed-order reduction
  // router GEMM: at decode it shares the down-projection's launch and a
  // kernel sums its split-K partials; otherwise it is a launch of its own
  if (p.router) n += 1;
  return n;
}

// The second stream of the forward: the shared expert runs there (and at
// large T the routing and the permutation), forked from and joined back to the
// caller's stream by events, so that a stream capture records the fork too.
// There is one per (device, caller stream): calls on different caller streams
// never share a second stream, so neither one's work is ordered behind the
// other's, and a capture on one caller stream pulls in only its own second
// stream.  An entry is created by the first call on that caller stream made
// (also inside a stream capture) and kept for the life of the process (a stream
// handle that is destroyed and reused maps to the same entry, which stays
// valid: the library owns it).  A call whose device already has
// kMaxAuxPerDevice entries, or that cannot create one, runs every stage on
// the caller's stream instead (same kernels, same results).
// The entry's mutex keeps the event pair of one call from interleaving with
// another host thread's call on the same caller stream.
struct AuxStream {
  int dev = -1;
  cudaStream_t caller = nullptr;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, routed = nullptr;
  std::mutex mu;
};
constexpr int kMaxAuxPerDevice = 64;
std::mutex g_aux_map_mu;
std::vector<std::unique_ptr<AuxStream>> g_aux_map;

// The second stream of `caller` on the current device, created on first use;
// nullptr when the forward must run on the caller's stream alone.
AuxStream* aux_for(cudaStream_t caller) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_aux_map_mu);
  int on_dev = 0;
  for (auto& a : g_aux_map) {
    if (a->dev != dev) continue;
    if (a->caller == caller) return a.get();
    ++on_dev;
  }
  if (on_dev >= kMaxAuxPerDevice) return nullptr;
  // (creating a stream and events is allowed while `caller` is capturing: they
  // are not stream work, and the fork event pulls the new stream into the
  // capture)
  auto a = std::make_unique<AuxStream>();
  a->dev = dev;
  a->caller = caller;
  if (cudaStreamCreateWithFlags(&a->stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&a->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a->join, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a->routed, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;   // (a partially created entry is not kept; its handles leak)
  }
  g_aux_map.push_back(std::move(a));
  return g_aux_map.back().get();
}

// Every non-NULL pointer addresses device memory of the current device
// (cudaMemoryTypeDevice, owned by this device).  A failed query (no device, a
// pointer the runtime does not know) counts as a refusal; its error is cleared
// so that it cannot surface from a later cudaGetLastError.
bool on_current_device(std::initializer_list<const void*> ptrs) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  for (const void* p : ptrs) {
    if (p == nullptr) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return false;
  }
  return true;
}

#define LMOE_TRY(x)                                  \
  do {                                               \
    if ((x) != cudaSuccess) return LMOE_ERR_CUDA;    \
  } while (0)

}  // namespace
}  // namespace lmoe

using namespace lmoe;

extern "C" {

int lmoe_abi_version(void) { return 103; }

const char* lmoe_status_string(int status) {
  switch (status) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_NULL: return "a required pointer is NULL";
    case LMOE_ERR_DIM: return "a size is out of range or not a supported multiple";
    case LMOE_ERR_UNSUPPORTED: return "unsupported routing mode (n_group/topk_group must be 1)";
    case LMOE_ERR_BETA: return "SituGLU beta must be finite and > 0";
    case LMOE_ERR_WORKSPACE: return "workspace is NULL, misaligned or too small";
    case LMOE_ERR_CUDA: return "a CUDA call failed";
    case LMOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case LMOE_ERR_DEVICE: return "a pointer is not device memory of the current device";
    default: return "unknown status";
  }
}

int lmoe_device_error(int clear) { return read_device_error(clear); }

int moe_route(const float* router_logits, const float* bias, int T, int E, int topk, int n_group,
              int topk_group, int renormalize, float rsf, int32_t* topk_ids, float* topk_weights,
              void* stream) {
  if (n_group != 1 || topk_group != 1) return LMOE_ERR_UNSUPPORTED;
  if (T < 0 || E < 1 || E > 1024 || topk < 1 || topk > E || topk > 32) return LMOE_ERR_DIM;
  if (!isfinite(rsf)) return LMOE_ERR_DIM;
  if (T == 0) return LMOE_OK;
  if (!router_logits || !topk_ids || !topk_weights) return LMOE_ERR_NULL;
  if (!aligned16(router_logits) || !aligned16(topk_ids) || !aligned16(topk_weights) ||
      (bias && !aligned16(bias)))
    return LMOE_ERR_ALIGN;
  if (!on_current_device({router_logits, bias, topk_ids, topk_weights})) return LMOE_ERR_DEVICE;
  if (launch_route(router_logits, E, bias, T, E, topk, renormalize, rsf, topk_ids, topk_weights,
                   (cudaStream_t)stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

int situ_and_mul(const lmoe_bf16* in, lmoe_bf16* out, int64_t N, int d, float beta,
                 float linear_beta, void* stream) {
  if (!finite_pos(beta)) return LMOE_ERR_BETA;
  if (N < 0 || d <= 0 || d % 8 || !isfinite(linear_beta)) return LMOE_ERR_DIM;
  if (N == 0) return LMOE_OK;
  if (!in || !out) return LMOE_ERR_NULL;
  if (!aligned16(in) || !aligned16(out)) return LMOE_ERR_ALIGN;
  if (!on_current_device({in, out})) return LMOE_ERR_DEVICE;
  if (launch_situ(in, out, N, d, beta, linear_beta, (cudaStream_t)stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

int masked_situ_and_mul(const lmoe_bf16* in, lmoe_bf16* out, const int32_t* expert_num_tokens,
                        int E, int T_max, int d, float beta, float linear_beta, void* stream) {
  if (!finite_pos(beta)) return LMOE_ERR_BETA;
  if (E < 0 || E > 65535 || T_max < 0 || d <= 0 || d % 8 || !isfinite(linear_beta))
    return LMOE_ERR_DIM;
  if (E == 0 || T_max == 0) return LMOE_OK;
  if (!in || !out || !expert_num_tokens) return LMOE_ERR_NULL;
  if (!aligned16(in) || !aligned16(out) || !aligned16(expert_num_tokens)) return LMOE_ERR_ALIGN;
  if (!on_current_device({in, out, expert_num_tokens})) return LMOE_ERR_DEVICE;
  if (launch_masked_situ(in, out, expert_num_tokens, E, T_max, d, beta, linear_beta,
                         (cudaStream_t)stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

int lmoe_linear(const lmoe_bf16* x, const lmoe_bf16* w, const lmoe_bf16* add, lmoe_bf16* out,
                int T, int N, int K, void* stream) {
  if (T < 0 || N <= 0 || N % 128 || K <= 0 || K % 64) return LMOE_ERR_DIM;
  if (T == 0) return LMOE_OK;
  if (!x || !w || !out) return LMOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (add && !aligned16(add)))
    return LMOE_ERR_ALIGN;
  if (!on_current_device({x, w, add, out})) return LMOE_ERR_DEVICE;
  DenseCfg c = dense_cfg(T, N, K, num_sms());
  c.splits = 1;
  if (gemm_dense(w, N, x, T, K, c, out, 0, 0, add, (cudaStream_t)stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

int latent_moe_workspace_offsets(const lmoe_dims* dims, size_t* offsets) {
  const int v = validate_dims(dims);
  if (v != LMOE_OK) return v;
  if (!offsets) return LMOE_ERR_NULL;
  Ws w;
  char* const base = reinterpret_cast<char*>(256);   // never dereferenced
  carve(*dims, base, &w);
  const void* p[LMOE_WS_COUNT] = {w.ids, w.w, w.counts, w.offsets, w.row_of, w.Z, w.A,
                                  w.G, w.act, w.Y, w.N, w.Gs, w.As, w.Sh, w.logits};
  for (int i = 0; i < LMOE_WS_COUNT; ++i)
    offsets[i] = (size_t)(reinterpret_cast<const char*>(p[i]) - base);
  return LMOE_OK;
}

int latent_moe_launch_count(const lmoe_dims* dims, int has_shared_expert) {
  if (validate_dims(dims) != LMOE_OK) return 0;
  if (dims->T == 0) return 0;
  return plan_launches(make_plan(*dims, num_sms()), has_shared_expert != 0);
}

size_t latent_moe_workspace_bytes(const lmoe_dims* dims) {
  if (validate_dims(dims) != LMOE_OK) return 0;
  return carve(*dims, nullptr, nullptr);
}

// The layer forward.  Exactly one of router_logits (the layer routes) and
// pre_ids/pre_w (routing done ahead by the caller) is given.  own_workspace:
// the workspace is the library's own static scratch (known device memory of
// the current device), so its pointer is not queried.
static int forward_impl(const lmoe_dims* dims, const lmoe_weights* wt, const lmoe_bf16* hidden,
                        const float* router_logits, const int32_t* pre_ids, const float* pre_w,
                        const lmoe_bf16* w_router, lmoe_bf16* out, void* workspace,
                        size_t workspace_bytes, const lmoe_debug* dbg, void* stream,
                        bool own_workspace, const lmoe_mxfp4_experts* fq = nullptr) {
  const int v = validate_dims(dims);
  if (v != LMOE_OK) return v;
  if (!wt) return LMOE_ERR_NULL;
  const lmoe_dims d = *dims;
  if (d.T == 0) return LMOE_OK;
  // exactly one routing source: the caller's logits, the router GEMM on
  // w_router, or ids and weights routed ahead
  const bool router = w_router != nullptr;
  const bool pre_routed = !router && router_logits == nullptr;
  if (!hidden || (pre_routed && (!pre_ids || !pre_w)) || !out || !wt->w_down || !wt->w_up)
    return LMOE_ERR_NULL;
  // routed experts: bf16 (w13, w2) or MXFP4 (fq)
  if (fq) {
    if (!fq->w13_codes || !fq->w13_scales || !fq->w2_codes || !fq->w2_scales) return LMOE_ERR_NULL;
    if (d.inter > 4096 || d.latent > 4096) return LMOE_ERR_DIM;
    if (!aligned16(fq->w13_codes) || !aligned16(fq->w2_codes) || !aligned16(fq->w13_scales) ||
        !aligned16(fq->w2_scales))
      return LMOE_ERR_ALIGN;
  } else if (!wt->w13 || !wt->w2) {
    return LMOE_ERR_NULL;
  }
  const bool shared = wt->ws13 != nullptr;
  if (shared != (wt->ws2 != nullptr)) return LMOE_ERR_NULL;
  if (shared && d.shared_inter <= 0) return LMOE_ERR_DIM;
  const void* ptrs[] = {hidden, router_logits, pre_ids, pre_w, out, wt->w_down,
                        fq ? nullptr : wt->w13, fq ? nullptr : wt->w2, wt->w_up, wt->ws13,
                        wt->ws2, wt->norm_w, wt->e_score_correction_bias, w_router};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return LMOE_ERR_ALIGN;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return LMOE_ERR_WORKSPACE;
  Ws ws;
  const size_t need = carve(d, static_cast<char*>(workspace), &ws, fq != nullptr);
  if (workspace_bytes < need) return LMOE_ERR_WORKSPACE;
  if (dbg) {
    const void* dp[] = {dbg->topk_ids, dbg->topk_weights, dbg->expert_num_tokens,
                        dbg->expert_offsets, dbg->row_of};
    for (const void* p : dp)
      if (p && !aligned16(p)) return LMOE_ERR_ALIGN;
  }
  if (!on_current_device({hidden, router_logits, pre_ids, pre_w, out, wt->w_down,
                          fq ? nullptr : wt->w13, fq ? nullptr : wt->w2, wt->w_up, wt->ws13,
                          wt->ws2, wt->norm_w, wt->e_score_correction_bias, w_router,
                          own_workspace ? nullptr : workspace}))
    return LMOE_ERR_DEVICE;
  if (fq && !on_current_device({fq->w13_codes, fq->w13_scales, fq->w2_codes, fq->w2_scales}))
    return LMOE_ERR_DEVICE;
  if (dbg && !on_current_device({dbg->topk_ids, dbg->topk_weights, dbg->expert_num_tokens,
                                 dbg->expert_offsets, dbg->row_of}))
    return LMOE_ERR_DEVICE;

  cudaStream_t s = (cudaStream_t)stream;
  const int T = d.T, k = d.topk, E = d.num_experts, H = d.hidden, L = d.latent;
  // the routing result: the layer's own, or the caller's (whose ids the
  // permutation checks against [0, E), recording kErrExpertId)
  const int32_t* ids = pre_routed ? pre_ids : ws.ids;
  const float* topw = pre_routed ? pre_w : ws.w;
  int* id_err = pre_routed ? device_error_word() : nullptr;
  if (pre_routed && !id_err) return LMOE_ERR_CUDA;
  const int dI = d.inter, ds = d.shared_inter;
  const long long rows = (long long)T * k;
  const Plan pl = make_plan(d, num_sms(), router);
  const int Ep = pl.Ep;
  const bool decode = pl.decode;
  const int tile = pl.tile;
  const uint16_t* X = hidden;
  void** ev = dbg ? dbg->stage_events : nullptr;
  auto mark = [&](int i) -> bool {
    return ev == nullptr || cudaEventRecord((cudaEvent_t)ev[i], s) == cudaSuccess;
  };
  if (!mark(0)) return LMOE_ERR_CUDA;
  // the shared expert gets the second stream, where it fills the gaps the
  // routed path's latency-bound stages leave (not when per-stage timing was
  // asked for, which needs the stages one after another)
  AuxStream* aux = (shared && ev == nullptr) ? aux_for(s) : nullptr;
  const bool concurrent = aux != nullptr;
  std::unique_lock<std::mutex> aux_lock;
  if (concurrent) {
    aux_lock = std::unique_lock<std::mutex>(aux->mu);
    if (cudaEventRecord(aux->fork, s) != cudaSuccess) return LMOE_ERR_CUDA;
  }
  // 9-11. shared expert on the original hidden states (enqueued by a lambda:
  // on the caller's stream, or on the second stream so that it overlaps the
  // routed path)
  const float* sh_part = nullptr;
  int sh_splits = 0;
  long long sh_stride = 0;
  const uint16_t* sh_bf16 = nullptr;
  auto shared_expert = [&](cudaStream_t ss, bool marks) -> int {
    if (shared) {
      const DenseCfg c1 = pl.s1;
      const long long s1_stride = (long long)T * 2 * ds;
      if (c1.splits > 1) {
        LMOE_TRY(gemm_dense(wt->ws13, 2 * ds, X, T, H, c1, ws.Pb, 1, s1_stride, nullptr, ss));
        LMOE_TRY(launch_reduce_situ(ws.Pb, c1.splits, s1_stride, T, ds, d.beta, d.linear_beta,
                                    ws.As, ss));
      } else if (pl.fuse_s1) {
        // As = bf16(SituGLU(bf16(X Ws13^T))) straight from the GEMM epilogue
        LMOE_TRY(gemm_dense(wt->ws13, 2 * ds, X, T, H, c1, ws.As, 0, 0, nullptr, ss, 1, d.beta,
                            d.linear_beta));
      } else {
        LMOE_TRY(gemm_dense(wt->ws13, 2 * ds, X, T, H, c1, ws.Gs, 0, 0, nullptr, ss));
        LMOE_TRY(launch_situ(ws.Gs, ws.As, T, ds, d.beta, d.linear_beta, ss));
      }
    }
    if (marks && !mark(LMOE_STAGE_SHARED1 + 1)) return LMOE_ERR_CUDA;
    if (shared) {
      const DenseCfg c2 = pl.s2;
      sh_stride = (long long)T * H;
      if (c2.splits > 1) {
        LMOE_TRY(gemm_dense(wt->ws2, H, ws.As, T, ds, c2, ws.Pb, 1, sh_stride, nullptr, ss));
        sh_part = ws.Pb;
        sh_splits = c2.splits;
      } else {
        LMOE_TRY(gemm_dense(wt->ws2, H, ws.As, T, ds, c2, ws.Sh, 0, 0, nullptr, ss));
        sh_bf16 = ws.Sh;
      }
    }
    if (marks && !mark(LMOE_STAGE_SHARED2 + 1)) return LMOE_ERR_CUDA;
    return LMOE_OK;
  };
  // 1. routing and 3. permutation: at large T they run first on the second
  // stream, beside the down-projection (which leaves SMs idle in its last
  // wave), and the caller's stream waits for them before the scatter (at
  // decode sizes this measured slower: they stay on the caller's stream)
  // the logits the routing reads: the caller's [T, E], or the router GEMM's
  // [T, Ep] in the workspace
  const float* lg = router ? ws.logits : router_logits;
  const long long lg_ld = router ? Ep : E;
  auto route_and_permute = [&](cudaStream_t rs, bool marks) -> int {
    if (router && !decode) {
      // router GEMM of its own (fp32 logits straight from the epilogue)
      DenseCfg cr = pl.rtr;
      LMOE_TRY(gemm_dense(w_router, Ep, X, T, H, cr, ws.logits, 1, 0, nullptr, rs, 0, 1.0f, 0.0f,
                          E));
    }
    if (!pre_routed)
      LMOE_TRY(launch_route(lg, lg_ld, wt->e_score_correction_bias, T, E, k, d.renormalize,
                            d.routed_scaling_factor, ws.ids, ws.w, rs));
    if (marks && !mark(LMOE_STAGE_ROUTE + 1)) return LMOE_ERR_CUDA;
    return LMOE_OK;
  };
  // MXFP4 experts with heavy slots: the permutation also splits the experts
  // by count (heavy ones in token tiles of the grouped GEMMs)
  const bool fp4_split = fq && pl.fp4_direct && pl.fp4_heavy > 0;
  const HeavySplit hsplit{kFp4HeavyTokens + 1, kFp4MinHeavy, pl.fp4_heavy, tile, ws.light,
                          ws.n_light, ws.h_expert, ws.h_count, ws.h_offset, ws.h_prefix};
  auto permute = [&](cudaStream_t rs) -> int {
    LMOE_TRY(launch_permute(ids, T, k, E, tile, ws.perm_scratch, ws.counts, ws.offsets,
                            ws.tile_prefix, ws.row_of, ws.tok_of_row, id_err, rs,
                            fp4_split ? &hsplit : nullptr));
    return LMOE_OK;
  };
  int st = LMOE_OK;
  const bool side_route = concurrent && !decode;
  // At decode sizes the shared expert forks off late.  With bf16 experts after
  // the routed GEMM1: from the start it held SMs that GEMM1's persistent CTAs
  // then reached late (its CTAs finished up to 26 us apart); after GEMM1 it
  // runs beside GEMM2, the combine and the up-projection (182.5-182.8 against
  // 186.9 us per decode step).  With MXFP4 experts after the scatter, ahead of
  // the expert kernels (151.7 against 154.7 us in graph replays after an L2
  // flush; after GEMM1 it was slower: their blocks take an SM's shared memory,
  // so nothing of the shared expert runs beside them).
  const bool late_shared = concurrent && decode;
  auto fork_shared_late = [&]() -> int {
    if (!late_shared) return LMOE_OK;
    if (cudaEventRecord(aux->fork, s) != cudaSuccess) return LMOE_ERR_CUDA;
    if (cudaStreamWaitEvent(aux->stream, aux->fork, 0) != cudaSuccess) return LMOE_ERR_CUDA;
    const int r = shared_expert(aux->stream, false);
    if (r != LMOE_OK) return r;
    if (cudaEventRecord(aux->join, aux->stream) != cudaSuccess) return LMOE_ERR_CUDA;
    return LMOE_OK;
  };
  if (concurrent && !late_shared) {
    if (cudaStreamWaitEvent(aux->stream, aux->fork, 0) != cudaSuccess) return LMOE_ERR_CUDA;
    if (side_route) {
      st = route_and_permute(aux->stream, false);
      if (st != LMOE_OK) return st;
      st = permute(aux->stream);
      if (st != LMOE_OK) return st;
      if (cudaEventRecord(aux->routed, aux->stream) != cudaSuccess) return LMOE_ERR_CUDA;
    }
    st = shared_expert(aux->stream, false);
    if (st != LMOE_OK) return st;
    if (cudaEventRecord(aux->join, aux->stream) != cudaSuccess) return LMOE_ERR_CUDA;
  }
  // 2. latent down-projection.  Router GEMM at decode sizes: the router rows
  // follow the latent rows in one split-K launch over the hidden states
  // (fp32 partials [splits][T][L + Ep]), a kernel sums the logit columns and
  // the routing reads them; the per-stage events then show the router GEMM,
  // the sum and the routing as the routing stage and the down-projection as
  // an empty stage.
  const bool stacked = router && decode;
  const DenseCfg cdown = pl.down;
  const bool down_split = cdown.splits > 1 || stacked;
  const int ldz = stacked ? L + Ep : L;
  const long long down_stride = (long long)T * ldz;
  if (!side_route && !stacked) {
    st = route_and_permute(s, true);
    if (st != LMOE_OK) return st;
  }
  if (stacked) {
    LMOE_TRY(gemm_dense(wt->w_down, L + Ep, X, T, H, cdown, ws.Pa, 1, down_stride, nullptr, s, 0,
                        1.0f, 0.0f, 0, w_router, E, L));
    LMOE_TRY(launch_sum_splits_cols(ws.Pa, cdown.splits, down_stride, T, ldz, L, E, Ep, ws.logits,
                                    s));
    st = route_and_permute(s, true);
    if (st != LMOE_OK) return st;
  } else {
    LMOE_TRY(gemm_dense(wt->w_down, L, X, T, H, cdown, down_split ? (void*)ws.Pa : (void*)ws.Z,
                        down_split, down_stride, nullptr, s));
  }
  if (!mark(LMOE_STAGE_DOWN + 1)) return LMOE_ERR_CUDA;
  // small T: permutation and scatter in one launch (every block rebuilds the
  // small counting sort); large T: the scatter after the separate permutation
  const bool fused_scatter = decode;
  if (side_route) {
    if (cudaStreamWaitEvent(s, aux->routed, 0) != cudaSuccess) return LMOE_ERR_CUDA;
  } else if (fused_scatter) {
    LMOE_TRY(launch_permute_scatter_small(ids, T, k, E, tile, ws.counts, ws.offsets,
                                          ws.tile_prefix, ws.row_of, ws.tok_of_row,
                                          down_split ? nullptr : ws.Z,
                                          down_split ? ws.Pa : nullptr, cdown.splits, down_stride,
                                          ldz, L, ws.A, ws.active, id_err, s,
                                          fp4_split ? &hsplit : nullptr));
  } else {
    st = permute(s);
    if (st != LMOE_OK) return st;
  }
  if (!mark(LMOE_STAGE_PERMUTE + 1)) return LMOE_ERR_CUDA;
  // 4. routed input into the expert-major rows
  if (!fused_scatter)
    LMOE_TRY(launch_scatter_rows(down_split ? nullptr : ws.Z, down_split ? ws.Pa : nullptr,
                                 cdown.splits, down_stride, ldz, T, L, k, ws.row_of, ws.A, s));
  if (!mark(LMOE_STAGE_SCATTER + 1)) return LMOE_ERR_CUDA;
  if (fq && pl.fp4_direct) {
    st = fork_shared_late();
    if (st != LMOE_OK) return st;
  }
  // 5-7. experts
  const uint16_t* W13 = wt->w13;
  const uint16_t* W2 = wt->w2;
  if (fq && pl.fp4_direct) {
    // MXFP4: GEMM1 + SituGLU and GEMM2 straight from the 4-bit weights, one
    // block per (active expert, column strip).  With heavy
    // slots (T > kFp4HeavyTokens) the permutation has split the active experts
    // by their counts: the light ones stay on the 4-bit kernels, the heavy
    // ones are widened to bf16 into the slots and run on the tensor-core GEMMs
    // (each path writes only its own experts' rows of act and Y)
    const int slots = (long long)E < rows ? E : (int)rows;
    const int H = pl.fp4_heavy;
    int* dev_err = device_error_word();
    if (!dev_err) return LMOE_ERR_CUDA;
    const int32_t* list = ws.active;
    const int32_t* n_list = ws.tile_prefix + E;
    Ws wh = ws;
    if (H > 0) {
      list = ws.light;
      n_list = ws.n_light;
      LMOE_TRY(launch_dequant_mxfp4_pair(fq->w13_codes, fq->w13_scales, ws.Wd13,
                                         (long long)H * 2 * dI, L, fq->w2_codes, fq->w2_scales,
                                         ws.Wd2, (long long)H * L, dI, s, ws.h_count, 2 * dI, L,
                                         ws.h_expert));
      wh.counts = ws.h_count;
      wh.offsets = ws.h_offset;
      wh.tile_prefix = ws.h_prefix;
    }
    LMOE_TRY(launch_fp4_expert_gemv(fq->w13_codes, fq->w13_scales, ws.A, ws.act, ws.counts,
                                    ws.offsets, list, n_list, slots, E, L, dI, 1, d.beta,
                                    d.linear_beta, dev_err, s));
    if (H > 0)
      LMOE_TRY(gemm_grouped(ws.Wd13, H, 2 * dI, ws.A, rows, L, !decode, pl.g1_bn, wh, tile,
                            ws.act, s, 1, d.beta, d.linear_beta));
    if (!mark(LMOE_STAGE_GEMM1 + 1) || !mark(LMOE_STAGE_SITU + 1)) return LMOE_ERR_CUDA;
    LMOE_TRY(launch_fp4_expert_gemv(fq->w2_codes, fq->w2_scales, ws.act, ws.Y, ws.counts,
                                    ws.offsets, list, n_list, slots, E, dI, L, 0, d.beta,
                                    d.linear_beta, dev_err, s));
    if (H > 0)
      LMOE_TRY(gemm_grouped(ws.Wd2, H, L, ws.act, rows, dI, !decode, pl.g2_bn, wh, tile, ws.Y, s));
    if (!mark(LMOE_STAGE_GEMM2 + 1)) return LMOE_ERR_CUDA;
  } else {
    if (fq) {
      // MXFP4 without the 4-bit kernels (inter % 128 != 0 above decode
      // sizes): the weights of every expert with routed
      // tokens dequantized to bf16 in the workspace, then the tensor-core path
      // (the grouped GEMMs read no rows of the others)
      LMOE_TRY(launch_dequant_mxfp4_pair(fq->w13_codes, fq->w13_scales, ws.Wd13,
                                         (long long)E * 2 * dI, L, fq->w2_codes, fq->w2_scales,
                                         ws.Wd2, (long long)E * L, dI, s, ws.counts, 2 * dI, L,
                                         nullptr));
      W13 = ws.Wd13;
      W2 = ws.Wd2;
    }
    if (pl.fuse_g1) {
      // act = bf16(SituGLU(bf16(A W13_e^T))) straight from GEMM1's epilogue
      LMOE_TRY(gemm_grouped(W13, E, 2 * dI, ws.A, rows, L, !decode, pl.g1_bn, ws, tile, ws.act, s,
                            1, d.beta, d.linear_beta));
      if (!mark(LMOE_STAGE_GEMM1 + 1)) return LMOE_ERR_CUDA;
    } else {
      LMOE_TRY(gemm_grouped(W13, E, 2 * dI, ws.A, rows, L, !decode, pl.g1_bn, ws, tile, ws.G, s));
      if (!mark(LMOE_STAGE_GEMM1 + 1)) return LMOE_ERR_CUDA;
      LMOE_TRY(launch_situ(ws.G, ws.act, rows, dI, d.beta, d.linear_beta, s));
    }
    if (!mark(LMOE_STAGE_SITU + 1)) return LMOE_ERR_CUDA;
    st = fork_shared_late();
    if (st != LMOE_OK) return st;
    LMOE_TRY(gemm_grouped(W2, E, L, ws.act, rows, dI, !decode, pl.g2_bn, ws, tile, ws.Y, s));
    if (!mark(LMOE_STAGE_GEMM2 + 1)) return LMOE_ERR_CUDA;
  }
  // 8. combine + RMSNorm
  LMOE_TRY(launch_combine_norm(ws.Y, topw, ws.row_of, T, k, L, wt->norm_w, d.rms_eps, ws.N, s));
  if (!mark(LMOE_STAGE_COMBINE + 1)) return LMOE_ERR_CUDA;
  // 12. up-projection with the shared output added in the epilogue
  const DenseCfg cup = pl.up;
  if (!concurrent) {
    st = shared_expert(s, true);
    if (st != LMOE_OK) return st;
  }
  if (cup.splits > 1) {
    const long long up_stride = (long long)T * H;
    LMOE_TRY(gemm_dense(wt->w_up, H, ws.N, T, L, cup, ws.Pa, 1, up_stride, nullptr, s));
    if (concurrent && cudaStreamWaitEvent(s, aux->join, 0) != cudaSuccess) return LMOE_ERR_CUDA;
    LMOE_TRY(launch_reduce_splits(ws.Pa, cup.splits, up_stride, sh_part, sh_splits, sh_stride,
                                  sh_bf16, (long long)T * H, out, s));
  } else {
    if (concurrent && cudaStreamWaitEvent(s, aux->join, 0) != cudaSuccess) return LMOE_ERR_CUDA;
    if (sh_part) {
      // shared output still in partials: materialise it in bf16 first
      LMOE_TRY(launch_reduce_splits(sh_part, sh_splits, sh_stride, nullptr, 0, 0, nullptr,
                                    (long long)T * H, ws.Sh, s));
      sh_bf16 = ws.Sh;
    }
    LMOE_TRY(gemm_dense(wt->w_up, H, ws.N, T, L, cup, out, 0, 0, sh_bf16, s));
  }
  if (!mark(LMOE_STAGE_UP + 1)) return LMOE_ERR_CUDA;
  // optional copies of the routing and permutation
  if (dbg) {
    if (dbg->topk_ids)
      LMOE_TRY(cudaMemcpyAsync(dbg->topk_ids, ids, rows * 4, cudaMemcpyDeviceToDevice, s));
    if (dbg->topk_weights)
      LMOE_TRY(cudaMemcpyAsync(dbg->topk_weights, topw, rows * 4, cudaMemcpyDeviceToDevice, s));
    if (dbg->expert_num_tokens)
      LMOE_TRY(cudaMemcpyAsync(dbg->expert_num_tokens, ws.counts, (size_t)E * 4,
                               cudaMemcpyDeviceToDevice, s));
    if (dbg->expert_offsets)
      LMOE_TRY(cudaMemcpyAsync(dbg->expert_offsets, ws.offsets, (size_t)(E + 1) * 4,
                               cudaMemcpyDeviceToDevice, s));
    if (dbg->row_of)
      LMOE_TRY(cudaMemcpyAsync(dbg->row_of, ws.row_of, rows * 4, cudaMemcpyDeviceToDevice, s));
  }
  return LMOE_OK;
}

int latent_moe_forward(const lmoe_dims* dims, const lmoe_weights* wt, const lmoe_bf16* hidden,
                       const float* router_logits, lmoe_bf16* out, void* workspace,
                       size_t workspace_bytes, const lmoe_debug* dbg, void* stream) {
  return forward_impl(dims, wt, hidden, router_logits, nullptr, nullptr, nullptr, out, workspace,
                      workspace_bytes, dbg, stream, false);
}

int latent_moe_forward_router(const lmoe_dims* dims, const lmoe_weights* wt,
                              const lmoe_bf16* w_router, const lmoe_bf16* hidden, lmoe_bf16* out,
                              void* workspace, size_t workspace_bytes, const lmoe_debug* dbg,
                              void* stream) {
  if (dims && dims->T != 0 && !w_router) return LMOE_ERR_NULL;
  return forward_impl(dims, wt, hidden, nullptr, nullptr, nullptr, w_router, out, workspace,
                      workspace_bytes, dbg, stream, false);
}

int latent_moe_launch_count_router(const lmoe_dims* dims, int has_shared_expert) {
  if (validate_dims(dims) != LMOE_OK) return 0;
  if (dims->T == 0) return 0;
  return plan_launches(make_plan(*dims, num_sms(), true), has_shared_expert != 0);
}

size_t lmoe_router_logits_workspace_bytes(int T, int E, int H) {
  if (T < 0 || E < 1 || E > 1024 || H <= 0 || H % 64) return 0;
  const size_t Ep = padded_experts(E);
  size_t n = 0;
  if (T <= kDecodeMaxT) n = (size_t)kMaxSplits * T * Ep * 4;   // split-K partials
  else if ((size_t)E != Ep) n = (size_t)T * Ep * 4;          // padded rows
  return ((n + 255) & ~size_t(255)) + 256;
}

int lmoe_router_logits(const lmoe_bf16* hidden, const lmoe_bf16* w_router, float* logits, int T,
                       int E, int H, void* workspace, size_t workspace_bytes, void* stream) {
  const size_t need = lmoe_router_logits_workspace_bytes(T, E, H);
  if (need == 0) return LMOE_ERR_DIM;
  if (T == 0) return LMOE_OK;
  if (!hidden || !w_router || !logits) return LMOE_ERR_NULL;
  if (!aligned16(hidden) || !aligned16(w_router) || !aligned16(logits)) return LMOE_ERR_ALIGN;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return LMOE_ERR_WORKSPACE;
  if (!on_current_device({hidden, w_router, logits, workspace})) return LMOE_ERR_DEVICE;
  cudaStream_t s = (cudaStream_t)stream;
  const int Ep = (int)padded_experts(E);
  const DenseCfg c = dense_cfg(T, Ep, H, num_sms());
  float* P = static_cast<float*>(workspace);
  if (!c.tok_on_m) {
    // weights on M, split K: fp32 partials, then their fixed-order sum
    const long long stride = (long long)T * Ep;
    LMOE_TRY(gemm_dense(w_router, Ep, hidden, T, H, c, P, 1, stride, nullptr, s, 0, 1.0f, 0.0f,
                        E));
    LMOE_TRY(launch_sum_splits_cols(P, c.splits, stride, T, Ep, 0, E, E, logits, s));
  } else if (E == Ep) {
    LMOE_TRY(gemm_dense(w_router, Ep, hidden, T, H, c, logits, 1, 0, nullptr, s));
  } else {
    LMOE_TRY(gemm_dense(w_router, Ep, hidden, T, H, c, P, 1, 0, nullptr, s, 0, 1.0f, 0.0f, E));
    LMOE_TRY(launch_sum_splits_cols(P, 1, 0, T, Ep, 0, E, E, logits, s));
  }
  return LMOE_OK;
}

int latent_moe_forward_routed(const lmoe_dims* dims, const lmoe_weights* wt,
                              const lmoe_bf16* hidden, const int32_t* topk_ids,
                              const float* topk_weights, lmoe_bf16* out, void* workspace,
                              size_t workspace_bytes, const lmoe_debug* dbg, void* stream) {
  return forward_impl(dims, wt, hidden, nullptr, topk_ids, topk_weights, nullptr, out, workspace,
                      workspace_bytes, dbg, stream, false);
}

int lmoe_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, lmoe_bf16* out, int64_t rows,
                       int K, void* stream) {
  if (rows < 0 || K <= 0 || K % 32) return LMOE_ERR_DIM;
  if (rows == 0) return LMOE_OK;
  if (!codes || !scales || !out) return LMOE_ERR_NULL;
  if (!aligned16(codes) || !aligned16(out)) return LMOE_ERR_ALIGN;
  if (!on_current_device({codes, scales, out})) return LMOE_ERR_DEVICE;
  if (launch_dequant_mxfp4(codes, scales, out, rows, K, (cudaStream_t)stream) != cudaSuccess)
    return LMOE_ERR_CUDA;
  return LMOE_OK;
}

size_t latent_moe_workspace_bytes_mxfp4(const lmoe_dims* dims) {
  if (validate_dims(dims) != LMOE_OK || dims->inter > 4096 || dims->latent > 4096) return 0;
  return carve(*dims, nullptr, nullptr, true);
}

int latent_moe_forward_mxfp4(const lmoe_dims* dims, const lmoe_weights* wt,
                             const lmoe_mxfp4_experts* experts, const lmoe_bf16* hidden,
                             const float* router_logits, lmoe_bf16* out, void* workspace,
                             size_t workspace_bytes, const lmoe_debug* dbg, void* stream) {
  if (dims && dims->T != 0 && (!experts || !router_logits)) return LMOE_ERR_NULL;
  lmoe_mxfp4_experts none{};
  return forward_impl(dims, wt, hidden, router_logits, nullptr, nullptr, nullptr, out, workspace,
                      workspace_bytes, dbg, stream, false, experts ? experts : &none);
}

int latent_moe_launch_count_mxfp4(const lmoe_dims* dims, int has_shared_expert) {
  if (validate_dims(dims) != LMOE_OK || dims->inter > 4096 || dims->latent > 4096) return 0;
  if (dims->T == 0) return 0;
  return plan_launches(make_plan(*dims, num_sms()), has_shared_expert != 0, true);
}

}  // extern "C"

namespace lmoe {
int forward_on_library_scratch(const lmoe_dims* dims, const lmoe_weights* wt,
                               const lmoe_bf16* hidden, const float* router_logits,
                               lmoe_bf16* out, void* scratch, size_t scratch_bytes,
                               const lmoe_debug* dbg, void* stream) {
  return forward_impl(dims, wt, hidden, router_logits, nullptr, nullptr, nullptr, out, scratch,
                      scratch_bytes, dbg, stream, true);
}
}  // namespace lmoe
