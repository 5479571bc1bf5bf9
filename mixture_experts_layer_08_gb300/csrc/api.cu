// C ABI of the MoE block forward: validation, workspace carving, dispatch of the kernel
// chains on the caller's stream. Allocates nothing and never synchronises the host (except
// moe_read_device_status, which exists to do exactly that).
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (`forward_prefill` picks the
// grouped GEMM body above a row threshold and the per-token path below it; named refusals
// instead of silent wrong results), "spark_model/layers/moe/forward_batched.rs" (refuses
// identity-expert routing except on the softmax + correction-bias arm),
// "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (scratch-size check reporting the
// bytes needed and available; the FP32 accumulator sits at a 256-byte aligned offset).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <map>
#include <mutex>

#include "kernels.h"

using namespace moe;

namespace {

constexpr int kSmallRouterMaxTokens = 64;

enum Region {
  // the decode chain's accumulators follow the header so one memset clears them all
  R_HDR, R_SYNC, R_HD, R_YD, R_ACC, R_SHY, R_LOGITS, R_IDX, R_W, R_ZSUM, R_BLK, R_LRANK, R_OFFS,
  R_P2R, R_SPAIRS, R_ACTIVE, R_TILES, R_XQT, R_XST, R_XP, R_XS, R_HH, R_HS, R_Y, R_SHH, R_XN, R_NUM
};

struct Layout {
  size_t off[R_NUM];
  size_t size[R_NUM];
  size_t total;
  int path;
  int te, max_mtiles, nblk;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Weight bytes a forward may stream (every expert the batch can touch, and the shared
// expert), below which the grouped chain's short launches beat the decode kernel's fixed cost
// (its cross-block waits and run-once code: ~50 us for a few MB of weights, against ~36 us).
constexpr double kDecodeMinWeightBytes = 8.0 * (1 << 20);

double touched_weight_bytes(const moe_config_t* c) {
  const double per_weight = c->weight_dtype == MOE_W_BF16            ? 2.0
                            : c->weight_dtype == MOE_W_FP8_E4M3_B128 ? 1.0
                                                                     : 0.5625;
  const int experts = std::min(c->num_experts, c->num_tokens * c->top_k);
  return (double)experts * 3.0 * c->inter * c->hidden * per_weight +
         3.0 * c->shared_inter * c->hidden * 2.0;
}

int resolve_path(const moe_config_t* c) {
  if (c->path != MOE_PATH_AUTO) return c->path;
  const bool decode_ok = c->num_tokens <= kDecodeMaxTokens && c->inter <= 1024 &&
                         c->shared_inter <= 1024 &&
                         (c->weight_dtype == MOE_W_BF16 || c->hidden % 256 == 0) &&
                         touched_weight_bytes(c) >= kDecodeMinWeightBytes;
  return decode_ok ? MOE_PATH_DECODE : MOE_PATH_GROUPED;
}

moe_status_t validate_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->num_tokens < 0 || c->hidden <= 0 || c->num_experts <= 0 || c->router_width <= 0 ||
      c->top_k <= 0 || c->inter <= 0 || c->shared_inter < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->router_width < c->num_experts || c->top_k > c->router_width) return MOE_ERR_INVALID_ARG;
  if (c->scoring != MOE_SCORING_SOFTMAX && c->scoring != MOE_SCORING_SOFTMAX_BIAS &&
      c->scoring != MOE_SCORING_SIGMOID_BIAS)
    return MOE_ERR_INVALID_ARG;
  if (c->weight_dtype != MOE_W_BF16 && c->weight_dtype != MOE_W_FP8_E4M3_B128 &&
      c->weight_dtype != MOE_W_NVFP4)
    return MOE_ERR_INVALID_ARG;
  if (c->path < MOE_PATH_AUTO || c->path > MOE_PATH_GROUPED) return MOE_ERR_INVALID_ARG;
  if (c->pre_expert_norm && !(c->rms_norm_eps >= 0.0f && c->rms_norm_eps < INFINITY))
    return MOE_ERR_INVALID_ARG;
  // identity experts are wired only on the softmax + correction-bias arm
  if (c->router_width != c->num_experts && c->scoring != MOE_SCORING_SOFTMAX_BIAS)
    return MOE_ERR_UNSUPPORTED;
  if (c->hidden % 128 || c->inter % 128 || c->shared_inter % 128) return MOE_ERR_UNSUPPORTED;
  if (c->top_k > 32 || c->router_width > 1024 || c->num_experts > 1024) return MOE_ERR_UNSUPPORTED;
  // FP8 experts: the down projection's N-tile is 256 wide
  // FP8 experts: the down projection's N-tile is 256 wide; each tile keeps the scales of at
  // most 32 K blocks of 128
  if (c->weight_dtype == MOE_W_FP8_E4M3_B128 &&
      (c->hidden % 256 || c->hidden > 4096 || c->inter > 4096))
    return MOE_ERR_UNSUPPORTED;
  // NVFP4 experts: the scale codes of 16 groups (256 elements) are one 16-byte TMA box
  if (c->weight_dtype == MOE_W_NVFP4 && (c->hidden % 256 || c->inter % 256))
    return MOE_ERR_UNSUPPORTED;
  const int path = resolve_path(c);
  if (path == MOE_PATH_DECODE &&
      (c->num_tokens > kDecodeMaxTokens || c->inter > 1024 || c->shared_inter > 1024 ||
       c->hidden > 8192))
    return MOE_ERR_UNSUPPORTED;
  const long long te = (long long)c->num_tokens * c->top_k;
  if (te > (1ll << 30) || (long long)c->num_tokens * c->hidden > (1ll << 40))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

Layout make_layout(const moe_config_t* c) {
  Layout L{};
  const size_t N = c->num_tokens, H = c->hidden, E = c->num_experts, R = c->router_width;
  const size_t K = c->top_k, I = c->inter, S = c->shared_inter;
  const size_t te = N * K;
  L.path = resolve_path(c);
  L.te = (int)te;
  L.nblk = (int)((te + 1023) / 1024);
  L.max_mtiles = (int)((te < E ? te : E) + te / 128);
  size_t sz[R_NUM] = {};
  sz[R_HDR] = sizeof(WsHeader);
  sz[R_LOGITS] = N * R * 4;
  sz[R_IDX] = te * 4;
  sz[R_W] = te * 4;
  sz[R_ZSUM] = N * 4;
  sz[R_OFFS] = (E + 1) * 4;
  sz[R_P2R] = te * 4;
  sz[R_SPAIRS] = te * 4;
  sz[R_ACTIVE] = E * 4;
  sz[R_XN] = c->pre_expert_norm ? N * H * 2 : 0;   // the routed experts' normed input
  if (L.path == MOE_PATH_GROUPED) {
    sz[R_BLK] = (size_t)L.nblk * E * 4;
    sz[R_LRANK] = te * 4;
    sz[R_TILES] = (size_t)3 * L.max_mtiles * 16;   // the list + two scratch lists
    if (c->weight_dtype == MOE_W_FP8_E4M3_B128) {
      sz[R_XQT] = N * H;                 // E4M3 codes of each token row
      sz[R_XST] = (H / 128) * N * 4;     // and their scales
      sz[R_XP] = te * H;                 // E4M3 codes of the gathered rows
      sz[R_XS] = (H / 128) * te * 4;     // their 1x128 scales, [H/128, te]
      sz[R_HH] = te * I;                 // E4M3 codes of the SwiGLU intermediate
      sz[R_HS] = (I / 128) * te * 4;
    } else {
      sz[R_XP] = te * H * 2;             // x rows in expert-sorted order
      sz[R_HH] = te * I * 2;
    }
    sz[R_Y] = te * H * 2;
    sz[R_SHH] = N * S * 2;
    sz[R_SHY] = S ? N * H * 2 : 0;
  } else {
    sz[R_SYNC] = (kDecodeMaxPairs + 1) * 4;   // per-slot gate/up item counts
    const size_t L2 = I > S ? I : S;
    // gate and up products of every row (E4M3 experts: the shared expert's rows twice, one
    // block per contraction part)
    sz[R_HD] = (te + (c->weight_dtype == MOE_W_FP8_E4M3_B128 ? 2 : 1) * N) * 2 * L2 * 4;
    if (c->deterministic) sz[R_YD] = te * H * 4;
    else sz[R_ACC] = N * H * 4;
    sz[R_SHY] = S ? N * H * 4 : 0;
    if (c->weight_dtype == MOE_W_FP8_E4M3_B128) {
      sz[R_XQT] = N * H;                 // E4M3 codes of the routed experts' input
      sz[R_XST] = (H / 128) * N * 4;     // and their 1x128 scales
    }
    if (c->weight_dtype == MOE_W_NVFP4) sz[R_XQT] = N * H * 2;   // its f16 copy
  }
  size_t off = 0;
  for (int r = 0; r < R_NUM; ++r) {
    L.off[r] = off;
    L.size[r] = sz[r];
    off += align256(sz[r]);
  }
  L.total = off;
  return L;
}

// ------------------------------------------------------------------ device attributes

int g_num_sms[64];
std::mutex g_mu;

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

cudaError_t moe::ensure_dyn_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> have;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  size_t& cur = have[{dev, func}];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

namespace {

bool encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return true;
}

// 2D bf16 map over a [rows, inner] row-major matrix; box {64, box_rows}, 128-byte swizzle,
// zero fill outside the matrix.
bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                   uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D byte map over a [rows, inner] row-major matrix, box {box_inner, box_rows}, no swizzle
// (NVFP4 codes and scale codes).
bool make_map_u8_plain(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                       uint32_t box_inner, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D E4M3 (byte) map over a [rows, inner] row-major matrix; box {128, box_rows}.
bool make_map_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                 uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status_t validate_weights(const moe_config_t* c, const moe_weights_t* w) {
  if (!w || !w->router_w || !w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  if (c->scoring != MOE_SCORING_SOFTMAX && !w->correction_bias) return MOE_ERR_INVALID_ARG;
  if (c->weight_dtype == MOE_W_FP8_E4M3_B128 && (!w->s_gate || !w->s_up || !w->s_down))
    return MOE_ERR_INVALID_ARG;
  if (c->weight_dtype == MOE_W_NVFP4 &&
      (!w->sf_gate || !w->sf_up || !w->sf_down || !w->scale2_gate || !w->scale2_up ||
       !w->scale2_down || !aligned16(w->sf_gate) || !aligned16(w->sf_up) ||
       !aligned16(w->sf_down)))
    return MOE_ERR_INVALID_ARG;
  if (c->shared_inter > 0 && (!w->sh_gate || !w->sh_up || !w->sh_down)) return MOE_ERR_INVALID_ARG;
  if (c->pre_expert_norm && !w->pre_expert_norm_w) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {w->router_w, w->w_gate, w->w_up, w->w_down, w->sh_gate, w->sh_up,
                      w->sh_down, w->sh_gate_vec, c->pre_expert_norm ? w->pre_expert_norm_w
                                                                     : nullptr};
  for (const void* p : ps)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Text of the last failing CUDA call of this thread (moe_last_error_detail).
thread_local char g_detail[256];

moe_status_t cuda_fail(cudaError_t e, const char* what, int line) {
  snprintf(g_detail, sizeof g_detail, "%s failed at api.cu:%d: %s (%d)", what, line,
           cudaGetErrorString(e), (int)e);
  return MOE_ERR_CUDA;
}

#define CK(expr)                                                     \
  do {                                                               \
    cudaError_t ck_e = (expr);                                       \
    if (ck_e != cudaSuccess) return cuda_fail(ck_e, #expr, __LINE__); \
  } while (0)

struct Marks {
  void** ev;
  cudaStream_t st;
  // Records the caller's event for the start (end = 0) or end (end = 1) of a stage.
  moe_status_t mark(int stage, int end) const {
    if (ev && ev[2 * stage + end])
      CK(cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * stage + end]), st));
    return MOE_OK;
  }
};

#define MARK(stage, end)                          \
  do {                                            \
    moe_status_t mk_s = M.mark((stage), (end));   \
    if (mk_s != MOE_OK) return mk_s;              \
  } while (0)

struct Ptrs {
  uint8_t* base;
  const Layout* L;
  template <typename T>
  T* at(Region r) const {
    return L->size[r] ? reinterpret_cast<T*>(base + L->off[r]) : nullptr;
  }
};

// Router + top-K + sort (+ gather of x rows for the grouped chain).
moe_status_t run_routing(const moe_config_t* c, const moe_weights_t* w, const void* x,
                         const Ptrs& P, const uint32_t* forced, bool gather, cudaStream_t st) {
  const Layout& L = *P.L;
  WsHeader* hdr = P.at<WsHeader>(R_HDR);
  RouteArgs ra{};
  ra.x = static_cast<const __nv_bfloat16*>(x);
  ra.router_w = static_cast<const __nv_bfloat16*>(w->router_w);
  ra.logit_bias = w->router_logit_bias;
  ra.corr_bias = c->scoring != MOE_SCORING_SOFTMAX ? w->correction_bias : nullptr;
  ra.forced = forced;
  ra.N = c->num_tokens;
  ra.H = c->hidden;
  ra.E = c->num_experts;
  ra.R = c->router_width;
  ra.K = c->top_k;
  ra.scoring = c->scoring;
  ra.norm = c->norm_topk_prob;
  ra.scale = c->routed_scaling_factor;
  ra.logits = P.at<float>(R_LOGITS);
  ra.idx = P.at<uint32_t>(R_IDX);
  ra.w = P.at<float>(R_W);
  ra.zsum = P.at<float>(R_ZSUM);
  ra.hdr = hdr;
  SortArgs sa{};
  sa.idx = ra.idx;
  sa.te = L.te;
  sa.E = c->num_experts;
  sa.K = c->top_k;
  sa.blk_counts = P.at<uint32_t>(R_BLK);
  sa.local_rank = P.at<uint32_t>(R_LRANK);
  sa.offsets = P.at<uint32_t>(R_OFFS);
  sa.pair_to_row = P.at<uint32_t>(R_P2R);
  sa.sorted_pairs = P.at<uint32_t>(R_SPAIRS);
  sa.active = P.at<uint32_t>(R_ACTIVE);
  sa.tiles = P.at<int4>(R_TILES);
  sa.tiles_tmp = sa.tiles ? sa.tiles + L.max_mtiles : nullptr;
  sa.max_mtiles = L.max_mtiles;
  sa.xq_tok = P.at<uint8_t>(R_XQT);
  sa.xs_tok = P.at<float>(R_XST);
  sa.xp_f16 = c->weight_dtype == MOE_W_NVFP4;
  sa.N = c->num_tokens;
  sa.hdr = hdr;

  // the header starts at zero
  CK(cudaMemsetAsync(hdr, 0, L.off[R_HDR] + L.size[R_HDR], st));
  if (L.path == MOE_PATH_DECODE) {
    CK(launch_router_small(ra, sa, true, st));
    return MOE_OK;
  }
  if (c->num_tokens <= kSmallRouterMaxTokens) {
    CK(launch_router_small(ra, sa, false, st));
    CK(launch_topk(ra, st));
  } else if (router_topk_tc_supported(c->num_tokens, c->hidden, c->router_width, num_sms())) {
    // router GEMM + scoring + top-K in one launch
    CUtensorMap mx, mw;
    const int R = c->router_width;
    if (!make_map_bf16(&mx, x, c->hidden, c->num_tokens, 128) ||
        !make_map_bf16(&mw, w->router_w, c->hidden, R, R <= 256 ? R : 128))
      return MOE_ERR_CUDA;
    CK(launch_router_topk_tc(ra, mx, mw, num_sms(), st));
  } else {
    // router logits on the tensor cores: [N,H] x [R,H]^T -> fp32 [N,R]
    CUtensorMap maps[2][3];
    if (!make_map_bf16(&maps[0][0], x, c->hidden, c->num_tokens, 128) ||
        !make_map_bf16(&maps[0][1], w->router_w, c->hidden, c->router_width, 128))
      return MOE_ERR_CUDA;
    maps[0][2] = maps[0][1];
    GemmArgs g{};
    g.nprob = 1;
    g.p[0].dense_m = c->num_tokens;
    g.p[0].max_mtiles = (c->num_tokens + 127) / 128;
    g.p[0].n_tiles = (c->router_width + 127) / 128;
    g.p[0].num_kb = c->hidden / 64;
    g.p[0].out = ra.logits;
    g.p[0].ldo = c->router_width;
    g.p[0].n_valid = c->router_width;
    g.status = hdr;
    CK(launch_gemm_bf16(kGemmStoreF32, 128, maps, g, num_sms(), st));
    CK(launch_topk(ra, st));
  }
  const bool fp8 = c->weight_dtype == MOE_W_FP8_E4M3_B128;
  // the routed experts' input: x, or its pre-expert RMSNorm (after the routing, which read x)
  const __nv_bfloat16* xe = ra.x;
  if (gather && c->pre_expert_norm) {
    CK(launch_rms_norm_rows(ra.x, static_cast<const __nv_bfloat16*>(w->pre_expert_norm_w),
                            c->rms_norm_eps, c->num_tokens, c->hidden,
                            P.at<__nv_bfloat16>(R_XN), st));
    xe = P.at<__nv_bfloat16>(R_XN);
  }
  if (gather && fp8)
    CK(launch_quant_rows(xe, c->num_tokens, c->hidden, P.at<uint8_t>(R_XQT),
                         P.at<float>(R_XST), st));
  CK(launch_sort(sa, xe, c->hidden, gather && !fp8 ? P.at<__nv_bfloat16>(R_XP) : nullptr,
                 gather && fp8 ? P.at<uint8_t>(R_XP) : nullptr,
                 gather && fp8 ? P.at<float>(R_XS) : nullptr, st));
  return MOE_OK;
}

moe_status_t run_grouped(const moe_config_t* c, const moe_weights_t* w, const void* x, void* out,
                         const Ptrs& P, cudaStream_t st, const Marks& M) {
  const Layout& L = *P.L;
  const int N = c->num_tokens, H = c->hidden, E = c->num_experts, I = c->inter,
            S = c->shared_inter;
  WsHeader* hdr = P.at<WsHeader>(R_HDR);
  const int sms = num_sms();
  const int bn_h = (H % 256 == 0) ? 256 : 128;   // N-tile of the projections back to H
  const bool fp8 = c->weight_dtype == MOE_W_FP8_E4M3_B128;
  const bool nv = c->weight_dtype == MOE_W_NVFP4;
  // Shared expert: a dense SwiGLU FFN on all N rows. With bf16 experts it is problem 0 of the
  // routed launches below; with FP8 or NVFP4 experts it runs as its own bf16 launches here.
  CUtensorMap sh_gu[3], sh_dn[3];
  GemmProblem sh_gu_p{}, sh_dn_p{};
  if (S > 0) {
    if (!make_map_bf16(&sh_gu[0], x, H, N, 128) ||
        !make_map_bf16(&sh_gu[1], w->sh_gate, H, S, 128) ||
        !make_map_bf16(&sh_gu[2], w->sh_up, H, S, 128) ||
        !make_map_bf16(&sh_dn[0], P.at<void>(R_SHH), S, N, 128) ||
        !make_map_bf16(&sh_dn[1], w->sh_down, S, H, bn_h))
      return MOE_ERR_CUDA;
    sh_dn[2] = sh_dn[1];
    sh_gu_p.dense_m = N;
    sh_gu_p.max_mtiles = (N + 127) / 128;
    sh_gu_p.n_tiles = S / 128;
    sh_gu_p.num_kb = H / 64;
    sh_gu_p.out = P.at<void>(R_SHH);
    sh_gu_p.ldo = S;
    sh_dn_p = sh_gu_p;
    sh_dn_p.n_tiles = H / bn_h;
    sh_dn_p.num_kb = S / 64;
    sh_dn_p.out = P.at<void>(R_SHY);
    sh_dn_p.ldo = H;
  }
  MARK(MOE_STAGE_SHARED, 0);
  if (S > 0 && (fp8 || nv)) {
    CUtensorMap maps[2][3] = {{sh_gu[0], sh_gu[1], sh_gu[2]}, {sh_gu[0], sh_gu[1], sh_gu[2]}};
    GemmArgs g{};
    g.nprob = 1;
    g.p[0] = sh_gu_p;
    g.status = hdr;
    CK(launch_gemm_bf16(kGemmSwiGLU, 256, maps, g, sms, st));
    CUtensorMap dmaps[2][3] = {{sh_dn[0], sh_dn[1], sh_dn[2]}, {sh_dn[0], sh_dn[1], sh_dn[2]}};
    g.p[0] = sh_dn_p;
    CK(launch_gemm_bf16(kGemmStoreBF16, bn_h, dmaps, g, sms, st));
  }
  MARK(MOE_STAGE_SHARED, 1);
  // routed experts: grouped gate/up + SiLU*up, then grouped down, over the sorted rows
  if (c->weight_dtype == MOE_W_FP8_E4M3_B128) {
    CUtensorMap ma, mg, mu, mh, md;
    const uint64_t rows = (uint64_t)L.te;
    if (!make_map_u8(&ma, P.at<void>(R_XP), H, rows, 128) ||
        !make_map_u8(&mg, w->w_gate, H, (uint64_t)E * I, 128) ||
        !make_map_u8(&mu, w->w_up, H, (uint64_t)E * I, 128) ||
        !make_map_u8(&mh, P.at<void>(R_HH), I, rows, 128) ||
        !make_map_u8(&md, w->w_down, I, (uint64_t)E * H, 256))
      return MOE_ERR_CUDA;
    Fp8GemmArgs g{};
    g.tiles = P.at<int4>(R_TILES);
    g.hdr = hdr;
    g.max_mtiles = L.max_mtiles;
    g.n_tiles = I / 128;
    g.num_kb = H / 128;
    g.b_rows_per_expert = I;
    g.b_blocks_per_expert = I / 128;
    g.sa = P.at<float>(R_XS);
    g.sa_stride = L.te;
    g.sb0 = w->s_gate;
    g.sb1 = w->s_up;
    g.out = P.at<void>(R_HH);
    g.ldo = I;
    g.out_scales = P.at<float>(R_HS);
    g.out_scale_stride = L.te;
    g.status = hdr;
    MARK(MOE_STAGE_GATE_UP, 0);
    CK(launch_gemm_fp8(0, ma, mg, mu, g, sms, st));
    MARK(MOE_STAGE_GATE_UP, 1);
    g.n_tiles = H / 256;
    g.num_kb = I / 128;
    g.b_rows_per_expert = H;
    g.b_blocks_per_expert = H / 128;
    g.sa = P.at<float>(R_HS);
    g.sb0 = w->s_down;
    g.sb1 = nullptr;
    g.out = P.at<void>(R_Y);
    g.ldo = H;
    g.out_scales = nullptr;
    MARK(MOE_STAGE_DOWN, 0);
    CK(launch_gemm_fp8(1, mh, md, md, g, sms, st));
    MARK(MOE_STAGE_DOWN, 1);
  } else if (nv) {
    // NVFP4 experts: codes and scale codes streamed, dequantised to f16 in shared memory;
    // the gathered rows and the SwiGLU intermediate are f16 (2-byte maps)
    CUtensorMap gu[5], dn[5];
    const uint64_t rows = (uint64_t)L.te;
    if (!make_map_bf16(&gu[0], P.at<void>(R_XP), H, rows, 128) ||
        !make_map_u8_plain(&gu[1], w->w_gate, H / 2, (uint64_t)E * I, 32, 128) ||
        !make_map_u8_plain(&gu[2], w->w_up, H / 2, (uint64_t)E * I, 32, 128) ||
        !make_map_u8_plain(&gu[3], w->sf_gate, H / 16, (uint64_t)E * I, 16, 128) ||
        !make_map_u8_plain(&gu[4], w->sf_up, H / 16, (uint64_t)E * I, 16, 128) ||
        !make_map_bf16(&dn[0], P.at<void>(R_HH), I, rows, 128) ||
        !make_map_u8_plain(&dn[1], w->w_down, I / 2, (uint64_t)E * H, 32, bn_h) ||
        !make_map_u8_plain(&dn[3], w->sf_down, I / 16, (uint64_t)E * H, 16, bn_h))
      return MOE_ERR_CUDA;
    dn[2] = dn[1];
    dn[4] = dn[3];
    NvGemmArgs g{};
    g.tiles = P.at<int4>(R_TILES);
    g.hdr = hdr;
    g.max_mtiles = L.max_mtiles;
    g.n_tiles = I / 128;
    g.num_kb = H / 64;
    g.b_rows_per_expert = I;
    g.s2_0 = w->scale2_gate;
    g.s2_1 = w->scale2_up;
    g.out = P.at<void>(R_HH);
    g.ldo = I;
    g.status = hdr;
    MARK(MOE_STAGE_GATE_UP, 0);
    CK(launch_gemm_nvfp4(kGemmSwiGLU, 256, gu, g, sms, st));
    MARK(MOE_STAGE_GATE_UP, 1);
    g.n_tiles = H / bn_h;
    g.num_kb = I / 64;
    g.b_rows_per_expert = H;
    g.s2_0 = w->scale2_down;
    g.s2_1 = w->scale2_down;
    g.out = P.at<void>(R_Y);
    g.ldo = H;
    MARK(MOE_STAGE_DOWN, 0);
    CK(launch_gemm_nvfp4(kGemmStoreBF16, bn_h, dn, g, sms, st));
    MARK(MOE_STAGE_DOWN, 1);
  } else {
    // routed problem (plus the shared expert as problem 0 when present)
    CUtensorMap gu[3], dn[3];
    const uint64_t rows = (uint64_t)L.te;
    if (!make_map_bf16(&gu[0], P.at<void>(R_XP), H, rows, 128) ||
        !make_map_bf16(&gu[1], w->w_gate, H, (uint64_t)E * I, 128) ||
        !make_map_bf16(&gu[2], w->w_up, H, (uint64_t)E * I, 128) ||
        !make_map_bf16(&dn[0], P.at<void>(R_HH), I, rows, 128) ||
        !make_map_bf16(&dn[1], w->w_down, I, (uint64_t)E * H, bn_h))
      return MOE_ERR_CUDA;
    dn[2] = dn[1];
    GemmProblem rgu{};
    rgu.tiles = P.at<int4>(R_TILES);
    rgu.count = hdr;
    rgu.max_mtiles = L.max_mtiles;
    rgu.n_tiles = I / 128;
    rgu.num_kb = H / 64;
    rgu.b_rows_per_expert = I;
    rgu.out = P.at<void>(R_HH);
    rgu.ldo = I;
    GemmProblem rdn = rgu;
    rdn.n_tiles = H / bn_h;
    rdn.num_kb = I / 64;
    rdn.b_rows_per_expert = H;
    rdn.out = P.at<void>(R_Y);
    rdn.ldo = H;
    GemmArgs g{};
    g.status = hdr;
    CUtensorMap maps[2][3];
    if (S > 0) {
      g.nprob = 2;
      g.p[0] = sh_gu_p;
      g.p[1] = rgu;
      for (int i = 0; i < 3; ++i) { maps[0][i] = sh_gu[i]; maps[1][i] = gu[i]; }
    } else {
      g.nprob = 1;
      g.p[0] = rgu;
      for (int i = 0; i < 3; ++i) maps[0][i] = maps[1][i] = gu[i];
    }
    MARK(MOE_STAGE_GATE_UP, 0);
    CK(launch_gemm_bf16(kGemmSwiGLU, 256, maps, g, sms, st));
    MARK(MOE_STAGE_GATE_UP, 1);
    if (S > 0) {
      g.p[0] = sh_dn_p;
      g.p[1] = rdn;
      for (int i = 0; i < 3; ++i) { maps[0][i] = sh_dn[i]; maps[1][i] = dn[i]; }
    } else {
      g.p[0] = rdn;
      for (int i = 0; i < 3; ++i) maps[0][i] = maps[1][i] = dn[i];
    }
    MARK(MOE_STAGE_DOWN, 0);
    CK(launch_gemm_bf16(kGemmStoreBF16, bn_h, maps, g, sms, st));
    MARK(MOE_STAGE_DOWN, 1);
  }
  CombineArgs ca{};
  ca.x = static_cast<const __nv_bfloat16*>(x);
  ca.pair_to_row = P.at<uint32_t>(R_P2R);
  ca.w = P.at<float>(R_W);
  ca.zsum = c->router_width > c->num_experts ? P.at<float>(R_ZSUM) : nullptr;
  ca.y = P.at<void>(R_Y);
  ca.y_is_f32 = 0;
  ca.shy = S > 0 ? P.at<void>(R_SHY) : nullptr;
  ca.shy_is_f32 = 0;
  ca.sh_gate_vec = static_cast<const __nv_bfloat16*>(w->sh_gate_vec);
  ca.N = N;
  ca.H = H;
  ca.K = c->top_k;
  ca.out = static_cast<__nv_bfloat16*>(out);
  MARK(MOE_STAGE_COMBINE, 0);
  CK(launch_combine(ca, st));
  MARK(MOE_STAGE_COMBINE, 1);
  return MOE_OK;
}

// The decode chain: one memset of the header and the fp32 accumulators, one cooperative kernel
// (router, top-K, sort, projections, combine). Its time is reported as the gate/up stage.
moe_status_t run_decode(const moe_config_t* c, const moe_weights_t* w, const void* x, void* out,
                        const Ptrs& P, const uint32_t* forced, cudaStream_t st, const Marks& M) {
  const Layout& L = *P.L;
  const int N = c->num_tokens, H = c->hidden, S = c->shared_inter;
  const int E = c->num_experts, I = c->inter;
  WsHeader* hdr = P.at<WsHeader>(R_HDR);
  MARK(MOE_STAGE_ROUTE, 0);
  CK(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));   // the kernel clears its accumulators
  // the routed experts' input: x, or its pre-expert RMSNorm (written by the kernel's phase 0)
  const void* xn = c->pre_expert_norm ? P.at<void>(R_XN) : x;
  MARK(MOE_STAGE_ROUTE, 1);
  DecodeArgs d{};
  d.x = static_cast<const __nv_bfloat16*>(x);
  d.router_w = static_cast<const __nv_bfloat16*>(w->router_w);
  d.logit_bias = w->router_logit_bias;
  d.corr_bias = c->scoring != MOE_SCORING_SOFTMAX ? w->correction_bias : nullptr;
  d.forced = forced;
  d.sh_gate_vec = S > 0 ? static_cast<const __nv_bfloat16*>(w->sh_gate_vec) : nullptr;
  d.norm_w = c->pre_expert_norm ? static_cast<const __nv_bfloat16*>(w->pre_expert_norm_w) : nullptr;
  d.eps = c->rms_norm_eps;
  d.xn = c->pre_expert_norm ? P.at<__nv_bfloat16>(R_XN) : nullptr;
  d.N = N;
  d.H = H;
  d.E = E;
  d.R = c->router_width;
  d.K = c->top_k;
  d.I = I;
  d.S = S;
  d.te = L.te;
  d.scoring = c->scoring;
  d.norm = c->norm_topk_prob;
  d.scale = c->routed_scaling_factor;
  d.logits = P.at<float>(R_LOGITS);
  d.idx = P.at<uint32_t>(R_IDX);
  d.w = P.at<float>(R_W);
  d.zsum = P.at<float>(R_ZSUM);
  d.offsets = P.at<uint32_t>(R_OFFS);
  d.sorted_pairs = P.at<uint32_t>(R_SPAIRS);
  d.pair_to_row = P.at<uint32_t>(R_P2R);
  d.active = P.at<uint32_t>(R_ACTIVE);
  d.hd = P.at<float>(R_HD);
  d.ldh = I > S ? I : S;
  d.yd = P.at<float>(R_YD);
  d.acc = P.at<float>(R_ACC);
  d.shy = P.at<float>(R_SHY);
  d.h_cnt = P.at<uint32_t>(R_SYNC);
  d.hdr = hdr;
  d.out = static_cast<__nv_bfloat16*>(out);
  const bool fp8 = c->weight_dtype == MOE_W_FP8_E4M3_B128;
  d.fp8 = fp8 ? 1 : 0;
  d.s_gate = fp8 ? w->s_gate : nullptr;
  d.s_up = fp8 ? w->s_up : nullptr;
  d.s_down = fp8 ? w->s_down : nullptr;
  d.xq = fp8 ? P.at<uint8_t>(R_XQT) : nullptr;
  d.xs = fp8 ? P.at<float>(R_XST) : nullptr;
  const bool nv = c->weight_dtype == MOE_W_NVFP4;
  d.nv = nv ? 1 : 0;
  d.s2_gate = nv ? w->scale2_gate : nullptr;
  d.s2_up = nv ? w->scale2_up : nullptr;
  d.s2_down = nv ? w->scale2_down : nullptr;
  d.xh = nv ? P.at<__half>(R_XQT) : nullptr;
  CUtensorMap maps[kDmNum];
  int bg = 0, bd = 0;
  decode_tile_rows(H, I, S, &bg, &bd);
  if (fp8) {   // E4M3 routed weights and expert input: 128 codes per 128-byte box row
    if (!make_map_u8(&maps[kDmWg], w->w_gate, H, (uint64_t)E * I, bg) ||
        !make_map_u8(&maps[kDmWu], w->w_up, H, (uint64_t)E * I, bg) ||
        !make_map_u8(&maps[kDmWd], w->w_down, I, (uint64_t)E * H, bd) ||
        !make_map_bf16(&maps[kDmX], x, H, N, kDecodeBoxRowsX) ||
        !make_map_u8(&maps[kDmXn], d.xq, H, N, kDecodeBoxRowsX))
      return MOE_ERR_CUDA;
  } else if (nv) {   // NVFP4: codes {32, rows}, scale codes {16, rows}, f16 input copy
    if (!make_map_u8_plain(&maps[kDmWg], w->w_gate, H / 2, (uint64_t)E * I, 32, bg) ||
        !make_map_u8_plain(&maps[kDmWu], w->w_up, H / 2, (uint64_t)E * I, 32, bg) ||
        !make_map_u8_plain(&maps[kDmWd], w->w_down, I / 2, (uint64_t)E * H, 32, bd) ||
        !make_map_u8_plain(&maps[kDmFg], w->sf_gate, H / 16, (uint64_t)E * I, 16, bg) ||
        !make_map_u8_plain(&maps[kDmFu], w->sf_up, H / 16, (uint64_t)E * I, 16, bg) ||
        !make_map_u8_plain(&maps[kDmFd], w->sf_down, I / 16, (uint64_t)E * H, 16, bd) ||
        !make_map_bf16(&maps[kDmX], x, H, N, kDecodeBoxRowsX) ||
        !make_map_bf16(&maps[kDmXn], d.xh, H, N, kDecodeBoxRowsX))
      return MOE_ERR_CUDA;
  } else if (!make_map_bf16(&maps[kDmWg], w->w_gate, H, (uint64_t)E * I, bg) ||
             !make_map_bf16(&maps[kDmWu], w->w_up, H, (uint64_t)E * I, bg) ||
             !make_map_bf16(&maps[kDmWd], w->w_down, I, (uint64_t)E * H, bd) ||
             !make_map_bf16(&maps[kDmX], x, H, N, kDecodeBoxRowsX) ||
             !make_map_bf16(&maps[kDmXn], xn, H, N, kDecodeBoxRowsX)) {
    return MOE_ERR_CUDA;
  }
  if (S > 0) {
    if (!make_map_bf16(&maps[kDmSg], w->sh_gate, H, S, bg) ||
        !make_map_bf16(&maps[kDmSu], w->sh_up, H, S, bg) ||
        !make_map_bf16(&maps[kDmSd], w->sh_down, S, H, bd))
      return MOE_ERR_CUDA;
  } else {   // never read without a shared expert
    maps[kDmSg] = maps[kDmWg];
    maps[kDmSu] = maps[kDmWu];
    maps[kDmSd] = maps[kDmWd];
  }
  if (!nv) {   // never read without NVFP4 experts
    maps[kDmFg] = maps[kDmWg];
    maps[kDmFu] = maps[kDmWu];
    maps[kDmFd] = maps[kDmWd];
  }
  MARK(MOE_STAGE_SHARED, 0);
  MARK(MOE_STAGE_SHARED, 1);
  MARK(MOE_STAGE_GATE_UP, 0);
  CK(launch_decode_forward(d, maps, st));
  MARK(MOE_STAGE_GATE_UP, 1);
  MARK(MOE_STAGE_DOWN, 0);
  MARK(MOE_STAGE_DOWN, 1);
  MARK(MOE_STAGE_COMBINE, 0);
  MARK(MOE_STAGE_COMBINE, 1);
  return MOE_OK;
}

moe_status_t check_call(const moe_config_t* cfg, const moe_weights_t* w, const void* x,
                        void* workspace, size_t workspace_bytes, Layout* L) {
  moe_status_t s = validate_config(cfg);
  if (s != MOE_OK) return s;
  s = validate_weights(cfg, w);
  if (s != MOE_OK) return s;
  *L = make_layout(cfg);
  if (cfg->num_tokens == 0) return MOE_OK;
  if (!x || !workspace || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < L->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!encode_fn()) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t forward_impl(const moe_config_t* cfg, const moe_weights_t* weights, const void* x,
                          void* out, void* workspace, size_t workspace_bytes, void* stream,
                          uint32_t* topk_idx_out, float* topk_w_out, const uint32_t* forced_idx,
                          void** events) {
  Layout L;
  moe_status_t s = check_call(cfg, weights, x, workspace, workspace_bytes, &L);
  if (s != MOE_OK) return s;
  if (cfg->num_tokens == 0) return MOE_OK;
  if (!out || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  (void)cudaGetLastError();   // a stale error of an earlier call must not fail this one
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ptrs P{static_cast<uint8_t*>(workspace), &L};
  Marks M{events, st};
  if (L.path == MOE_PATH_GROUPED) {
    MARK(MOE_STAGE_ROUTE, 0);
    s = run_routing(cfg, weights, x, P, forced_idx, true, st);
    if (s != MOE_OK) return s;
    MARK(MOE_STAGE_ROUTE, 1);
    s = run_grouped(cfg, weights, x, out, P, st, M);
  } else {
    s = run_decode(cfg, weights, x, out, P, forced_idx, st, M);
  }
  if (s != MOE_OK) return s;
  const size_t te = (size_t)L.te;
  if (topk_idx_out)
    CK(cudaMemcpyAsync(topk_idx_out, P.at<void>(R_IDX), te * 4, cudaMemcpyDeviceToDevice, st));
  if (topk_w_out)
    CK(cudaMemcpyAsync(topk_w_out, P.at<void>(R_W), te * 4, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* weights, const void* x,
                         void* out, void* workspace, size_t workspace_bytes, void* stream,
                         uint32_t* topk_idx_out, float* topk_w_out, const uint32_t* forced_idx) {
  return forward_impl(cfg, weights, x, out, workspace, workspace_bytes, stream, topk_idx_out,
                      topk_w_out, forced_idx, nullptr);
}

moe_status_t moe_forward_profiled(const moe_config_t* cfg, const moe_weights_t* weights,
                                  const void* x, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream, void** events) {
  return forward_impl(cfg, weights, x, out, workspace, workspace_bytes, stream, nullptr, nullptr,
                      nullptr, events);
}


moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status_t s = validate_config(cfg);
  if (s != MOE_OK) return s;
  *bytes = make_layout(cfg).total;
  return MOE_OK;
}

moe_status_t moe_route(const moe_config_t* cfg, const moe_weights_t* weights, const void* x,
                       void* workspace, size_t workspace_bytes, void* stream, uint32_t* idx_out,
                       float* w_out, float* zsum_out, uint32_t* offsets_out,
                       uint32_t* sorted_pairs_out, uint32_t* pair_to_row_out) {
  Layout L;
  moe_status_t s = check_call(cfg, weights, x, workspace, workspace_bytes, &L);
  if (s != MOE_OK) return s;
  if (cfg->num_tokens == 0) return MOE_OK;
  (void)cudaGetLastError();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ptrs P{static_cast<uint8_t*>(workspace), &L};
  s = run_routing(cfg, weights, x, P, nullptr, false, st);
  if (s != MOE_OK) return s;
  const size_t te = (size_t)L.te, N = cfg->num_tokens, E = cfg->num_experts;
  struct Copy { void* dst; Region r; size_t bytes; } copies[] = {
      {idx_out, R_IDX, te * 4},        {w_out, R_W, te * 4},
      {zsum_out, R_ZSUM, N * 4},       {offsets_out, R_OFFS, (E + 1) * 4},
      {sorted_pairs_out, R_SPAIRS, te * 4}, {pair_to_row_out, R_P2R, te * 4}};
  for (const Copy& cp : copies)
    if (cp.dst)
      CK(cudaMemcpyAsync(cp.dst, P.at<void>(cp.r), cp.bytes, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

moe_status_t moe_read_device_status(const void* workspace, void* stream, int32_t* status) {
  if (!workspace || !status) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaStreamSynchronize(st));
  CK(cudaMemcpy(status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_selftest_bounded_wait(void* workspace, long long limit_cycles, void* stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || limit_cycles < 1 ||
      limit_cycles > kSpinLimitCycles)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  CK(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
  CK(launch_bounded_wait_selftest(hdr, limit_cycles, st));
  return MOE_OK;
}

const char* moe_last_error_detail(void) { return g_detail; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
