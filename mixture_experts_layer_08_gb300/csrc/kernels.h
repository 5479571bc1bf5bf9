// Host-side launchers of the MoE kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace moe {

// Launches `k` as a programmatic dependent of the previous kernel on `st`: it may start
// before that kernel finishes and must call pdl_wait() before reading its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

struct RouteArgs {
  const __nv_bfloat16* x;          // [N,H]
  const __nv_bfloat16* router_w;   // [R,H]
  const float* logit_bias;         // [R] or null
  const float* corr_bias;          // [R] or null (selection only)
  const uint32_t* forced;          // [N,K] or null
  int N, H, E, R, K, scoring, norm;
  float scale;
  float* logits;                   // [N,R]
  uint32_t* idx;                   // [N,K]
  float* w;                        // [N,K]
  float* zsum;                     // [N]
  WsHeader* hdr;
};

struct SortArgs {
  const uint32_t* idx;             // [te]
  int te, E, K;
  uint32_t* blk_counts;            // [ceil(te/1024), E]
  uint32_t* local_rank;            // [te]
  uint32_t* offsets;               // [E+1]
  uint32_t* pair_to_row;           // [te]
  uint32_t* sorted_pairs;          // [te]
  uint32_t* active;                // [E] experts with rows, ascending
  int4* tiles;                     // [max m-tiles] (expert, row0, row1, 0)
  int4* tiles_tmp;                 // [2 * max m-tiles] scratch for ordering the list
  int max_mtiles;
  const uint8_t* xq_tok;           // FP8 experts: E4M3 codes of each token row [N, H]
  const float* xs_tok;             // and their 1x128 scales [H/128, N]
  int xp_f16;                      // gather x rows as f16 (NVFP4 experts) instead of bf16
  int N;
  WsHeader* hdr;
};

// Router logits (warp per router column, up to 16 tokens per block) followed, when
// `fuse_tail` is set (N <= 16), by top-K of every token and the stable sort in the last
// block to finish. Otherwise only the logits are written.
cudaError_t launch_router_small(const RouteArgs& a, const SortArgs& s, bool fuse_tail,
                                cudaStream_t st);
// Scoring + top-K + weights, one warp per token.
cudaError_t launch_topk(const RouteArgs& a, cudaStream_t st);
// Router GEMM on the tensor cores with the scoring + top-K fused (logits, idx, w, zsum): the
// contraction of each 128-token tile split over a cluster of CTAs whose partial sums are
// combined in a fixed order. tm_x: x [N,H], box {64, 128}; tm_w: router [R,H], box {64, R}
// for R <= 256, else {64, 128}. Supported when router_topk_tc_supported().
bool router_topk_tc_supported(int N, int H, int R, int num_sms);
cudaError_t launch_router_topk_tc(const RouteArgs& a, const CUtensorMap& tm_x,
                                  const CUtensorMap& tm_w, int num_sms, cudaStream_t st);
// Per 1x128 E4M3 quantisation of the token rows (FP8 experts): codes [N,H], scales [H/128,N].
// xn[t,:] = bf16(x[t,:] * g / sqrt(mean(x[t,:]^2) + eps)), fp32 arithmetic; one warp per row.
cudaError_t launch_rms_norm_rows(const __nv_bfloat16* x, const __nv_bfloat16* g, float eps, int N,
                                 int H, __nv_bfloat16* xn, cudaStream_t st);
cudaError_t launch_quant_rows(const __nv_bfloat16* x, int N, int H, uint8_t* q, float* sc,
                              cudaStream_t st);
// Stable counting sort of the (token, slot) pairs by expert (count / scan / scatter) and the
// m-tile list of the grouped GEMM. Scatter also gathers x rows (bf16) into `xp` when given,
// or the quantised token rows (s.xq_tok / s.xs_tok) into `xq` + `xs` (scales [H/128, te]).
cudaError_t launch_sort(const SortArgs& s, const __nv_bfloat16* x, int H, __nv_bfloat16* xp,
                        uint8_t* xq, float* xs, cudaStream_t st);

// Decode chain limits: tokens per forward and (token, slot) pairs.
constexpr int kDecodeMaxTokens = 16;
constexpr int kDecodeMaxPairs = 512;

// Raises `func`'s dynamic shared memory limit on the current device to at least `bytes`,
// calling the runtime only when the limit has to grow (not on every launch).
cudaError_t ensure_dyn_smem(const void* func, size_t bytes);

// Decode chain: the whole block forward of a few tokens in one cooperative launch -- router,
// top-K and sort, gate/up and down projections of the active experts and the shared expert as
// skinny tensor-core GEMMs (weights as the wide B operand, the tokens as A rows), combine.
struct DecodeArgs {
  const __nv_bfloat16* x;          // [N,H]
  const __nv_bfloat16* router_w;   // [R,H]
  const float* logit_bias;         // [R] or null
  const float* corr_bias;          // [R] or null (selection only)
  const uint32_t* forced;          // [N,K] or null
  const __nv_bfloat16* sh_gate_vec;    // [H] or null
  const __nv_bfloat16* norm_w;     // [H] pre-expert RMSNorm weight, or null (no norm)
  float eps;                       // its epsilon
  __nv_bfloat16* xn;               // [N,H] the routed experts' input, written in phase 0 (norm)
  int N, H, E, R, K, I, S, te, scoring, norm;
  float scale;
  float* logits;                   // [N,R]
  // routing results, written by block 0 for inspection and the top-K outputs
  uint32_t* idx;                   // [N,K]
  float* w;                        // [N,K]
  float* zsum;                     // [N]
  uint32_t* offsets;               // [E+1]
  uint32_t* sorted_pairs;          // [te]
  uint32_t* pair_to_row;           // [te]
  uint32_t* active;                // [E]
  // fp32 accumulators, cleared by the kernel
  float* hd;                       // [te + N, 2*ldh] gate (cols < ldh) and up products
                                   // (row = sorted row, shared rows te + t)
  int ldh;                         // max(I, S)
  float* yd;                       // [te, H] expert outputs (deterministic) or null
  float* acc;                      // [N, H] atomic accumulator (atomic mode) or null
  float* shy;                      // [N, H] shared expert output
  uint32_t* h_cnt;                 // [kDecodeMaxPairs + 1] gate/up work items finished per slot
                                   // (the last entry: shared expert)
  WsHeader* hdr;                   // done_blocks (grid barriers) zero on entry
  __nv_bfloat16* out;              // [N,H]
  // E4M3 routed experts (the shared expert stays bf16)
  int fp8;
  const float* s_gate;             // [E, I/128, H/128] block scales of Wg
  const float* s_up;               // [E, I/128, H/128] of Wu
  const float* s_down;             // [E, H/128, I/128] of Wd
  uint8_t* xq;                     // [N, H] E4M3 codes of the routed experts' input (phase 0)
  float* xs;                       // [H/128, N] their 1x128 scales
  // NVFP4 routed experts (the shared expert stays bf16)
  int nv;
  const float* s2_gate;            // [E] scale2 of Wg
  const float* s2_up;              // [E] of Wu
  const float* s2_down;            // [E] of Wd
  __half* xh;                      // [N, H] f16 copy of the routed experts' input (phase 0)
};
// Tensor maps (box 128 bytes wide, 128-byte swizzle) the decode kernel streams from: bf16
// {64, rows}, or with E4M3 routed experts uint8 {128, rows} for Wg, Wu, Wd and the routed
// experts' input (kDmXn then maps the E4M3 codes xq). With NVFP4 routed experts Wg, Wu, Wd map
// the packed codes (uint8 {32, rows}, no swizzle), kDmFg, kDmFu, kDmFd their scale codes
// (uint8 {16, rows}), and kDmXn the f16 input copy xh ({64, 16}, 128-byte swizzle).
enum DecodeMap { kDmWg = 0, kDmWu, kDmSg, kDmSu, kDmWd, kDmSd, kDmX, kDmXn, kDmFg, kDmFu, kDmFd,
                 kDmNum };
// Box rows: x and the routed experts' input xn (x itself without a pre-expert norm) 16;
// gate/up weights (Wg, Wu, Sg, Su) *bn_g; down weights (Wd, Sd) *bn_d.
constexpr int kDecodeBoxRowsX = 16;
void decode_tile_rows(int H, int I, int S, int* bn_g, int* bn_d);
// The decode forward as one cooperative launch.
cudaError_t launch_decode_forward(const DecodeArgs& a, const CUtensorMap* maps, cudaStream_t st);

// out[t] = sum_k w[t,k] * Y[pair_to_row[t,k]] (+ acc[t]) + zsum[t] * x[t] + gamma_t * shy[t]
struct CombineArgs {
  const __nv_bfloat16* x;
  const uint32_t* pair_to_row;
  const float* w;
  const float* zsum;               // identity-expert weight per token; null without them
  const void* y;                   // [rows, H] bf16 (y_is_f32 = 0) or fp32; may be null
  int y_is_f32;
  const float* acc;                // [N,H] or null
  const void* shy;                 // [N,H] bf16 or fp32 (shy_is_f32) or null
  int shy_is_f32;
  const __nv_bfloat16* sh_gate_vec;    // [H] or null
  int N, H, K;
  __nv_bfloat16* out;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);

// Exercises the bounded device wait: waits `limit_cycles` on a barrier that never completes,
// then records MOE_ERR_DEVICE_TIMEOUT in the header.
cudaError_t launch_bounded_wait_selftest(WsHeader* hdr, long long limit_cycles, cudaStream_t st);

// tcgen05 grouped GEMM. Epilogue modes.
enum GemmMode { kGemmSwiGLU = 0, kGemmStoreBF16 = 1, kGemmStoreF32 = 2 };

// One GEMM problem of a launch: rows grouped into 128-row m-tiles (from a device-built list,
// or dense), each m-tile times n_tiles output tiles.
struct GemmProblem {
  const int4* tiles;               // m-tile list (expert, row0, row1, 0), or null: dense
  const WsHeader* count;           // its num_mtiles (when `tiles` is given)
  int dense_m;                     // rows of a dense problem
  int max_mtiles;                  // upper bound on m-tiles (grid sizing)
  int n_tiles;                     // output tiles along N per m-tile
  int num_kb;                      // contraction blocks of 64 (bf16)
  int b_rows_per_expert;           // rows of one expert in the B tensor map
  void* out;
  int ldo;                         // elements
  int n_valid;                     // valid output columns (fp32 store mode)
};

// Up to two problems share one persistent launch (problem 0's tiles first), e.g. the shared
// expert and the routed experts.
struct GemmArgs {
  GemmProblem p[2];
  int nprob;
  WsHeader* status;
};

// maps[i] = {A, B0, B1} of problem i. A: [rows, K] bf16, box {64, 128}; B0 (and B1 for
// SwiGLU): [rows, K] bf16, box {64, BN/2 (SwiGLU) or BN}.
cudaError_t launch_gemm_bf16(int mode, int bn, const CUtensorMap maps[2][3], const GemmArgs& g,
                             int num_sms, cudaStream_t st);

// FP8 (E4M3, block-scaled) grouped GEMM over the expert-sorted rows. mode 0: gate/up with
// SwiGLU and 1x128 E4M3 quantisation of the intermediate; mode 1: down projection to bf16.
struct Fp8GemmArgs {
  const int4* tiles;               // m-tile list (expert, row0, row1, 0)
  const WsHeader* hdr;             // number of m-tiles
  int max_mtiles;
  int n_tiles;                     // mode 0: I/128 (gate/up pairs); mode 1: H/256
  int num_kb;                      // contraction / 128
  int b_rows_per_expert;           // rows of one expert in the B maps
  int b_blocks_per_expert;         // b_rows_per_expert / 128 (scale rows per expert)
  const float* sa;                 // A scales [num_kb, sa_stride]
  int sa_stride;
  const float* sb0;                // B scales [E, b_blocks, num_kb] (gate, or down)
  const float* sb1;                // up scales (mode 0)
  void* out;                       // mode 0: E4M3 codes [rows, ldo]; mode 1: bf16 [rows, ldo]
  int ldo;
  float* out_scales;               // mode 0: [ldo/128, out_scale_stride]
  int out_scale_stride;
  WsHeader* status;
};
// A: uint8 map [rows, K], box {128, 128}; B: uint8 map [rows, K], box {128, 128 (mode 0) or
// 256 (mode 1)}.
cudaError_t launch_gemm_fp8(int mode, const CUtensorMap& a, const CUtensorMap& b0,
                            const CUtensorMap& b1, const Fp8GemmArgs& g, int num_sms,
                            cudaStream_t st);

// NVFP4 grouped GEMM over the expert-sorted f16 rows (weights dequantised exactly to f16 in
// shared memory, f16 MMA, scale2 in the epilogue). mode kGemmSwiGLU (bn 256: 128 gate + 128 up
// rows) or kGemmStoreBF16 (bn 256 or 128).
struct NvGemmArgs {
  const int4* tiles;               // m-tile list (expert, row0, row1, 0)
  const WsHeader* hdr;             // number of m-tiles
  int max_mtiles;
  int n_tiles;                     // output tiles along N per m-tile
  int num_kb;                      // contraction / 64
  int b_rows_per_expert;           // rows of one expert matrix (I for gate/up, H for down)
  const float* s2_0;               // [E] scale2 of B0 (gate, or down)
  const float* s2_1;               // [E] scale2 of B1 (up)
  void* out;                       // f16 [rows, ldo] (SwiGLU) or bf16 (store)
  int ldo;
  WsHeader* status;
};
// maps: A f16 [rows, K] box {64, 128} (128-byte swizzle); codes of B0 and B1: uint8
// [E*rows, K/2] box {32, b_rows}; scale codes of B0 and B1: uint8 [E*rows, K/16] box
// {16, b_rows} (no swizzle); b_rows = bn/2 for SwiGLU, else bn. Needs K % 256 == 0.
cudaError_t launch_gemm_nvfp4(int mode, int bn, const CUtensorMap maps[5], const NvGemmArgs& g,
                              int num_sms, cudaStream_t st);

}  // namespace moe
