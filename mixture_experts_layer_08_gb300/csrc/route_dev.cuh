// Routing device functions shared by the routing kernels and the fused decode kernel: the
// per-token softmax / top-K / renormalisation of one warp and a block-wide exclusive scan.
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (`moe_topk_softmax_batched` with
// `norm_topk_prob`) and "spark_model/layers/moe/forward.rs" (`forward`: softmax scores +
// correction bias for selection, unbiased softmax x scaling for the weights, selected
// identity experts folded into zero_accum).
#pragma once
#include "kernels.h"

namespace moe {
namespace {

// Does candidate (va, ia) rank before (vb, ib)? Higher score first, lower id on a tie.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Does the scoring add the correction bias to the selection score (never to the weights)?
__device__ __forceinline__ bool selection_biased(int scoring) {
  return scoring == MOE_SCORING_SOFTMAX_BIAS || scoring == MOE_SCORING_SIGMOID_BIAS;
}

// The sigmoid arm's score: 1 / (1 + e^-x).
__device__ __forceinline__ float sigmoid_score(float x) { return 1.0f / (1.0f + expf(-x)); }

// One warp routes one token. `L` is the token's fp32 logit row; `p` and `sel` are per-warp
// shared scratch of R floats. Lane k < K writes slot k of idx/w; lane 0 writes zsum.
__device__ void route_token_warp(const float* L, const float* logit_bias, const float* corr_bias,
                                 int R, int E, int K, int scoring, int norm, float scale,
                                 const uint32_t* forced, float* p, float* sel, uint32_t* idx_out,
                                 float* w_out, float* zsum_out, uint32_t* idx_smem) {
  const int lane = threadIdx.x & 31;
  const bool biased = selection_biased(scoring) && corr_bias;
  float mx = -INFINITY;
  for (int r0 = 0; r0 < R; r0 += 128) {
    // four columns' logits and biases in flight before any is used
    float v[4], lb[4], cb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * 32 + lane;
      v[u] = r < R ? __ldcg(L + r) : 0.0f;
      lb[u] = (r < R && logit_bias) ? logit_bias[r] : 0.0f;
      cb[u] = (r < R && biased) ? corr_bias[r] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * 32 + lane;
      if (r < R) {
        const float x = v[u] + lb[u];
        p[r] = x;
        sel[r] = cb[u];   // the selection bias; the score is added below
        mx = fmaxf(mx, x);
      }
    }
  }
  if (scoring == MOE_SCORING_SIGMOID_BIAS) {
#pragma unroll 4
    for (int r = lane; r < R; r += 32) {
      const float pr = sigmoid_score(p[r]);
      p[r] = pr;
      sel[r] = pr + sel[r];
    }
  } else {
    mx = warp_max(mx);
    float den = 0.0f;
#pragma unroll 4
    for (int r = lane; r < R; r += 32) {
      float e = expf(p[r] - mx);
      p[r] = e;
      den += e;
    }
    den = warp_sum(den);
#pragma unroll 4
    for (int r = lane; r < R; r += 32) {
      float pr = p[r] / den;
      p[r] = pr;
      sel[r] = pr + sel[r];
    }
  }
  __syncwarp();
  uint32_t my_idx = 0;
  for (int k = 0; k < K; ++k) {
    int best;
    if (forced) {
      best = (int)forced[k];
    } else {
      float bv = -INFINITY;
      best = 0x7fffffff;
#pragma unroll 4
      for (int r = lane; r < R; r += 32) {
        float v = sel[r];
        if (ranks_before(v, r, bv, best)) { bv = v; best = r; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, best, o);
        if (ranks_before(ov, oi, bv, best)) { bv = ov; best = oi; }
      }
      __syncwarp();
      if (lane == 0) sel[best] = -INFINITY;   // taken
      __syncwarp();
    }
    if (lane == k) my_idx = (uint32_t)best;
  }
  // weights: unbiased probabilities of the chosen ids, renormalised over all K slots
  float wk = (lane < K) ? p[my_idx] : 0.0f;
  float sum = warp_sum(wk);
  if (norm) wk = wk / sum;
  wk *= scale;
  float z = (lane < K && (int)my_idx >= E) ? wk : 0.0f;
  z = warp_sum(z);
  if (lane < K) {
    idx_out[lane] = my_idx;
    w_out[lane] = wk;
    if (idx_smem) idx_smem[lane] = my_idx;
  }
  if (lane == 0) *zsum_out = z;
}


// Register-resident variant of route_token_warp for R <= 32 * VPL: each lane holds the scores
// of router columns lane, lane + 32, ...; K rounds of a warp arg-max (same order: higher
// selection score first, lower id on a tie). Lane k < K writes slot k; lane 0 writes zsum.
template <int VPL>
__device__ void route_token_warp_reg(const float* L, const float* logit_bias,
                                     const float* corr_bias, int R, int E, int K, int scoring,
                                     int norm, float scale, const uint32_t* forced,
                                     uint32_t* idx_out, float* w_out, float* zsum_out) {
  const int lane = threadIdx.x & 31;
  float v[VPL], sel[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int r = i * 32 + lane;
    v[i] = r < R ? __ldcg(L + r) : 0.0f;
  }
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int r = i * 32 + lane;
    if (r < R) {
      if (logit_bias) v[i] += logit_bias[r];
      mx = fmaxf(mx, v[i]);
    }
  }
  const bool sig = scoring == MOE_SCORING_SIGMOID_BIAS;
  float den = 1.0f;
  if (!sig) {
    mx = warp_max(mx);
    den = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int r = i * 32 + lane;
      if (r < R) {
        v[i] = expf(v[i] - mx);
        den += v[i];
      }
    }
    den = warp_sum(den);
  }
  const bool biased = selection_biased(scoring) && corr_bias;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int r = i * 32 + lane;
    if (r < R) {
      v[i] = sig ? sigmoid_score(v[i]) : v[i] / den;
      sel[i] = v[i] + (biased ? corr_bias[r] : 0.0f);
    } else {
      sel[i] = -INFINITY;
    }
  }
  uint32_t my_idx = 0;
  float my_p = 0.0f;
  for (int k = 0; k < K; ++k) {
    int best;
    if (forced) {
      best = (int)forced[k];
    } else {
      float bv = -INFINITY;
      best = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int r = i * 32 + lane;
        if (r < R && ranks_before(sel[i], r, bv, best)) {
          bv = sel[i];
          best = r;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best, o);
        if (ranks_before(ov, oi, bv, best)) {
          bv = ov;
          best = oi;
        }
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (i * 32 + lane == best) sel[i] = -INFINITY;   // taken
    }
    float pb = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (i * 32 + lane == best) pb = v[i];
    pb = __shfl_sync(0xffffffffu, pb, best & 31);
    if (lane == k) {
      my_idx = (uint32_t)best;
      my_p = pb;
    }
  }
  // weights: unbiased probabilities of the chosen ids, renormalised over all K slots
  float wk = lane < K ? my_p : 0.0f;
  const float sum = warp_sum(wk);
  if (norm) wk = wk / sum;
  wk *= scale;
  float z = (lane < K && (int)my_idx >= E) ? wk : 0.0f;
  z = warp_sum(z);
  if (lane < K) {
    idx_out[lane] = my_idx;
    w_out[lane] = wk;
  }
  if (lane == 0) *zsum_out = z;
}

// route_token_warp_reg for any R <= 1024.
__device__ __forceinline__ void route_token_warp_fast(const float* L, const float* logit_bias,
                                                      const float* corr_bias, int R, int E, int K,
                                                      int scoring, int norm, float scale,
                                                      const uint32_t* forced, uint32_t* idx_out,
                                                      float* w_out, float* zsum_out) {
  if (R <= 128)
    route_token_warp_reg<4>(L, logit_bias, corr_bias, R, E, K, scoring, norm, scale, forced,
                            idx_out, w_out, zsum_out);
  else if (R <= 256)
    route_token_warp_reg<8>(L, logit_bias, corr_bias, R, E, K, scoring, norm, scale, forced,
                            idx_out, w_out, zsum_out);
  else if (R <= 512)
    route_token_warp_reg<16>(L, logit_bias, corr_bias, R, E, K, scoring, norm, scale, forced,
                             idx_out, w_out, zsum_out);
  else
    route_token_warp_reg<32>(L, logit_bias, corr_bias, R, E, K, scoring, norm, scale, forced,
                             idx_out, w_out, zsum_out);
}

// Block-wide exclusive scan of one value per thread (blockDim.x <= 1024, multiple of 32).
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    uint32_t t = lane < nw ? warp_tot[lane] : 0;
    uint32_t ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t n = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += n;
    }
    if (lane < nw) warp_tot[lane] = ti - t;
    if (lane == 31 && total) *total = ti;
  }
  __syncthreads();
  uint32_t r = warp_tot[wid] + inc - v;
  __syncthreads();
  return r;
}

}  // namespace
}  // namespace moe
