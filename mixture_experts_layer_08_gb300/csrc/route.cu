// Routing: router logits, softmax (+ selection-only correction bias) top-K with
// renormalisation and identity-expert fold, and the stable sort of (token, slot) pairs by
// expert.
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (`forward_prefill`: the gate
// GEMM keeps a fixed accumulation order; `moe_topk_softmax_batched` with `norm_topk_prob`;
// `moe_sort_by_expert` writes sorted ids, expert offsets [E+1] and token_to_perm [te]),
// "spark_model/layers/moe/forward.rs" (`forward`: softmax scores + correction bias for
// selection, unbiased softmax x scaling for the weights, selected identity experts folded
// into zero_accum; the single-CTA fused gate+top-K was too slow for 256 experts, so here
// routing is one warp per token and the router spreads its columns over many blocks).
#include <cuda_fp16.h>

#include "kernels.h"
#include "route_dev.cuh"

namespace moe {

namespace {

// ------------------------------------------------------------------ small-N router

constexpr int kRouterWarps = 4;      // router columns per block (one per warp)
constexpr int kRouterTok = 16;       // most tokens per block

// Stable sort of te <= 1024 * k pairs inside one block (used by the fused decode tail).
// idx_s: the pair expert ids in shared memory.
__device__ void sort_in_block(const uint32_t* idx_s, int te, int E, int K, uint32_t* cnt_s,
                              uint32_t* scan_s, const SortArgs& s) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < te; j += blockDim.x) {
    uint32_t e = idx_s[j];
    if ((int)e < E) atomicAdd(&cnt_s[e], 1u);
  }
  __syncthreads();
  // exclusive scans of counts (row offsets) and of the "has rows" flags (active list),
  // E <= 1024 handled in chunks of blockDim
  uint32_t run_off = 0, run_act = 0;
  for (int base = 0; base < E; base += blockDim.x) {
    int e = base + threadIdx.x;
    uint32_t c = e < E ? cnt_s[e] : 0;
    uint32_t tot_c, tot_a;
    uint32_t off = block_excl_scan(c, scan_s, &scan_s[32]);
    tot_c = scan_s[32];
    __syncthreads();
    uint32_t act = block_excl_scan(c > 0 ? 1u : 0u, scan_s, &scan_s[32]);
    tot_a = scan_s[32];
    __syncthreads();
    if (e < E) {
      s.offsets[e] = run_off + off;
      if (c > 0) s.active[run_act + act] = (uint32_t)e;
      cnt_s[e] = run_off + off;     // becomes the row base of expert e
    }
    run_off += tot_c;
    run_act += tot_a;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    s.offsets[E] = run_off;
    s.hdr->num_active = run_act;
  }
  __syncthreads();
  // rank of each pair among the earlier pairs of its expert (stable in the pair index)
  for (int j = threadIdx.x; j < te; j += blockDim.x) {
    uint32_t e = idx_s[j];
    if ((int)e >= E) {
      s.pair_to_row[j] = kNoRow;
      continue;
    }
    uint32_t rank = 0;
    for (int i = 0; i < j; ++i) rank += (idx_s[i] == e) ? 1u : 0u;
    uint32_t row = cnt_s[e] + rank;
    s.pair_to_row[j] = row;
    s.sorted_pairs[row] = (uint32_t)j;
  }
}

// NT: tokens per block (a power of two >= the block's token count, <= 16).
template <int NT>
__global__ void __launch_bounds__(32 * kRouterWarps) router_small_kernel(RouteArgs a, SortArgs s,
                                                                         int fuse_tail) {
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);     // [tok, H]
  pdl_trigger();    // the next kernel may launch now and wait for this one's results
  const int H = a.H, R = a.R;
  const int tok0 = blockIdx.y * NT;
  const int ntok = min(NT, a.N - tok0);
  // stage the block's tokens in shared memory (16-byte chunks)
  const int chunks = H / 8;
  for (int i = threadIdx.x; i < ntok * chunks; i += blockDim.x) {
    int t = i / chunks, c = i % chunks;
    reinterpret_cast<uint4*>(xs)[t * chunks + c] =
        reinterpret_cast<const uint4*>(a.x + (size_t)(tok0 + t) * H)[c];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int r = blockIdx.x * kRouterWarps + wid;
  if (r < R) {
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    const uint4* wrow = reinterpret_cast<const uint4*>(a.router_w + (size_t)r * H);
    for (int c0 = 0; c0 < chunks; c0 += 256) {
      uint4 wv[8];            // all of this lane's loads in flight before any arithmetic
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = c0 + q * 32 + lane;
        if (c < chunks) wv[q] = __ldg(wrow + c);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = c0 + q * 32 + lane;
        if (c < chunks) {
          float wf[8];
          bf16x8_to_f32(wv[q], wf);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            // rows past ntok repeat the block's first token (computed, never stored)
            float xf[8];
            bf16x8_to_f32(reinterpret_cast<const uint4*>(xs)[(t < ntok ? t : 0) * chunks + c], xf);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[t] = fmaf(wf[i], xf[i], acc[t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float v = warp_sum(acc[t]);
      if (lane == 0 && t < ntok) a.logits[(size_t)(tok0 + t) * R + r] = v;
    }
  }
  if (!fuse_tail) return;
  // ---- last block to finish: top-K of every token and the stable sort (N <= 16)
  __shared__ uint32_t is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t prev = atomicAdd(&a.hdr->done_blocks, 1u);
    is_last = (prev == gridDim.x * gridDim.y - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  float* pbuf = reinterpret_cast<float*>(smem);                   // [8 warps][R] probs
  float* sbuf = pbuf + kRouterWarps * R;                          // [8 warps][R] scores
  uint32_t* idx_s = reinterpret_cast<uint32_t*>(sbuf + kRouterWarps * R);   // [te]
  uint32_t* cnt_s = idx_s + a.N * a.K;                            // [E]
  uint32_t* scan_s = cnt_s + a.E;                                 // [33]
  for (int t = wid; t < a.N; t += kRouterWarps) {
    route_token_warp(a.logits + (size_t)t * R, a.logit_bias, a.corr_bias, R, a.E, a.K,
                     a.scoring, a.norm, a.scale, a.forced ? a.forced + (size_t)t * a.K : nullptr,
                     pbuf + wid * R, sbuf + wid * R, a.idx + (size_t)t * a.K,
                     a.w + (size_t)t * a.K, a.zsum + t, idx_s + t * a.K);
  }
  __syncthreads();
  sort_in_block(idx_s, a.N * a.K, a.E, a.K, cnt_s, scan_s, s);
  if (threadIdx.x == 0) a.hdr->done_blocks = 0;
}

// One warp per token (with thousands of tokens in flight the shared-memory version keeps up
// better than the register-resident ones, which win only for a lone warp).
__global__ void __launch_bounds__(256) topk_kernel(RouteArgs a) {
  extern __shared__ __align__(16) float sm[];
  const int wid = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + wid;
  if (t >= a.N) return;
  float* p = sm + wid * 2 * a.R;
  route_token_warp(a.logits + (size_t)t * a.R, a.logit_bias, a.corr_bias, a.R, a.E, a.K,
                   a.scoring, a.norm, a.scale, a.forced ? a.forced + (size_t)t * a.K : nullptr,
                   p, p + a.R, a.idx + (size_t)t * a.K, a.w + (size_t)t * a.K, a.zsum + t,
                   nullptr);
}

// ------------------------------------------------------------------ large-N sort

constexpr int kSortBlock = 1024;

// Per block of 1024 pairs: per-expert counts and each pair's rank among the block's earlier
// pairs of the same expert.
__global__ void __launch_bounds__(kSortBlock) sort_count_kernel(SortArgs s) {
  pdl_wait();   // the routing (or count) results
  extern __shared__ uint32_t wcnt[];                 // [32 warps][E]
  const int E = s.E;
  const int j = blockIdx.x * kSortBlock + threadIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * E; i += kSortBlock) wcnt[i] = 0;
  __syncthreads();
  uint32_t e = j < s.te ? s.idx[j] : kNoRow;
  bool real = e != kNoRow && e < (uint32_t)E;
  uint32_t key = real ? e : kNoRow;
  uint32_t peers = __match_any_sync(0xffffffffu, key);
  uint32_t lt = (1u << lane) - 1u;
  uint32_t rank_w = __popc(peers & lt);
  if (real && rank_w == 0) wcnt[wid * E + e] = __popc(peers);
  __syncthreads();
  for (int ex = threadIdx.x; ex < E; ex += kSortBlock) {
    uint32_t run = 0;
    for (int w = 0; w < 32; ++w) {
      uint32_t c = wcnt[w * E + ex];
      wcnt[w * E + ex] = run;
      run += c;
    }
    s.blk_counts[(size_t)blockIdx.x * E + ex] = run;
  }
  __syncthreads();
  if (j < s.te) s.local_rank[j] = real ? wcnt[wid * E + e] + rank_w : kNoRow;
}

// Number of the n one-tile slots that sit before position p of a list of T m-tiles, the j-th
// one-tile slot being at floor((2j + 1) * T / (2n)) (n <= T, so the slots are distinct).
__device__ __forceinline__ uint32_t slots_before(uint32_t p, uint32_t n, uint32_t T) {
  const uint64_t a = 2ull * n * p;
  if (a <= T) return 0;
  const uint64_t l = (a + T - 1) / (2ull * T);
  return l < n ? (uint32_t)l : n;
}

// Expert offsets, active experts, per-block row starts and the m-tile list. The list puts the
// m-tiles of the experts with a single m-tile (whose weights are read from HBM for that one
// tile) evenly among the m-tiles of the others (kept consecutive per expert, so their weight
// tiles are reused from L2), so that every wave of the persistent GEMMs mixes HBM-bound and
// tensor-bound tiles instead of meeting long runs of one kind.
__global__ void __launch_bounds__(1024) sort_scan_kernel(SortArgs s, int nblk) {
  pdl_wait();   // the counts
  __shared__ uint32_t scan_s[40];
  const int E = s.E;
  int4* heavy = s.tiles_tmp;                   // m-tiles of experts with two or more
  int4* single = s.tiles_tmp + s.max_mtiles;   // the one m-tile of each other expert
  uint32_t run_off = 0, run_act = 0, run_heavy = 0, run_single = 0;
  for (int base = 0; base < E; base += blockDim.x) {
    int e = base + threadIdx.x;
    uint32_t c = 0;
    if (e < E)
      for (int b = 0; b < nblk; ++b) c += s.blk_counts[(size_t)b * E + e];
    uint32_t off = block_excl_scan(c, scan_s, &scan_s[32]);
    uint32_t tot_c = scan_s[32];
    __syncthreads();
    uint32_t act = block_excl_scan(c > 0 ? 1u : 0u, scan_s, &scan_s[32]);
    uint32_t tot_a = scan_s[32];
    __syncthreads();
    const uint32_t nt = (c + 127) / 128;
    uint32_t hstart = block_excl_scan(nt > 1 ? nt : 0u, scan_s, &scan_s[32]);
    uint32_t tot_h = scan_s[32];
    __syncthreads();
    uint32_t sidx = block_excl_scan(nt == 1 ? 1u : 0u, scan_s, &scan_s[32]);
    uint32_t tot_s = scan_s[32];
    __syncthreads();
    if (e < E) {
      uint32_t o = run_off + off;
      s.offsets[e] = o;
      if (c > 0) s.active[run_act + act] = (uint32_t)e;
      uint32_t r = o;
      for (int b = 0; b < nblk; ++b) {
        uint32_t cb = s.blk_counts[(size_t)b * E + e];
        s.blk_counts[(size_t)b * E + e] = r;
        r += cb;
      }
      if (nt == 1) {
        single[run_single + sidx] = make_int4(e, (int)o, (int)(o + c), 0);
      } else {
        for (uint32_t i = 0; i < nt; ++i) {
          uint32_t r0 = o + 128 * i;
          uint32_t r1 = min(o + c, r0 + 128);
          heavy[run_heavy + hstart + i] = make_int4(e, (int)r0, (int)r1, 0);
        }
      }
    }
    run_off += tot_c;
    run_act += tot_a;
    run_heavy += tot_h;
    run_single += tot_s;
    __syncthreads();
  }
  // merge: position p holds one-tile slot j = slots_before(p) if the next position has one
  // more slot before it, else the (p - slots_before(p))-th m-tile of the others
  const uint32_t T = run_heavy + run_single;
  for (uint32_t p = threadIdx.x; p < T; p += blockDim.x) {
    const uint32_t lp = slots_before(p, run_single, T);
    const uint32_t lq = slots_before(p + 1, run_single, T);
    s.tiles[p] = lq > lp ? single[lp] : heavy[p - lp];
  }
  if (threadIdx.x == 0) {
    s.offsets[E] = run_off;
    s.hdr->num_active = run_act;
    s.hdr->num_mtiles = T;
  }
}

// One warp per pair: final row, inverse map, and the gathered (or quantised) x row.
__global__ void __launch_bounds__(256) sort_scatter_kernel(SortArgs s, const __nv_bfloat16* x,
                                                           int H, __nv_bfloat16* xp,
                                                           uint8_t* xq, float* xsc) {
  pdl_wait();   // the counts and offsets
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (j >= s.te) return;
  uint32_t e = s.idx[j];
  if ((int)e >= s.E) {
    if (lane == 0) s.pair_to_row[j] = kNoRow;
    return;
  }
  uint32_t row = s.blk_counts[(size_t)(j / kSortBlock) * s.E + e] + s.local_rank[j];
  const int t = j / s.K;
  if (lane == 0) {
    s.pair_to_row[j] = row;
    s.sorted_pairs[row] = (uint32_t)j;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  if (xp) {
    // all of this lane's loads in flight before the stores; the copy is read once, by the
    // GEMM, so it is written evict-first
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)row * H);
    for (int c0 = 0; c0 < H / 8; c0 += 8 * 32) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < H / 8) v[u] = __ldg(src + c);
      }
      if (s.xp_f16) {
        // the NVFP4 experts' f16 MMA operand: bf16 -> f16 (exact in f16's normal range)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t* w = reinterpret_cast<uint32_t*>(&v[u]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[q]);
            const __half2 h = __floats2half2_rn(__low2float(b), __high2float(b));
            w[q] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < H / 8) __stcs(dst + c, v[u]);
      }
    }
  }
  if (xq) {
    // E4M3 codes and 1x128 scales of the token row (quantised once per token)
    const uint4* qsrc = reinterpret_cast<const uint4*>(s.xq_tok + (size_t)t * H);
    uint4* qdst = reinterpret_cast<uint4*>(xq + (size_t)row * H);
    for (int c0 = 0; c0 < H / 16; c0 += 8 * 32) {
      uint4 v[8];   // loads in flight before the stores; the copy is read once
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < H / 16) v[u] = __ldg(qsrc + c);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < H / 16) __stcs(qdst + c, v[u]);
      }
    }
    for (int g = lane; g < H / 128; g += 32)
      xsc[(size_t)g * s.te + row] = s.xs_tok[(size_t)g * s.N + t];
  }
}

// Pre-expert RMSNorm ("metrale_model_layers/layers/moe/forward_prefill.rs",
// `pre_expert_norm`): one warp per token row; the sum of squares in fp32 (loads in flight four
// at a time), then xn = bf16(x * g * (1 / sqrt(mean + eps))).
__global__ void __launch_bounds__(256) rms_norm_rows_kernel(const __nv_bfloat16* x,
                                                            const __nv_bfloat16* g, float eps,
                                                            int N, int H, __nv_bfloat16* xn) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= N) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const uint4* gs = reinterpret_cast<const uint4*>(g);
  uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)t * H);
  const int C = H / 8;
  float ss = 0.0f;
  for (int c0 = 0; c0 < C; c0 += 4 * 32) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * 32 + lane;
      v[u] = c < C ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float f[8];
      bf16x8_to_f32(v[u], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
  }
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / (float)H + eps);
  for (int c = lane; c < C; c += 32) {
    float f[8], w[8];
    bf16x8_to_f32(__ldg(src + c), f);
    bf16x8_to_f32(__ldg(gs + c), w);
    uint4 o;
    o.x = pack_bf16x2(f[0] * w[0] * inv, f[1] * w[1] * inv);
    o.y = pack_bf16x2(f[2] * w[2] * inv, f[3] * w[3] * inv);
    o.z = pack_bf16x2(f[4] * w[4] * inv, f[5] * w[5] * inv);
    o.w = pack_bf16x2(f[6] * w[6] * inv, f[7] * w[7] * inv);
    dst[c] = o;
  }
}

// One warp per token row: per 1x128 group, amax, scale = amax/448 (1 if 0) and the E4M3
// code of value/scale (round to nearest even, saturating), all decided in fp32.
// Codes [N, H]; scales [H/128, N].
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* x, int N, int H,
                                                         uint8_t* q, float* sc) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= N) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  for (int c4 = 0; c4 < H / 8; c4 += 4 * 32) {
    uint4 raw[4];   // four loads in flight before the first group is quantised
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c4 + u * 32 + lane;
      raw[u] = c < H / 8 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (c4 + u * 32 >= H / 8) break;   // (warp-uniform)
      const int c = c4 + u * 32 + lane;
      const bool on = c < H / 8;
      float f[8];
      bf16x8_to_f32(raw[u], f);
      float am = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      const float s = am > 0.0f ? __fdiv_rn(am, 448.0f) : 1.0f;
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        lo |= (uint32_t)__nv_cvt_float2_to_fp8x2(
                  make_float2(__fdiv_rn(f[i], s), __fdiv_rn(f[i + 1], s)), __NV_SATFINITE,
                  __NV_E4M3) << (8 * i);
        hi |= (uint32_t)__nv_cvt_float2_to_fp8x2(
                  make_float2(__fdiv_rn(f[4 + i], s), __fdiv_rn(f[5 + i], s)), __NV_SATFINITE,
                  __NV_E4M3) << (8 * i);
      }
      if (on) {
        reinterpret_cast<uint2*>(q + (size_t)t * H)[c] = make_uint2(lo, hi);
        if ((lane & 15) == 0) sc[(size_t)(c / 16) * N + t] = s;
      }
    }
  }
}

}  // namespace

cudaError_t launch_rms_norm_rows(const __nv_bfloat16* x, const __nv_bfloat16* g, float eps, int N,
                                 int H, __nv_bfloat16* xn, cudaStream_t st) {
  rms_norm_rows_kernel<<<(N + 7) / 8, 256, 0, st>>>(x, g, eps, N, H, xn);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const __nv_bfloat16* x, int N, int H, uint8_t* q, float* sc,
                              cudaStream_t st) {
  quant_rows_kernel<<<(N + 7) / 8, 256, 0, st>>>(x, N, H, q, sc);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_router_small_t(const RouteArgs& a, const SortArgs& s, bool fuse_tail,
                                  cudaStream_t st) {
  dim3 grid((a.R + kRouterWarps - 1) / kRouterWarps, (a.N + NT - 1) / NT);
  size_t sm_x = (size_t)NT * a.H * 2;
  size_t sm_tail = fuse_tail ? (size_t)2 * kRouterWarps * a.R * 4 + (size_t)a.N * a.K * 4 +
                                   (size_t)a.E * 4 + 40 * 4
                             : 0;
  size_t sm = sm_x > sm_tail ? sm_x : sm_tail;
  if (sm > 32 * 1024) {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(router_small_kernel<NT>), sm);
    if (e != cudaSuccess) return e;
  }
  router_small_kernel<NT><<<grid, 32 * kRouterWarps, sm, st>>>(a, s, fuse_tail ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_router_small(const RouteArgs& a, const SortArgs& s, bool fuse_tail,
                                cudaStream_t st) {
  if (fuse_tail && a.N > kRouterTok) return cudaErrorInvalidValue;
  if (a.N <= 1) return launch_router_small_t<1>(a, s, fuse_tail, st);
  if (a.N <= 2) return launch_router_small_t<2>(a, s, fuse_tail, st);
  if (a.N <= 4) return launch_router_small_t<4>(a, s, fuse_tail, st);
  if (a.N <= 8) return launch_router_small_t<8>(a, s, fuse_tail, st);
  return launch_router_small_t<16>(a, s, fuse_tail, st);
}

cudaError_t launch_topk(const RouteArgs& a, cudaStream_t st) {
  size_t sm = (size_t)8 * 2 * a.R * 4;
  if (sm > 32 * 1024) {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(topk_kernel), sm);
    if (e != cudaSuccess) return e;
  }
  topk_kernel<<<(a.N + 7) / 8, 256, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sort(const SortArgs& s, const __nv_bfloat16* x, int H, __nv_bfloat16* xp,
                        uint8_t* xq, float* xs, cudaStream_t st) {
  const int nblk = (s.te + kSortBlock - 1) / kSortBlock;
  size_t sm = (size_t)32 * s.E * 4;
  if (sm > 32 * 1024) {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(sort_count_kernel), sm);
    if (e != cudaSuccess) return e;
  }
  // programmatic dependents: each kernel launches as its predecessor drains and waits for
  // its results (pdl_wait) before reading them
  cudaError_t e = launch_dependent(sort_count_kernel, dim3(nblk), dim3(kSortBlock), sm, st, s);
  if (e != cudaSuccess) return e;
  e = launch_dependent(sort_scan_kernel, dim3(1), dim3(1024), 0, st, s, nblk);
  if (e != cudaSuccess) return e;
  e = launch_dependent(sort_scatter_kernel, dim3((s.te + 7) / 8), dim3(256), 0, st, s, x, H, xp,
                       xq, xs);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
