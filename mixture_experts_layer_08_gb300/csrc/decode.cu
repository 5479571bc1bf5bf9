// Decode chain (few tokens): the whole block forward in one persistent, cooperatively launched
// kernel -- router, top-K and sort, the expert projections as skinny GEMMs on the
// 5th-generation tensor cores, and the weighted combine -- streaming the weights of every
// expert the batch touches from HBM once, for all the tokens routed to it. The shared expert
// is one more slot.
//
// Pages: "spark_model/layers/moe/forward.rs" (`forward`: gate GEMM, softmax + correction-bias
// top-K, fused gate/up projection for the K routed experts plus the shared expert, fused SiLU
// and down projection, weighted sum + sigmoid-gated shared blend + identity-expert add, all on
// device with no host synchronisation; the single-CTA fused gate+top-K it rejects is replaced
// by router rows spread over every block and a per-block top-K) and
// "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (few-row decode: routed down
// projections weighted and FP32-atomic-added into an [N,H] accumulator zeroed first, then a
// finalize that casts to BF16 and blends the shared expert).
//
// Phases, separated by two grid barriers (all blocks are resident: a bounded spin on a
// counter in the workspace header):
//   0  router logits: one router row per block (the contraction over all its threads), rows
//      spread over the blocks; with a pre-expert norm, blocks past the router rows write the
//      routed experts' input xn = RMSNorm(x);
//   1  every block routes the whole batch into its own shared memory (softmax or sigmoid
//      scores, top-K, renormalisation, identity-expert sums, shared-expert gate, stable sort
//      by expert); block 0 also writes the routing to the workspace. With at most 32 routed
//      pairs (and a router up to 256 wide) this phase stops once the experts in use are
//      known, and the epilogue warps finish the sort and the weights during phase 2;
//   2  gate/up then down projections (below);
//   3  out[t] = bf16(sum_k w * y[row(t,k)] (or the atomic accumulator) + zsum * x + gamma * Sh),
//      output chunks spread over the blocks.
//
// Shape of the work. The weights are the wide B operand: a tile is BN (256, or 128 when a
// dimension is not a multiple of 256) rows of one projection of one slot, so every MMA reads
// its weights at the full-rate N. The batch is the A operand (M = 128): rows 0..15 hold the
// tokens (x -- or xn for routed experts under a pre-expert norm -- for gate/up,
// SiLU(gate)*up of the slot's tokens for down), rows 16..127 read
// whatever shared memory follows and only produce accumulator rows that are never read. A
// work item is one tile times one 64-column swizzle box of its contraction (BN x 128 bytes).
// Items are numbered slot-major; every block takes a contiguous, balanced range of the gate/up
// items and then of the down items, so a block's consecutive items of one tile form a run
// that accumulates in TMEM. The grid of each phase is capped so that no tile is split over
// more than two blocks: the two fp32 partial sums then meet in a zeroed buffer through atomic
// adds, and a + b == b + a makes the result independent of their order.
//
// Roles (192 threads, one block per SM, all blocks resident):
//   warp 0     TMA producer: per item one BN x 64 weight box (+ one 16 x 64 box of x on
//              gate/up) into a ring of stages.
//   warp 1     allocates all 512 TMEM columns (two accumulators of up to 256 columns); one
//              lane issues tcgen05.mma (M=128, N=BN, K=16) x 4 per item and commits stage
//              releases and finished runs.
//   warps 2-5  epilogue. Warp 4 (TMEM lanes 0..31 = the token rows) drains a finished run:
//              fp32 atomic adds of each token's row into the gate/up buffer (then one count
//              per run for the slot) or into the down output. Before the first down run of a
//              slot, all four wait for the slot's gate/up count (other blocks; bounded spin)
//              and build SiLU(gate)*up of its tokens as the bf16 A operand (128-byte swizzle).
#include <mutex>
#include <set>

#include "kernels.h"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kThreads = 192;             // block size (NVFP4 experts: + kConvWarps warps)
constexpr int kConvBase = 192;            // warps 6-9: NVFP4 converters
constexpr int kConvWarps = 4;
constexpr int kMaxWarps = (kThreads + 32 * kConvWarps) / 32;
constexpr int kBox = 64;                  // contraction columns per item (one 128-byte row)
constexpr int kMaxBN = 256;
constexpr int kWBytes = kMaxBN * 128;     // weight box of a stage, 32 KB
constexpr int kCodeBytes = kMaxBN * 48;   // NVFP4: codes (32 B) + scale codes (16 B) per row
constexpr int kTokBytes = 16 * 128;       // token rows of one contraction box, 2 KB
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 512;            // two accumulators of up to 256 columns
constexpr int kEpiThreads = 128;
constexpr int kDrainWarp = 4;             // warp % 4 == 0: TMEM lanes 0..31
constexpr int kStageLd = 68;              // drain staging row stride (floats; 16-byte rows)
constexpr int kRaccLd = 260;              // E4M3 runs: fp32 run accumulator row stride (floats)
constexpr int kRaccBytes = 16 * kRaccLd * 4;
constexpr int kMaxHGroups = 8;            // 1x128 groups of a routed intermediate row (I <= 1024)
constexpr int kSmemLimit = 227 * 1024;

struct Plan {
  int stages;
  int bn_g, bn_d;   // weight rows per tile: gate/up, down
  int hbytes;       // down-projection A operand: boxes of 16 rows x 128 bytes (max(I, S) / 64;
                    // E4M3 routed experts: max(I / 128, S / 64))
};

constexpr uint16_t kNoRow16 = 0xFFFF;

// This launch's block size (kThreads, or kThreads + 32 * kConvWarps with NVFP4 experts).
__device__ __forceinline__ int nthr() { return (int)blockDim.x; }
__device__ __forceinline__ int nwarps() { return (int)(blockDim.x >> 5); }

// Routing of the batch; every block computes its own copy in shared memory.
struct Routing {
  int n_active;                          // active (expert, rows) slots
  int rows;                              // routed rows (pairs on real experts)
  uint16_t slot_e[kDecodeMaxPairs];      // expert of each active slot
  uint16_t slot_r0[kDecodeMaxPairs];     // its first sorted row
  uint16_t slot_n[kDecodeMaxPairs];      // its row count
  uint16_t row_tok[kDecodeMaxPairs];     // token of each sorted row
  uint16_t row_pair[kDecodeMaxPairs];    // (token, slot) pair of each sorted row
  uint16_t pair_row[kDecodeMaxPairs];    // sorted row of each pair, kNoRow16: identity expert
  float w[kDecodeMaxPairs];              // routing weight of each pair
  float zsum[kDecodeMaxTokens];          // identity-expert weight sum of each token
  float gamma[kDecodeMaxTokens];         // shared-expert blend weight of each token
  uint16_t idx[32];                      // chosen router column of each pair (split routing)
  uint32_t bits[32];                     // experts in use, one bit each (split routing)
};

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Adds `v` to a global counter after every write this thread has made or seen ordered before
// (a release: acq_rel fence, then a relaxed reduction).
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}

// Grid-wide barrier of the co-resident blocks: the header counter reaches `target` (the number
// of blocks times the barriers passed so far). Bounded: a timeout is reported and the block
// carries on (its results are then not used).
__device__ void grid_barrier(WsHeader* hdr, uint32_t target) {
  __syncthreads();
  if (threadIdx.x == 0) {
    red_release_add(&hdr->done_blocks, 1u);   // (the block's writes, ordered before by the barrier)
    if (ld_acquire(&hdr->done_blocks) < target) {
      const long long t0 = clock64();
      while (ld_acquire(&hdr->done_blocks) < target) {
        if (clock64() - t0 > kSpinLimitCycles) {
          report_timeout(hdr);
          break;
        }
      }
    }
  }
  __syncthreads();
}

// Phase 0: logits[t, r] = x[t] . Wr[r] for every token, and the shared-gate products
// x[t] . g (the gate vector as one more row, R), one row per block at a time with the
// contraction spread over all its threads. x (and g) are staged in shared memory when they fit
// (`scratch`), else read from global memory; the block's first row is loaded before the
// staging so the two latencies overlap.
__device__ void router_rows(const DecodeArgs& a, uint8_t* scratch, size_t scratch_bytes,
                            float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunks = a.H / 8;
  const bool gated = a.S > 0 && a.sh_gate_vec;
  const int rows = a.R + (gated ? 1 : 0);
  auto row_ptr = [&](int r) {
    return reinterpret_cast<const uint4*>(r < a.R ? a.router_w + (size_t)r * a.H : a.sh_gate_vec);
  };
  constexpr int kPer = 8;   // chunks per thread per pass (H <= 8 * 8 * nthr())
  uint4 wv[kPer];
  const int r_first = blockIdx.x;
  if (r_first < rows) {
    const uint4* wr = row_ptr(r_first);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int c = q * nthr() + tid;
      if (c < chunks) wv[q] = __ldg(wr + c);
    }
  }
  const size_t xbytes = (size_t)a.N * a.H * 2;
  const __nv_bfloat16* xs = a.x;
  if (xbytes <= scratch_bytes) {
    uint4* d = reinterpret_cast<uint4*>(scratch);
    const uint4* sx = reinterpret_cast<const uint4*>(a.x);
    const int n = (int)(xbytes / 16);
    for (int i0 = 0; i0 < n; i0 += 8 * nthr()) {
      uint4 tmp[8];   // eight loads in flight per thread
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * nthr() + tid;
        if (i < n) tmp[u] = __ldg(sx + i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * nthr() + tid;
        if (i < n) d[i] = tmp[u];
      }
    }
    __syncthreads();
    xs = reinterpret_cast<const __nv_bfloat16*>(scratch);
  }
  for (int r = r_first; r < rows; r += gridDim.x) {
    const uint4* wr = row_ptr(r);
    for (int c0 = 0; c0 < chunks; c0 += kPer * nthr()) {
      if (r != r_first || c0 != 0) {   // (the first pass was loaded above)
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const int c = c0 + q * nthr() + tid;
          if (c < chunks) wv[q] = __ldg(wr + c);
        }
      }
      // tokens in a rolled loop (run-once code: its size costs more than the loop), the
      // warps' partial sums of each token accumulated in shared memory
#pragma unroll 1
      for (int t = 0; t < a.N; ++t) {
        const uint4* xt = reinterpret_cast<const uint4*>(xs + (size_t)t * a.H);
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const int c = c0 + q * nthr() + tid;
          if (c < chunks) {
            float wf[8], xf[8];
            bf16x8_to_f32(wv[q], wf);
            bf16x8_to_f32(xt[c], xf);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], xf[i], acc);
          }
        }
        acc = warp_sum(acc);
        if (lane == 0) red[t * nwarps() + warp] = (c0 == 0 ? 0.0f : red[t * nwarps() + warp]) + acc;
      }
    }
    __syncthreads();
    if (tid < a.N) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < nwarps(); ++w) v += red[tid * nwarps() + w];
      if (r < a.R) a.logits[(size_t)tid * a.R + r] = v;
      else a.hdr->gate_dot[tid] = v;
    }
    __syncthreads();
  }
}

// Phase 0, with a pre-expert norm: xn[t] = bf16(x[t] * g / sqrt(mean(x[t]^2) + eps)), token t
// by block G-1-t (the blocks past the router rows are otherwise idle in this phase), from the
// staged x rows `xs`. The routed experts' gate/up items stream xn by TMA after the grid
// barrier, so the writes are fenced for the async proxy first.
__device__ void pre_expert_norm_rows(const DecodeArgs& a, const __nv_bfloat16* xs, float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = a.H / 8;
  bool wrote = false;
  for (int t = (int)gridDim.x - 1 - (int)blockIdx.x; t >= 0 && t < a.N; t += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(xs + (size_t)t * a.H);
    float ss = 0.0f;
#pragma unroll 1
    for (int c = tid; c < C; c += nthr()) {
      float f[8];
      bf16x8_to_f32(xr[c], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < nwarps(); ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)a.H + a.eps);
    const uint4* gs = reinterpret_cast<const uint4*>(a.norm_w);
    uint4* dst = reinterpret_cast<uint4*>(a.xn + (size_t)t * a.H);
#pragma unroll 1
    for (int c = tid; c < C; c += nthr()) {
      float f[8], w[8];
      bf16x8_to_f32(xr[c], f);
      bf16x8_to_f32(__ldg(gs + c), w);
      uint4 o;
      o.x = pack_bf16x2(f[0] * w[0] * inv, f[1] * w[1] * inv);
      o.y = pack_bf16x2(f[2] * w[2] * inv, f[3] * w[3] * inv);
      o.z = pack_bf16x2(f[4] * w[4] * inv, f[5] * w[5] * inv);
      o.w = pack_bf16x2(f[6] * w[6] * inv, f[7] * w[7] * inv);
      dst[c] = o;
    }
    wrote = true;
    __syncthreads();   // (red is reused)
  }
  if (wrote) asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Phase 0 with E4M3 routed experts: their input rows (x, or xn under a pre-expert norm) as
// E4M3 codes xq [N, H] with one scale per 1x128 group, xs [H/128, N]: scale = amax / 448 (1 if
// the group is zero), code = value / scale rounded to nearest even, saturating, all decided in
// fp32 (the rule of the grouped chain's quantiser). Token t by block G-1-t, one warp per group.
// The routed gate/up items stream xq by TMA after the grid barrier: fenced for the async proxy.
__device__ void quant_token_rows(const DecodeArgs& a, const __nv_bfloat16* src) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = (int)gridDim.x - 1 - (int)blockIdx.x;
  if (t < 0 || t >= a.N) return;
  const int G = a.H / 128;
  for (int g = warp; g < G; g += nwarps()) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + (size_t)t * a.H + g * 128 + lane * 4);
    float f[4];
    f[0] = __uint_as_float(raw.x << 16);
    f[1] = __uint_as_float(raw.x & 0xffff0000u);
    f[2] = __uint_as_float(raw.y << 16);
    f[3] = __uint_as_float(raw.y & 0xffff0000u);
    const float am = warp_max(fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
    const float sc = am > 0.0f ? __fdiv_rn(am, 448.0f) : 1.0f;
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(f[0], sc), __fdiv_rn(f[1], sc)), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(f[2], sc), __fdiv_rn(f[3], sc)), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<uint32_t*>(a.xq + (size_t)t * a.H + g * 128 + lane * 4) = lo | (hi << 16);
    if (lane == 0) a.xs[(size_t)g * a.N + t] = sc;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Phase 0 with NVFP4 routed experts: their input rows (x, or xn under a pre-expert norm) as
// f16 (exact for bf16 values in f16's normal range), the A operand of the routed f16 MMAs.
// Token t by block G-1-t; fenced for the TMA reads of phase 2.
__device__ void half_token_rows(const DecodeArgs& a, const __nv_bfloat16* src) {
  const int t = (int)gridDim.x - 1 - (int)blockIdx.x;
  if (t < 0 || t >= a.N) return;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)t * a.H);
  uint4* d4 = reinterpret_cast<uint4*>(a.xh + (size_t)t * a.H);
  for (int c = threadIdx.x; c < a.H / 8; c += nthr()) {
    uint4 v = s4[c];
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[q]);
      const __half2 h = __floats2half2_rn(__low2float(b), __high2float(b));
      w[q] = *reinterpret_cast<const uint32_t*>(&h);
    }
    d4[c] = v;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wide routers (R > 256): K rounds of a warp arg-max (route_token_warp_reg), then the same
// weights and blend gate.
__device__ void topk_rounds_warp(const DecodeArgs& a, int t, uint32_t* idx_s, Routing& rt) {
  const int lane = threadIdx.x & 31;
  route_token_warp_fast(a.logits + (size_t)t * a.R, a.logit_bias, a.corr_bias, a.R, a.E, a.K,
                        a.scoring, a.norm, a.scale,
                        a.forced ? a.forced + (size_t)t * a.K : nullptr, idx_s + t * a.K,
                        rt.w + t * a.K, rt.zsum + t);
  if (lane == 0) {
    const bool gated = a.S > 0 && a.sh_gate_vec;
    rt.gamma[t] = gated ? 1.0f / (1.0f + expf(-__ldcg(&a.hdr->gate_dot[t]))) : 1.0f;
  }
}

// Top-K of one token by one warp (R <= 32 * VPL). Lane l owns router columns l, l + 32, ...:
// softmax or sigmoid scores (into p_t[R], kept for the weights), selection score = score
// (+ the correction bias). Each score becomes a 64-bit key (order-preserving score bits above
// the complemented column id), so one unsigned compare orders by higher score, then lower id.
// Every lane sorts its VPL keys in registers; then K rounds of a warp max over the lanes' heads,
// the winning lane dropping its head. Also the shared-expert blend weight. This code runs once
// per launch with a cold instruction cache, where every instruction costs a fetch: the loops
// after the loads stay rolled over shared scratch (`p_t`, `cb_t`: R floats; `key_t`: R keys).
template <int VPL>
__device__ void token_topk(const DecodeArgs& a, int t, float* p_t, float* cb_t,
                           unsigned long long* key_t, uint32_t* idx_t, Routing& rt) {
  const int lane = threadIdx.x & 31;
  const int R = a.R;
  const float* L = a.logits + (size_t)t * R;
  const bool gated = a.S > 0 && a.sh_gate_vec;
  const bool biased = selection_biased(a.scoring) && a.corr_bias;
  const bool sig = a.scoring == MOE_SCORING_SIGMOID_BIAS;
  const float gd = gated ? __ldcg(&a.hdr->gate_dot[t]) : 0.0f;
  float v[VPL], cb[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {   // every load in flight at once
    const int r = i * 32 + lane;
    v[i] = r < R ? __ldcg(L + r) : 0.0f;
    cb[i] = (biased && r < R) ? a.corr_bias[r] : 0.0f;
    if (a.logit_bias && r < R) v[i] += a.logit_bias[r];
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int r = i * 32 + lane;
    if (r < R) {
      p_t[r] = v[i];
      cb_t[r] = cb[i];
    }
  }
  float den = 1.0f;
  if (!sig) {
    float mx = -INFINITY;
#pragma unroll 1
    for (int r = lane; r < R; r += 32) mx = fmaxf(mx, p_t[r]);
    mx = warp_max(mx);
    den = 0.0f;
#pragma unroll 1
    for (int r = lane; r < R; r += 32) {
      const float e = expf(p_t[r] - mx);
      p_t[r] = e;
      den += e;
    }
    den = warp_sum(den);
  }
#pragma unroll 1
  for (int r = lane; r < R; r += 32) {
    const float pr = sig ? sigmoid_score(p_t[r]) : p_t[r] / den;
    p_t[r] = pr;
    const float sc = pr + cb_t[r];
    const uint32_t bits = sc == 0.0f ? 0u : __float_as_uint(sc);   // -0 ties with +0
    const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    key_t[r] = ((unsigned long long)ord << 32) | (uint32_t)~(uint32_t)r;
  }
  if (lane == 0) rt.gamma[t] = gated ? 1.0f / (1.0f + expf(-gd)) : 1.0f;
  if (a.forced) {
    if (lane < a.K) idx_t[lane] = a.forced[(size_t)t * a.K + lane];
    return;
  }
  unsigned long long key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int r = i * 32 + lane;
    key[i] = r < R ? key_t[r] : 0ull;   // padding: below every real key
  }
  // each lane's keys, largest first (odd-even transposition network)
#pragma unroll
  for (int pass = 0; pass < VPL; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < VPL; i += 2) {
      const unsigned long long hi = key[i] > key[i + 1] ? key[i] : key[i + 1];
      const unsigned long long lo = key[i] > key[i + 1] ? key[i + 1] : key[i];
      key[i] = hi;
      key[i + 1] = lo;
    }
  }
#pragma unroll 1
  for (int k = 0; k < a.K; ++k) {
    unsigned long long best = key[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
      best = ob > best ? ob : best;
    }
    if (key[0] == best) {   // keys are unique: exactly one lane
#pragma unroll
      for (int i = 0; i + 1 < VPL; ++i) key[i] = key[i + 1];
      key[VPL - 1] = 0ull;
    }
    if (lane == k) idx_t[k] = ~(uint32_t)best;
  }
}

// Weights of one token's K chosen columns (warp): unbiased probabilities, renormalised over all K
// slots, times the scaling factor; the identity-expert sum.
__device__ void token_weights(const DecodeArgs& a, int t, const float* p_t,
                              const uint32_t* idx_t, Routing& rt) {
  const int lane = threadIdx.x & 31;
  const int K = a.K;
  const uint32_t my_idx = lane < K ? idx_t[lane] : 0u;
  float wk = lane < K ? p_t[my_idx < (uint32_t)a.R ? my_idx : 0u] : 0.0f;
  const float sum = warp_sum(wk);
  if (a.norm) wk = wk / sum;
  wk *= a.scale;
  float z = (lane < K && (int)my_idx >= a.E) ? wk : 0.0f;
  z = warp_sum(z);
  if (lane < K) rt.w[t * K + lane] = wk;
  if (lane == 0) rt.zsum[t] = z;
}

// Split routing, for at most 32 routed pairs and routers up to 256 wide. The projections need
// only the experts in use, in ascending id (the weight stream of the gate/up items does not
// depend on which tokens chose an expert), so the block's first part of the routing stops
// there and the stream starts; the epilogue warps compute the rest beside it (route_rows_split).
// Part one, all threads: per-token top-K (token_topk), the chosen columns and their
// probabilities kept in static shared memory (the dynamic scratch becomes the weight ring), a
// bit per expert in use, and each expert's slot = the number of experts in use below it.
__device__ void route_active_split(const DecodeArgs& a, Routing& rt, uint8_t* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.R, K = a.K, N = a.N, te = a.te;
  uint32_t* idx_s = reinterpret_cast<uint32_t*>(scratch);                  // [te]
  unsigned long long* k_s = reinterpret_cast<unsigned long long*>(scratch + 128);
  float* p_s = reinterpret_cast<float*>(k_s + (size_t)N * R);             // [N][R]
  float* cb_s = p_s + (size_t)N * R;                                        // [N][R]
  if (warp == nwarps() - 1) rt.bits[lane] = 0u;
  for (int t = warp; t < N; t += nwarps()) {
    const size_t o = (size_t)t * R;
    if (R <= 128) token_topk<4>(a, t, p_s + o, cb_s + o, k_s + o, idx_s + t * K, rt);
    else token_topk<8>(a, t, p_s + o, cb_s + o, k_s + o, idx_s + t * K, rt);
    __syncwarp();
    if (lane < K) {
      const uint32_t c = idx_s[t * K + lane];
      rt.idx[t * K + lane] = (uint16_t)c;
      rt.w[t * K + lane] = p_s[o + (c < (uint32_t)R ? c : 0u)];   // (normalised later)
    }
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t e = lane < te ? (uint32_t)rt.idx[lane] : 0xFFFFFFFFu;
    const bool real = e < (uint32_t)a.E;
    if (real) atomicOr(&rt.bits[e >> 5], 1u << (e & 31));
    __syncwarp();
    if (real) {   // (lanes of one expert write the same slot)
      uint32_t sl = (uint32_t)__popc(rt.bits[e >> 5] & ((1u << (e & 31)) - 1u));
#pragma unroll 1
      for (uint32_t w = 0; w < (e >> 5); ++w) sl += (uint32_t)__popc(rt.bits[w]);
      rt.slot_e[sl] = (uint16_t)e;
    }
    const int nw = (a.E + 31) >> 5;
    const uint32_t n = __reduce_add_sync(0xffffffffu, lane < nw ? (uint32_t)__popc(rt.bits[lane]) : 0u);
    if (lane == 0) rt.n_active = (int)n;
  }
  // the scratch is about to be overwritten by bulk copies (async proxy)
  fence_proxy_async_smem();
  __syncthreads();
}

// Part two, the 128 epilogue threads (named barrier 1) while the weight stream runs: the stable
// sort of the pairs by expert (one warp: match, then a rolled count over the 32 lanes), the
// routing weights (renormalised probabilities x scale, identity-expert sums), and block 0's copy
// of the routing into the workspace.
__device__ void route_rows_split(const DecodeArgs& a, Routing& rt) {
  const int et = threadIdx.x - 64, wq = et >> 5, lane = threadIdx.x & 31;
  const int E = a.E, K = a.K, te = a.te, N = a.N;
  if (wq == 0) {
    const bool valid = lane < te;
    const uint32_t e = valid ? (uint32_t)rt.idx[lane] : 0xFFFFFFFFu;
    const bool real = valid && (int)e < E;
    const uint32_t m = __match_any_sync(0xffffffffu, real ? e : 0xFFFFFFFFu);
    const uint32_t lrank = (uint32_t)__popc(m & ((1u << lane) - 1u));
    const uint32_t reals = __ballot_sync(0xffffffffu, real);
    uint32_t before = 0;
#pragma unroll 1
    for (int i = 0; i < 32; ++i) {
      const uint32_t ei = __shfl_sync(0xffffffffu, e, i);
      if (((reals >> i) & 1u) && ei < e) ++before;
    }
    if (real) {
      const uint32_t row = before + lrank;
      rt.pair_row[lane] = (uint16_t)row;
      rt.row_pair[row] = (uint16_t)lane;
      rt.row_tok[row] = (uint16_t)(lane / K);
      if (lrank == 0) {
        uint32_t sl = (uint32_t)__popc(rt.bits[e >> 5] & ((1u << (e & 31)) - 1u));
#pragma unroll 1
        for (uint32_t w = 0; w < (e >> 5); ++w) sl += (uint32_t)__popc(rt.bits[w]);
        rt.slot_r0[sl] = (uint16_t)before;
        rt.slot_n[sl] = (uint16_t)__popc(m);
      }
    } else if (valid) {
      rt.pair_row[lane] = kNoRow16;
    }
    if (lane == 0) rt.rows = __popc(reals);
  } else {
    for (int t = wq - 1; t < N; t += 3) {
      const uint32_t c = lane < K ? (uint32_t)rt.idx[t * K + lane] : 0u;
      float wk = lane < K ? rt.w[t * K + lane] : 0.0f;
      const float sum = warp_sum(wk);
      if (a.norm) wk = wk / sum;
      wk *= a.scale;
      const float z = warp_sum((lane < K && (int)c >= E) ? wk : 0.0f);
      if (lane < K) rt.w[t * K + lane] = wk;
      if (lane == 0) rt.zsum[t] = z;
    }
  }
  named_sync(1, kEpiThreads);
  if (blockIdx.x == 0) {
    for (int j = et; j < te; j += kEpiThreads) {
      a.idx[j] = rt.idx[j];
      a.w[j] = rt.w[j];
      a.pair_to_row[j] = rt.pair_row[j] == kNoRow16 ? kNoRow : (uint32_t)rt.pair_row[j];
    }
    for (int r = et; r < rt.rows; r += kEpiThreads) a.sorted_pairs[r] = rt.row_pair[r];
    for (int e = et; e < E; e += kEpiThreads) {   // first row of every expert
      uint32_t n = 0;
#pragma unroll 1
      for (int j = 0; j < te; ++j) n += ((uint32_t)rt.idx[j] < (uint32_t)e) ? 1u : 0u;
      a.offsets[e] = n;
    }
    for (int sl = et; sl < rt.n_active; sl += kEpiThreads) a.active[sl] = rt.slot_e[sl];
    for (int t = et; t < N; t += kEpiThreads) a.zsum[t] = rt.zsum[t];
    if (et == 0) {
      a.offsets[E] = (uint32_t)rt.rows;
      a.hdr->num_active = (uint32_t)rt.n_active;
    }
  }
  named_sync(1, kEpiThreads);
}

// Phase 1: the block's own copy of the routing. `scratch`: dynamic shared memory not yet in use.
// Top-K: one warp per token (token_topk up to 256 router columns, else K arg-max rounds). Then the
// stable sort of the pairs by expert: one warp when there are at most 32 pairs, else block-wide
// (ranks inside 32-pair chunks by match, per-chunk counts, block scans over the experts).
__device__ void route_block(const DecodeArgs& a, Routing& rt, uint8_t* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int R = a.R, E = a.E, K = a.K, te = a.te, N = a.N;
  const int nch = (te + 31) / 32;                                      // 32-pair chunks
  uint32_t* idx_s = reinterpret_cast<uint32_t*>(scratch);              // [te]
  uint32_t* lrank_s = idx_s + te;                                      // [te]
  uint32_t* chunk_s = lrank_s + te;                                    // [nch][E]
  uint32_t* base_s = chunk_s + (size_t)nch * E;                        // [E] first rows
  uint32_t* scan_s = base_s + E;                                       // [33]
  unsigned long long* k_s =
      reinterpret_cast<unsigned long long*>(scratch + (((size_t)(scan_s + 40 - idx_s) * 4 + 7) & ~(size_t)7));
  float* p_s = reinterpret_cast<float*>(k_s + (size_t)N * R);             // [N][R]
  float* cb_s = p_s + (size_t)N * R;                                        // [N][R]
  if (te > 32)
    for (int i = tid; i < nch * E; i += blockDim.x) chunk_s[i] = 0;
  for (int t = warp; t < N; t += nwarps()) {
    const size_t o = (size_t)t * R;
    if (R <= 128) token_topk<4>(a, t, p_s + o, cb_s + o, k_s + o, idx_s + t * K, rt);
    else if (R <= 256) token_topk<8>(a, t, p_s + o, cb_s + o, k_s + o, idx_s + t * K, rt);
    else topk_rounds_warp(a, t, idx_s, rt);   // (weights included)
    __syncwarp();
  }
  __syncthreads();
  // the weights (R <= 256) need only idx and p: they run beside the sort (warps 1.. when one
  // warp sorts, else ahead of it)
  if (R <= 256) {
    const int w0 = te <= 32 ? 1 : 0;
    for (int t = warp - w0; t >= 0 && t < N; t += nwarps() - w0)
      token_weights(a, t, p_s + (size_t)t * R, idx_s + t * K, rt);
  }
  if (te <= 32) {
    // one warp: lane j holds pair j; row = pairs of smaller experts + earlier pairs of its own;
    // slot = distinct smaller experts
    if (warp == 0) {
      const bool valid = lane < te;
      const uint32_t e = valid ? idx_s[lane] : 0xFFFFFFFFu;
      const bool real = valid && (int)e < E;
      const uint32_t m = __match_any_sync(0xffffffffu, real ? e : 0xFFFFFFFFu);
      const uint32_t lrank = (uint32_t)__popc(m & ((1u << lane) - 1u));
      const uint32_t reals = __ballot_sync(0xffffffffu, real);
      const uint32_t leaders = __ballot_sync(0xffffffffu, real && lrank == 0);
      uint32_t before = 0, slot = 0;
#pragma unroll 1
      for (int i = 0; i < 32; ++i) {
        const uint32_t ei = __shfl_sync(0xffffffffu, e, i);
        if (((reals >> i) & 1u) && ei < e) {
          ++before;
          if ((leaders >> i) & 1u) ++slot;
        }
      }
      if (real) {
        const uint32_t row = before + lrank;
        rt.pair_row[lane] = (uint16_t)row;
        rt.row_pair[row] = (uint16_t)lane;
        rt.row_tok[row] = (uint16_t)(lane / K);
        if (lrank == 0) {
          rt.slot_e[slot] = (uint16_t)e;
          rt.slot_r0[slot] = (uint16_t)before;
          rt.slot_n[slot] = (uint16_t)__popc(m);
        }
      } else if (valid) {
        rt.pair_row[lane] = kNoRow16;
      }
      if (lane == 0) {
        rt.n_active = __popc(leaders);
        rt.rows = __popc(reals);
      }
    }
    __syncthreads();
    if (blockIdx.x == 0)   // first row of every expert, for the workspace copy below
      for (int e = tid; e < E; e += blockDim.x) {
        uint32_t n = 0;
        for (int j = 0; j < te; ++j) n += (idx_s[j] < (uint32_t)e) ? 1u : 0u;
        base_s[e] = n;
      }
  } else {
    // ranks inside each chunk, and the chunk's count of every expert (its group's last lane)
    for (int j0 = 0; j0 < te; j0 += nthr()) {
      const int j = j0 + tid;
      const uint32_t e = j < te ? idx_s[j] : 0xFFFFFFFFu;
      const bool real = j < te && (int)e < E;
      const uint32_t m = __match_any_sync(0xffffffffu, real ? e : 0xFFFFFFFFu);
      if (j < te) lrank_s[j] = (uint32_t)__popc(m & ((1u << lane) - 1u));
      if (real && (m >> lane) == 1u) chunk_s[(size_t)(j >> 5) * E + e] = (uint32_t)__popc(m);
    }
    __syncthreads();
    // per expert: rows (sum over chunks), first row and slot (block scans), each chunk's first
    // row
    uint32_t carry_rows = 0, carry_slots = 0;
    for (int e0 = 0; e0 < E; e0 += nthr()) {
      const int e = e0 + tid;
      uint32_t tot = 0;
      if (e < E)
        for (int c = 0; c < nch; ++c) tot += chunk_s[(size_t)c * E + e];
      const uint32_t off = block_excl_scan(tot, scan_s, &scan_s[32]);
      const uint32_t tot_rows = scan_s[32];
      __syncthreads();
      const uint32_t sl = block_excl_scan(tot > 0 ? 1u : 0u, scan_s, &scan_s[32]);
      const uint32_t tot_slots = scan_s[32];
      __syncthreads();
      if (e < E) {
        uint32_t row = carry_rows + off;
        base_s[e] = row;
        if (tot > 0) {
          rt.slot_e[carry_slots + sl] = (uint16_t)e;
          rt.slot_r0[carry_slots + sl] = (uint16_t)row;
          rt.slot_n[carry_slots + sl] = (uint16_t)tot;
        }
        for (int c = 0; c < nch; ++c) {
          const uint32_t n = chunk_s[(size_t)c * E + e];
          chunk_s[(size_t)c * E + e] = row;
          row += n;
        }
      }
      carry_rows += tot_rows;
      carry_slots += tot_slots;
    }
    if (tid == 0) {
      rt.n_active = (int)carry_slots;
      rt.rows = (int)carry_rows;
    }
    __syncthreads();
    for (int j = tid; j < te; j += nthr()) {
      const uint32_t e = idx_s[j];
      if ((int)e >= E) {
        rt.pair_row[j] = kNoRow16;
        continue;
      }
      const uint32_t row = chunk_s[(size_t)(j >> 5) * E + e] + lrank_s[j];
      rt.pair_row[j] = (uint16_t)row;
      rt.row_pair[row] = (uint16_t)j;
      rt.row_tok[row] = (uint16_t)(j / K);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int j = tid; j < te; j += blockDim.x) {
      a.idx[j] = idx_s[j];
      a.w[j] = rt.w[j];
      a.pair_to_row[j] = rt.pair_row[j] == kNoRow16 ? kNoRow : (uint32_t)rt.pair_row[j];
    }
    for (int r = tid; r < rt.rows; r += blockDim.x) a.sorted_pairs[r] = rt.row_pair[r];
    for (int e = tid; e < E; e += blockDim.x) a.offsets[e] = base_s[e];
    for (int sl = tid; sl < rt.n_active; sl += blockDim.x) a.active[sl] = rt.slot_e[sl];
    for (int t = tid; t < N; t += blockDim.x) a.zsum[t] = rt.zsum[t];
    if (tid == 0) {
      a.offsets[E] = (uint32_t)rt.rows;
      a.hdr->num_active = (uint32_t)rt.n_active;
    }
  }
  // the scratch is about to be overwritten by bulk copies (async proxy)
  fence_proxy_async_smem();
  __syncthreads();
}

// Phase 3: 8 consecutive outputs per thread, chunks spread over the blocks.
__device__ void combine_chunks(const DecodeArgs& a, const Routing& rt) {
  const int C8 = a.H / 8, Q = a.N * C8;
  for (int q = blockIdx.x + gridDim.x * threadIdx.x; q < Q; q += gridDim.x * blockDim.x) {
    const int t = q / C8, c = q - t * C8;
    const size_t o8 = (size_t)t * a.H + (size_t)c * 8;
    float acc[8], xf[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a.x + o8)), xf);
    const float z = rt.zsum[t];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = z * xf[i];
    if (a.acc) {
      const float4* p = reinterpret_cast<const float4*>(a.acc + o8);
      const float4 u = __ldcg(p), v = __ldcg(p + 1);
      acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
      acc[4] += v.x; acc[5] += v.y; acc[6] += v.z; acc[7] += v.w;
    } else {
      for (int k0 = 0; k0 < a.K; k0 += 8) {   // 8 expert rows in flight per round
        float4 y0[8], y1[8];
        float wk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int k = k0 + u;
          const uint16_t row = k < a.K ? rt.pair_row[t * a.K + k] : kNoRow16;
          wk[u] = 0.0f;
          if (row != kNoRow16) {
            wk[u] = rt.w[t * a.K + k];
            const float4* p = reinterpret_cast<const float4*>(a.yd + (size_t)row * a.H + c * 8);
            y0[u] = __ldcg(p);
            y1[u] = __ldcg(p + 1);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int k = k0 + u;
          if (k < a.K && rt.pair_row[t * a.K + k] != kNoRow16) {
            acc[0] = fmaf(wk[u], y0[u].x, acc[0]);
            acc[1] = fmaf(wk[u], y0[u].y, acc[1]);
            acc[2] = fmaf(wk[u], y0[u].z, acc[2]);
            acc[3] = fmaf(wk[u], y0[u].w, acc[3]);
            acc[4] = fmaf(wk[u], y1[u].x, acc[4]);
            acc[5] = fmaf(wk[u], y1[u].y, acc[5]);
            acc[6] = fmaf(wk[u], y1[u].z, acc[6]);
            acc[7] = fmaf(wk[u], y1[u].w, acc[7]);
          }
        }
      }
    }
    if (a.S > 0) {
      const float g = rt.gamma[t];
      const float4* p = reinterpret_cast<const float4*>(a.shy + o8);
      const float4 u = __ldcg(p), v = __ldcg(p + 1);
      acc[0] = fmaf(g, u.x, acc[0]); acc[1] = fmaf(g, u.y, acc[1]);
      acc[2] = fmaf(g, u.z, acc[2]); acc[3] = fmaf(g, u.w, acc[3]);
      acc[4] = fmaf(g, v.x, acc[4]); acc[5] = fmaf(g, v.y, acc[5]);
      acc[6] = fmaf(g, v.z, acc[6]); acc[7] = fmaf(g, v.w, acc[7]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(a.out + o8) = o;
  }
}

// The block's work items: all gate/up items first, then the down items. Within a phase, items
// are numbered slot-major (a slot's tiles, each tile's contraction boxes in order) and every
// block takes a contiguous, balanced range. The grid of each phase is capped so that no tile
// is split over more than two blocks: the two fp32 partial sums of a tile then meet in a
// zeroed buffer through atomic adds, and a + b == b + a makes the result independent of their
// order (deterministic).
struct Sched {
  int nIt, nSt;     // weight tiles of one gate (or up) projection: routed, shared
  int Pg;           // items per shared gate/up tile (H / 64)
  int Pgr;          // items per routed gate/up tile (H / 64; E4M3: H / 128)
  int ks;           // parts a shared gate/up tile's contraction is split into (E4M3: 2, so
                    // that every gate/up part has Pgr items); part kh accumulates into its
                    // own rows of the gate/up buffer
  int nHt;          // weight tiles of a down projection
  int Pdr, Pds;     // items per down tile: routed (I / 64; E4M3: I / 128), shared (S / 64)
  int na;           // active routed slots
  int g_rt, g_items, d_ritems, d_items;
  int g0, ng, d0, total;   // this block's ranges
  static __device__ __forceinline__ void range(int n, int per_tile, int& i0, int& cnt) {
    int G = gridDim.x;
    int cap = n / per_tile;
    if (cap < 1) cap = 1;
    if (G > cap) G = cap;
    const int b = blockIdx.x;
    if (b >= G) {
      i0 = cnt = 0;
      return;
    }
    i0 = (int)((long long)n * b / G);
    cnt = (int)((long long)n * (b + 1) / G) - i0;
  }
  __device__ void init(const DecodeArgs& a, const Plan& pl, int n_active, bool fp8) {
    const int rbox = fp8 ? 2 * kBox : kBox;   // contraction columns of a routed item
    nIt = a.I / pl.bn_g;
    nSt = a.S / pl.bn_g;
    Pg = a.H / kBox;
    Pgr = a.H / rbox;
    ks = Pg / Pgr;
    nHt = a.H / pl.bn_d;
    Pdr = a.I / rbox;
    Pds = a.S / kBox;
    na = n_active;
    g_rt = na * 2 * nIt;
    g_items = g_rt * Pgr + (a.S ? 2 * nSt : 0) * Pg;
    d_ritems = na * nHt * Pdr;
    d_items = d_ritems + (a.S ? nHt * Pds : 0);
    int nd;
    range(g_items, Pgr, g0, ng);
    range(d_items, Pdr > Pds ? Pdr : Pds, d0, nd);
    total = ng + nd;
  }
  // this block's k-th item: phase, tile (unique within gate/up or within down; a shared
  // gate/up tile's contraction parts count as tiles of their own), contraction box kc, slot
  // (-1: shared expert), tile within the slot's projection(s) (gate/up: gate tiles first,
  // then up tiles), contraction part kh of a shared gate/up tile
  __device__ void item(int k, bool& down, int& tile, int& kc, int& slot, int& lt,
                       int& kh) const {
    down = k >= ng;
    kh = 0;
    if (!down) {
      const int it = g0 + k;
      if (it < g_rt * Pgr) {
        tile = it / Pgr;
        kc = it - tile * Pgr;
        slot = tile / (2 * nIt);
        lt = tile - slot * 2 * nIt;
      } else {
        const int j = it - g_rt * Pgr;
        const int part = j / Pgr;   // (Pg / ks == Pgr)
        lt = part / ks;
        kh = part - lt * ks;
        kc = kh * Pgr + (j - part * Pgr);
        tile = g_rt + part;
        slot = -1;
      }
    } else {
      const int it = d0 + (k - ng);
      if (it < d_ritems) {
        tile = it / Pdr;
        kc = it - tile * Pdr;
        slot = tile / nHt;
        lt = tile - slot * nHt;
      } else {
        const int j = it - d_ritems;
        lt = j / Pds;
        kc = j - lt * Pds;
        tile = na * nHt + lt;
        slot = -1;
      }
    }
  }
};

// Phase 0 also clears the fp32 accumulators the projections add into (the grid barrier before
// phase 2 orders it before every add).
__device__ void zero_accumulators(const DecodeArgs& a) {
  const size_t nth = (size_t)gridDim.x * blockDim.x, tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  auto zero16 = [&](void* p, size_t bytes) {   // bytes: a multiple of 16
    uint4* q = reinterpret_cast<uint4*>(p);
    for (size_t i = tid; i < bytes / 16; i += nth) q[i] = make_uint4(0u, 0u, 0u, 0u);
  };
  zero16(a.hd, (size_t)(a.te + (a.fp8 ? 2 : 1) * a.N) * 2 * a.ldh * 4);
  if (a.yd) zero16(a.yd, (size_t)a.te * a.H * 4);
  if (a.acc) zero16(a.acc, (size_t)a.N * a.H * 4);
  if (a.S > 0) zero16(a.shy, (size_t)a.N * a.H * 4);
  for (size_t i = tid; i < (size_t)kDecodeMaxPairs + 1; i += nth) a.h_cnt[i] = 0u;
}


__device__ __forceinline__ int slot_rows(const DecodeArgs& a, const Routing& m, int slot,
                                         int& r0) {
  if (slot < 0) {
    r0 = a.te;
    return a.N;
  }
  r0 = m.slot_r0[slot];
  return m.slot_n[slot];
}

// FP8: the routed experts' weights are E4M3 with 128 x 128 block scales (the maps of Wg, Wu, Wd
// and of the routed input are uint8 boxes of 128 codes); their items are 128 contraction
// columns, multiplied on the tensor cores as E4M3 x E4M3 (kind::f8f6f4) one item at a time, and
// each item's partial is scaled by its activation and weight block scales into an fp32 run
// accumulator in shared memory before the run is added out. The shared expert stays bf16.
//
// NVFP4: the routed experts' weights are packed E2M1 codes with one E4M3 scale per 16 elements
// and one fp32 scale2 per expert matrix. Their items keep the bf16 items' shape (64 contraction
// columns): the producer streams the codes and scale codes of the box into a codes ring, four
// converter warps (6-9) dequantise them exactly to f16 in the item's weight slot (128-byte
// swizzle), and the MMA multiplies f16 x f16 with the routed input (and the SwiGLU intermediate)
// in f16; scale2 multiplies each run's partial sums when it is drained.
template <bool FP8, bool NV>
__global__ void __launch_bounds__(NV ? kThreads + 32 * kConvWarps : kThreads, 1)
    decode_forward_kernel(const __grid_constant__ CUtensorMap tm_wg,
                          const __grid_constant__ CUtensorMap tm_wu,
                          const __grid_constant__ CUtensorMap tm_sg,
                          const __grid_constant__ CUtensorMap tm_su,
                          const __grid_constant__ CUtensorMap tm_wd,
                          const __grid_constant__ CUtensorMap tm_sd,
                          const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_xn,
                          const __grid_constant__ CUtensorMap tm_fg,
                          const __grid_constant__ CUtensorMap tm_fu,
                          const __grid_constant__ CUtensorMap tm_fd, const DecodeArgs a,
                          const Plan pl) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ Routing meta;
  __shared__ uint64_t bars[3 * kMaxStages + 8];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(16) float stage_rows[16 * kStageLd];   // drain staging, 16 rows x 64
  __shared__ float red_s[kDecodeMaxTokens * kMaxWarps];        // router block reductions
  __shared__ float hsc_s[FP8 ? 2 : 1][16 * kMaxHGroups];       // E4M3: the intermediate's scales
  // 1024-byte alignment for the 128-byte swizzle atoms. Layout: token boxes of the stages, two
  // buffers of the down-projection A operand, the weight ring (the A descriptors' rows 16..127
  // read on into what follows, always inside this allocation). An offset from the __shared__
  // array keeps the shared address space visible to the compiler.
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int stages = pl.stages;
  uint8_t* xtok = smem;                                   // [stages][16 x 128 B]
  uint8_t* hb = xtok + (size_t)stages * kTokBytes;        // [2][max(I,S)/64][16 x 128 B]
  uint8_t* ring = hb + 2 * (size_t)pl.hbytes;             // [stages][BN x 128 B]
  float* racc = reinterpret_cast<float*>(ring + (size_t)stages * kWBytes);   // E4M3: [16][kRaccLd]
  uint8_t* codes = ring + (size_t)stages * kWBytes;       // NVFP4: [stages][BN x 48 B]
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* afull = bars + 2 * kMaxStages;                // [2] run accumulated
  uint64_t* aempty = afull + 2;                           // [2] run drained
  uint64_t* bfull = aempty + 2;                           // [2] down A operand built
  uint64_t* drain = bfull + 2;                            // every MMA complete
  uint64_t* cfull = bars + 2 * kMaxStages + 8;            // NVFP4: a box's codes landed
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = a.hdr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], NV ? 1 + kConvWarps : 1);   // (NVFP4: + the converter warps)
      mbar_init(&empty[s], 1);
      if (NV) mbar_init(&cfull[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);   // the draining warp's lane 0
      mbar_init(&bfull[i], 1);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wu);
    tma_prefetch_desc(&tm_wd);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_xn);
    if (a.S) {
      tma_prefetch_desc(&tm_sg);
      tma_prefetch_desc(&tm_su);
      tma_prefetch_desc(&tm_sd);
    }
    if (NV) {
      tma_prefetch_desc(&tm_fg);
      tma_prefetch_desc(&tm_fu);
      tma_prefetch_desc(&tm_fd);
    }
  }
  if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
  // ---- phases 0 and 1: router logits (spread over the grid) and zeroed accumulators, then
  // each block's routing
  router_rows(a, smem, (size_t)stages * (kTokBytes + kWBytes), red_s);
  {
    // (x is still staged at the start of the dynamic region when it fit)
    const bool staged = (size_t)a.N * a.H * 2 <= (size_t)stages * (kTokBytes + kWBytes);
    const __nv_bfloat16* xs_src = staged ? reinterpret_cast<const __nv_bfloat16*>(smem) : a.x;
    if (a.norm_w) pre_expert_norm_rows(a, xs_src, red_s);
    if (FP8) {
      __syncthreads();   // (this block's xn row, written just above, is read back below)
      quant_token_rows(a, a.norm_w ? a.xn : xs_src);
    }
    if (NV) {
      __syncthreads();
      half_token_rows(a, a.norm_w ? a.xn : xs_src);
    }
  }
  zero_accumulators(a);
  grid_barrier(hdr, gridDim.x);
  const bool split_routing = a.te <= 32 && a.R <= 256;
  if (split_routing) route_active_split(a, meta, smem);   // (ends with a block barrier)
  else route_block(a, meta, smem);                        // (ends with a block barrier)
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;

  // ---- phase 2: the projections
  Sched sc;
  sc.init(a, pl, meta.n_active, FP8);
  const int nitems = sc.total;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      // the weight box of item k: its tensor map and coordinates
      auto locate = [&](int k, bool& down, int& kc, int& slot, const CUtensorMap*& m, int& row) {
        int tile, lt, kh;
        sc.item(k, down, tile, kc, slot, lt, kh);
        if (!down) {
          const int nt = slot >= 0 ? sc.nIt : sc.nSt;
          const bool up = lt >= nt;
          const int r = (up ? lt - nt : lt) * pl.bn_g;
          if (slot >= 0) {
            m = up ? &tm_wu : &tm_wg;
            row = (int)meta.slot_e[slot] * a.I + r;
          } else {
            m = up ? &tm_su : &tm_sg;
            row = r;
          }
        } else {
          m = slot >= 0 ? &tm_wd : &tm_sd;
          row = (slot >= 0 ? (int)meta.slot_e[slot] * a.H : 0) + lt * pl.bn_d;
        }
      };
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int k = 0; k < nitems; ++k) {
        if (!mbar_wait(&empty[s], ph ^ 1, hdr)) { ok = false; break; }
        bool down;
        int kc, slot, row;
        const CUtensorMap* m;
        locate(k, down, kc, slot, m, row);
        uint8_t* wst = ring + (size_t)s * kWBytes;
        // contraction coordinate of the box: 64 bf16 or (E4M3 routed experts) 128 codes
        const int xc = kc * ((FP8 && slot >= 0) ? 2 * kBox : kBox);
        // NVFP4 routed item: its weights reach the slot through the converters
        const bool nvi = NV && slot >= 0;
        const int bn = down ? pl.bn_d : pl.bn_g;
        const uint32_t wbytes = nvi ? 0u : (uint32_t)(bn * 128);
        if (!down) {   // (routed experts read their input xn / its codes, the shared expert x)
          mbar_arrive_expect_tx(&full[s], wbytes + kTokBytes);
          tma_load_2d(xtok + (size_t)s * kTokBytes, slot >= 0 ? &tm_xn : &tm_x, xc, 0, &full[s]);
        } else if (wbytes) {
          mbar_arrive_expect_tx(&full[s], wbytes);
        } else {
          mbar_arrive(&full[s]);
        }
        if (nvi) {
          uint8_t* cst = codes + (size_t)s * kCodeBytes;
          const CUtensorMap* f = m == &tm_wg ? &tm_fg : (m == &tm_wu ? &tm_fu : &tm_fd);
          mbar_arrive_expect_tx(&cfull[s], (uint32_t)(bn * 48));
          tma_load_2d(cst, m, kc * 32, row, &cfull[s]);
          tma_load_2d(cst + bn * 32, f, (kc >> 2) * 16, row, &cfull[s]);
        } else {
          tma_load_2d(wst, m, xc, row, &full[s]);
          if (NV) mbar_arrive(&cfull[s]);   // (the converters pass the item on)
        }
        ++issued;
        if (++s == stages) { s = 0; ph ^= 1; }
      }
      if (!ok)   // let the copies already issued land before the block can exit
        for (int i = issued > stages ? issued - stages : 0; i < issued; ++i) {
          if (NV) mbar_wait(&cfull[i % stages], (uint32_t)((i / stages) & 1), nullptr);
          mbar_wait(&full[i % stages], (uint32_t)((i / stages) & 1), nullptr);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_g = idesc_make(128, pl.bn_g, 1, 1);
      const uint32_t idesc_d = idesc_make(128, pl.bn_d, 1, 1);
      const uint32_t idesc_g8 = idesc_make(128, pl.bn_g, 0, 0);   // E4M3 x E4M3 (f8f6f4)
      const uint32_t idesc_d8 = idesc_make(128, pl.bn_d, 0, 0);   // (f16: f16 x f16, NVFP4)
      int s = 0, run = -1, prev_tile = -1, bslot = -2, nb = 0;
      uint32_t ph = 0, hb_cur = 0;
      bool prev_down = false, ok = true, first = false;
      for (int k = 0; k < nitems && ok; ++k) {
        bool down;
        int tile, kc, slot, lt, kh;
        sc.item(k, down, tile, kc, slot, lt, kh);
        // a new accumulation group: a new tile, or every item of an E4M3 routed expert (each
        // K block carries its own scales, so its partial is drained on its own)
        const bool f8 = FP8 && slot >= 0;
        const bool new_tile = run < 0 || down != prev_down || tile != prev_tile;
        if (new_tile || f8) {
          if (run >= 0) tc_commit(&afull[run & 1]);
          ++run;
          prev_down = down;
          prev_tile = tile;
          if (!mbar_wait(&aempty[run & 1], (((uint32_t)run >> 1) & 1) ^ 1, hdr)) { ok = false; break; }
          if (new_tile && down && slot != bslot) {   // the epilogue's nb-th build, buffer nb % 2
            if (!mbar_wait(&bfull[nb & 1], (uint32_t)(nb >> 1) & 1, hdr)) { ok = false; break; }
            hb_cur = smem_u32(hb) + (uint32_t)(nb & 1) * (uint32_t)pl.hbytes;
            ++nb;
            bslot = slot;
          }
          tc_fence_after();
          first = true;
        }
        if (!mbar_wait(&full[s], ph, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)((run & 1) * kMaxBN);
        const uint32_t a0 = down ? hb_cur + (uint32_t)kc * kTokBytes
                                 : smem_u32(xtok) + (uint32_t)s * kTokBytes;
        const uint32_t b0 = smem_u32(ring) + (uint32_t)s * kWBytes;
        if (f8) {   // 128 codes per row: 4 MMAs of K = 32
          const uint32_t idesc = down ? idesc_d8 : idesc_g8;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_fp8(d, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                       (first && kk == 0) ? 0u : 1u);
        } else {
          const bool f16 = NV && slot >= 0;   // NVFP4 routed item: f16 operands
          const uint32_t idesc = f16 ? (down ? idesc_d8 : idesc_g8) : (down ? idesc_d : idesc_g);
#pragma unroll
          for (int kk = 0; kk < kBox / 16; ++kk)
            tc_mma_bf16(d, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                        (first && kk == 0) ? 0u : 1u);
        }
        first = false;
        tc_commit(&empty[s]);
        if (++s == stages) { s = 0; ph ^= 1; }
      }
      if (ok && run >= 0) tc_commit(&afull[run & 1]);
      // every MMA of this thread complete before TMEM is released
      tc_commit(drain);
      mbar_wait(drain, 0, hdr);
    }
  } else if (warp >= kConvBase / 32) {
    // ------------------------------------------------ NVFP4 converters (warps 6-9)
    if (NV) {
      const int ct = threadIdx.x - kConvBase;   // 0..127
      int s = 0;
      uint32_t ph = 0;
      for (int k = 0; k < nitems; ++k) {
        bool down;
        int tile, kc, slot, lt, kh;
        sc.item(k, down, tile, kc, slot, lt, kh);
        if (!mbar_wait(&cfull[s], ph, hdr)) break;
        if (slot >= 0) {
          const int bn = down ? pl.bn_d : pl.bn_g;
          const uint8_t* cst = codes + (size_t)s * kCodeBytes;
          uint8_t* wst = ring + (size_t)s * kWBytes;
          for (int r = ct; r < bn; r += kConvWarps * 32) {
            const uint32_t sc4 =
                *reinterpret_cast<const uint32_t*>(cst + bn * 32 + r * 16 + (kc & 3) * 4);
            nvfp4_row_to_f16(cst + r * 32, sc4, wst + r * 128, r);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        if (++s == stages) { s = 0; ph ^= 1; }
      }
    }
  } else {
    // ------------------------------------------------ epilogue
    if (split_routing) route_rows_split(a, meta);
    const int et = threadIdx.x - 64;        // 0..127
    const bool drainer = warp == kDrainWarp;
    int run = -1, prev_tile = -1, bslot = -2, nb = 0;
    bool prev_down = false;
    // the accumulation group being drained next (phase, slot, tile within the slot, contraction
    // box, whether it is an E4M3 item, whether it opens its tile's run) and the items of its
    // tile's run so far; whether the previous group was drained already
    bool r_down = false, r_f8 = false, r_first = true, drained = true;
    int r_slot = 0, r_lt = 0, r_kc = 0, r_kh = 0, r_len = 0, r_idx = -1, r_buf = 0;
    bool ok = true;
    // Output row of accumulator row `lane` (lanes < 16; nullptr: not drained) of a group, the
    // factor its partial sums are scaled by (the routing weight in the atomic mode) and the
    // tile's columns.
    auto resolve_dst = [&](bool rdown, int rslot, int rlt, int rkh, float*& dst, float& scale,
                           int& bn) {
      int r0;
      const int ntok = slot_rows(a, meta, rslot, r0);
      dst = nullptr;
      scale = 1.0f;
      if (!rdown) {
        bn = pl.bn_g;
        int row = -1;            // sorted row of (slot, token lane)
        if (rslot < 0) {
          if (lane < a.N) row = a.te + rkh * a.N + lane;   // (part rkh's rows)
        } else {
          for (int j = 0; j < ntok; ++j)
            if ((int)meta.row_tok[r0 + j] == lane) row = r0 + j;
        }
        const int nt = rslot >= 0 ? sc.nIt : sc.nSt;
        const int col = (rlt < nt ? 0 : a.ldh) + (rlt < nt ? rlt : rlt - nt) * bn;
        if (row >= 0) dst = a.hd + (size_t)row * (2 * a.ldh) + col;
        if (NV && rslot >= 0) scale = (rlt < nt ? a.s2_gate : a.s2_up)[meta.slot_e[rslot]];
      } else {
        bn = pl.bn_d;
        const int c0 = rlt * bn;
        if (lane < ntok) {
          const int row = r0 + lane;
          if (rslot < 0) {
            dst = a.shy + (size_t)lane * a.H + c0;
          } else if (a.acc) {
            scale = meta.w[meta.row_pair[row]];
            dst = a.acc + (size_t)meta.row_tok[row] * a.H + c0;
          } else {
            dst = a.yd + (size_t)row * a.H + c0;
          }
          if (NV && rslot >= 0) scale *= a.s2_down[meta.slot_e[rslot]];
        }
      }
    };
    // publish a finished gate/up run: the slot's count moves only after every partial sum of
    // the run landed
    auto publish = [&](bool rdown, int rslot, int rlen) {
      if (!rdown) {
        __syncwarp();
        if (lane == 0)
          red_release_add(a.h_cnt + (rslot < 0 ? kDecodeMaxPairs : rslot), (uint32_t)rlen);
      }
    };
    // Warp 4 drains a finished run: TMEM lane j < 16 holds accumulator row j (token j of x on
    // gate/up, the slot's j-th token on down) across the tile's BN columns. 64 columns at a
    // time go through shared memory so that every row's partial sums leave as coalesced
    // 32-lane atomic adds.
    auto drain_run = [&](int rr, bool rdown, int rslot, int rlt, int rkh, int rlen) {
      if (!ok) return;
      if (!mbar_wait(&afull[rr & 1], ((uint32_t)rr >> 1) & 1, hdr)) { ok = false; return; }
      tc_fence_after();
      const uint32_t tacc = tmem_base + (uint32_t)((rr & 1) * kMaxBN);
      float* dst;
      float scale;
      int bn;
      resolve_dst(rdown, rslot, rlt, rkh, dst, scale, bn);
      const uint32_t rows = __ballot_sync(0xffffffffu, dst != nullptr);
#pragma unroll 1
      for (int c = 0; c < bn; c += 64) {
        float v[64];
        tmem_ld32_nowait(tacc + (uint32_t)c, v);
        tmem_ld32_nowait(tacc + (uint32_t)c + 32, v + 32);
        tmem_wait_ld();
        if (lane < 16 && dst) {
          float4* st = reinterpret_cast<float4*>(stage_rows + lane * kStageLd);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        __syncwarp();
        for (uint32_t m = rows; m; m &= m - 1) {
          const int j = __ffs(m) - 1;
          float* dj = reinterpret_cast<float*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), j));
          const float sj = __shfl_sync(0xffffffffu, scale, j);
          atomicAdd(dj + c + lane, sj * stage_rows[j * kStageLd + lane]);
          atomicAdd(dj + c + 32 + lane, sj * stage_rows[j * kStageLd + 32 + lane]);
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[rr & 1]);
      publish(rdown, rslot, rlen);
    };
    // E4M3: warp 4 drains one item (one 128-wide contraction block of a routed tile): every
    // token row's partial sums times its activation scale (the token's, or on down the
    // intermediate's) and the weight block scale of each 128-column half, into the fp32 run
    // accumulator in shared memory (set by the run's first item); the run's last item adds the
    // accumulator out like drain_run.
    auto drain_item_f8 = [&](int rr, bool rdown, int rslot, int rlt, int rkc, int rbuf,
                             bool rfirst, bool rlast, int rlen) {
      if (!ok) return;
      float* dst;
      float scale;
      int bn;
      resolve_dst(rdown, rslot, rlt, 0, dst, scale, bn);
      // the scales (loaded before the wait)
      const int e = meta.slot_e[rslot];
      float sa = 0.0f, sb0, sb1;
      if (!rdown) {
        if (lane < a.N) sa = a.xs[(size_t)rkc * a.N + lane];
        const bool up = rlt >= sc.nIt;
        const int rb = (up ? rlt - sc.nIt : rlt) * bn / 128;
        const float* sp = (up ? a.s_up : a.s_gate) + ((size_t)e * (a.I / 128) + rb) * (a.H / 128) + rkc;
        sb0 = __ldg(sp);
        sb1 = bn > 128 ? __ldg(sp + a.H / 128) : 0.0f;
      } else {
        if (lane < 16) sa = hsc_s[FP8 ? rbuf : 0][lane * kMaxHGroups + rkc];
        const int rb = rlt * bn / 128;
        const float* sp = a.s_down + ((size_t)e * (a.H / 128) + rb) * (a.I / 128) + rkc;
        sb0 = __ldg(sp);
        sb1 = bn > 128 ? __ldg(sp + a.I / 128) : 0.0f;
      }
      if (!mbar_wait(&afull[rr & 1], ((uint32_t)rr >> 1) & 1, hdr)) { ok = false; return; }
      tc_fence_after();
      const uint32_t tacc = tmem_base + (uint32_t)((rr & 1) * kMaxBN);
      float* ra = racc + lane * kRaccLd;
#pragma unroll 1
      for (int c = 0; c < bn; c += 64) {
        float v[64];
        tmem_ld32_nowait(tacc + (uint32_t)c, v);
        tmem_ld32_nowait(tacc + (uint32_t)c + 32, v + 32);
        tmem_wait_ld();
        if (lane < 16 && dst) {
          const float f = sa * (c < 128 ? sb0 : sb1);
          float4* r4 = reinterpret_cast<float4*>(ra + c);
          // all 16 loads in flight before the first update
          float4 o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = rfirst ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : r4[i];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            r4[i] = make_float4(fmaf(f, v[4 * i], o[i].x), fmaf(f, v[4 * i + 1], o[i].y),
                                fmaf(f, v[4 * i + 2], o[i].z), fmaf(f, v[4 * i + 3], o[i].w));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[rr & 1]);
      if (!rlast) return;
      const uint32_t rows = __ballot_sync(0xffffffffu, dst != nullptr);
      for (uint32_t m = rows; m; m &= m - 1) {
        const int j = __ffs(m) - 1;
        float* dj = reinterpret_cast<float*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), j));
        const float sj = __shfl_sync(0xffffffffu, scale, j);
#pragma unroll 1
        for (int c = 0; c < bn; c += 32) atomicAdd(dj + c + lane, sj * racc[j * kRaccLd + c + lane]);
      }
      __syncwarp();
      publish(rdown, rslot, rlen);
    };
    // drains the pending group; `run_ends`: the next group belongs to another tile (or there
    // is none), so an E4M3 run's accumulator is added out
    auto drain_current = [&](bool run_ends) {
      if (drainer && !drained && r_idx >= 0) {
        if (FP8 && r_f8)
          drain_item_f8(r_idx, r_down, r_slot, r_lt, r_kc, r_buf, r_first, run_ends, r_len);
        else
          drain_run(r_idx, r_down, r_slot, r_lt, r_kh, r_len);
      }
      drained = true;
    };
    // waits until every gate/up item of `slot` has been added out (other blocks; bounded)
    auto wait_slot = [&](int slot) {
      const uint32_t target =
          (uint32_t)(slot >= 0 ? 2 * sc.nIt * sc.Pgr : 2 * sc.nSt * sc.Pg);
      if (drainer && lane == 0) {
        const uint32_t* cnt = a.h_cnt + (slot < 0 ? kDecodeMaxPairs : slot);
        if (ld_acquire(cnt) < target) {
          const long long t0 = clock64();
          while (ld_acquire(cnt) < target) {
            if (clock64() - t0 > kSpinLimitCycles) {   // (the result is then not used)
              report_timeout(hdr);
              break;
            }
          }
        }
      }
      named_sync(1, kEpiThreads);
    };
    // SiLU(gate) * up of the slot's tokens as the bf16 A operand (buffer nb % 2), 16 rows per
    // 64-column box with the 128-byte swizzle: row j's 16-byte chunk c of box kb at
    // kb * 2048 + j * 128 + ((c ^ (j & 7)) * 16).
    auto build_a = [&](int slot, uint8_t* buf) {
      wait_slot(slot);
      int r0;
      const int ntok = slot_rows(a, meta, slot, r0);
      const int L = slot >= 0 ? a.I : a.S;
      const int cpr = L / 8;   // 16-byte chunks per row
      // (rows ntok..15 keep whatever they hold: an MMA row depends only on its own A row, and
      // those accumulator rows are never drained)
      for (int id = et; id < ntok * cpr; id += kEpiThreads) {
        const int j = id / cpr, c = id - j * cpr;
        uint4 o;
        const float* hr = a.hd + (size_t)(r0 + j) * (2 * a.ldh) + c * 8;
        float4 g0v = __ldcg(reinterpret_cast<const float4*>(hr));
        float4 g1v = __ldcg(reinterpret_cast<const float4*>(hr + 4));
        float4 u0 = __ldcg(reinterpret_cast<const float4*>(hr + a.ldh));
        float4 u1 = __ldcg(reinterpret_cast<const float4*>(hr + a.ldh + 4));
        if (FP8 && slot < 0) {   // the shared tiles' second contraction part, added in order
          const float* h2 = hr + (size_t)a.N * (2 * a.ldh);
          auto add4 = [](float4& x, const float4 y) { x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w; };
          add4(g0v, __ldcg(reinterpret_cast<const float4*>(h2)));
          add4(g1v, __ldcg(reinterpret_cast<const float4*>(h2 + 4)));
          add4(u0, __ldcg(reinterpret_cast<const float4*>(h2 + a.ldh)));
          add4(u1, __ldcg(reinterpret_cast<const float4*>(h2 + a.ldh + 4)));
        }
        if (NV && slot >= 0) {   // the NVFP4 down items' f16 operand
          o.x = pack_f16x2(silu(g0v.x) * u0.x, silu(g0v.y) * u0.y);
          o.y = pack_f16x2(silu(g0v.z) * u0.z, silu(g0v.w) * u0.w);
          o.z = pack_f16x2(silu(g1v.x) * u1.x, silu(g1v.y) * u1.y);
          o.w = pack_f16x2(silu(g1v.z) * u1.z, silu(g1v.w) * u1.w);
        } else {
          o.x = pack_bf16x2(silu(g0v.x) * u0.x, silu(g0v.y) * u0.y);
          o.y = pack_bf16x2(silu(g0v.z) * u0.z, silu(g0v.w) * u0.w);
          o.z = pack_bf16x2(silu(g1v.x) * u1.x, silu(g1v.y) * u1.y);
          o.w = pack_bf16x2(silu(g1v.z) * u1.z, silu(g1v.w) * u1.w);
        }
        *reinterpret_cast<uint4*>(buf + (size_t)(c >> 3) * 2048 + j * 128 +
                                  (((c & 7) ^ (j & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      named_sync(1, kEpiThreads);
      if (et == 0) mbar_arrive(&bfull[nb & 1]);
    };
    // E4M3 routed slot: the intermediate h = SiLU(gate) * up quantised per 1x128 group (the
    // rule of quant_token_rows) as the E4M3 A operand of the down items, 16 rows per 128-code
    // box with the 128-byte swizzle, one warp per (token row, group); scales into hsc_s[nb % 2].
    auto build_a_f8 = [&](int slot, uint8_t* buf) {
      wait_slot(slot);
      int r0;
      const int ntok = slot_rows(a, meta, slot, r0);
      const int G = a.I / 128;
      const int wq = et >> 5;
      for (int gi = wq; gi < ntok * G; gi += kEpiThreads / 32) {
        const int j = gi / G, g = gi - j * G;
        const float* hr = a.hd + (size_t)(r0 + j) * (2 * a.ldh) + g * 128 + lane * 4;
        const float4 gv = __ldcg(reinterpret_cast<const float4*>(hr));
        const float4 uv = __ldcg(reinterpret_cast<const float4*>(hr + a.ldh));
        const float h0 = silu(gv.x) * uv.x, h1 = silu(gv.y) * uv.y;
        const float h2 = silu(gv.z) * uv.z, h3 = silu(gv.w) * uv.w;
        const float am = warp_max(fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(h2), fabsf(h3))));
        const float sc8 = am > 0.0f ? __fdiv_rn(am, 448.0f) : 1.0f;
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(h0, sc8), __fdiv_rn(h1, sc8)), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(h2, sc8), __fdiv_rn(h3, sc8)), __NV_SATFINITE, __NV_E4M3);
        *reinterpret_cast<uint32_t*>(buf + (size_t)g * 2048 + j * 128 +
                                     ((((lane >> 2) ^ (j & 7)) << 4) | ((lane & 3) << 2))) =
            lo | (hi << 16);
        if (lane == 0) hsc_s[FP8 ? (nb & 1) : 0][j * kMaxHGroups + g] = sc8;
      }
      fence_proxy_async_smem();
      named_sync(1, kEpiThreads);
      if (et == 0) mbar_arrive(&bfull[nb & 1]);
    };
    for (int k = 0; k < nitems; ++k) {
      bool down;
      int tile, kc, slot, lt, kh;
      sc.item(k, down, tile, kc, slot, lt, kh);
      const bool f8 = FP8 && slot >= 0;
      const bool new_tile = run < 0 || down != prev_down || tile != prev_tile;
      if (new_tile || f8) {
        ++run;
        prev_down = down;
        prev_tile = tile;
        if (new_tile && down && slot != bslot) {
          // The previous gate/up run is published first (the count may wait on it). Otherwise
          // the next buffer is free -- the runs that read it, two slot changes back, are
          // drained -- and the build overlaps the MMAs of the previous run.
          if (!r_down) drain_current(true);
          if (f8) build_a_f8(slot, hb + (size_t)(nb & 1) * pl.hbytes);
          else build_a(slot, hb + (size_t)(nb & 1) * pl.hbytes);
          ++nb;
          bslot = slot;
        }
        drain_current(new_tile);
        r_idx = run;
        r_down = down;
        r_slot = slot;
        r_lt = lt;
        r_kc = kc;
        r_kh = kh;
        r_f8 = f8;
        r_buf = (nb - 1) & 1;   // (down: the buffer of this slot's build)
        r_first = new_tile;
        if (new_tile) r_len = 0;
        drained = false;
      }
      ++r_len;
    }
    drain_current(true);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // ---- phase 3: every block's partial sums have landed; combine
  grid_barrier(hdr, 2 * gridDim.x);
  combine_chunks(a, meta);
}

int sm_count() {
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

// Weight rows per tile of each phase; the tensor maps of the weights use them as box rows.
void decode_tile_rows(int H, int I, int S, int* bn_g, int* bn_d) {
  *bn_g = (I % 256 == 0 && S % 256 == 0) ? 256 : 128;
  *bn_d = H % 256 == 0 ? 256 : 128;
}

cudaError_t launch_decode_forward(const DecodeArgs& a, const CUtensorMap* maps, cudaStream_t st) {
  if (a.te > kDecodeMaxPairs || a.N > kDecodeMaxTokens || a.N < 1 || !a.h_cnt ||
      a.H % 128 || a.I % 128 || a.S % 128 || a.R > 1024 || a.E > 1024 || a.K > 32)
    return cudaErrorInvalidValue;
  if (a.fp8 && (!a.s_gate || !a.s_up || !a.s_down || !a.xq || !a.xs || a.I > 128 * kMaxHGroups))
    return cudaErrorInvalidValue;
  if (a.nv && (a.fp8 || !a.s2_gate || !a.s2_up || !a.s2_down || !a.xh || a.H % 256 || a.I % 256))
    return cudaErrorInvalidValue;
  Plan pl{};
  decode_tile_rows(a.H, a.I, a.S, &pl.bn_g, &pl.bn_d);
  // boxes of the down A operand: routed I / 64 (bf16) or I / 128 (E4M3), shared S / 64
  const int hb_boxes = a.fp8 ? (a.I / 128 > a.S / kBox ? a.I / 128 : a.S / kBox)
                             : (a.I > a.S ? a.I : a.S) / kBox;
  pl.hbytes = hb_boxes * kTokBytes;
  const int per_stage = kTokBytes + kWBytes + (a.nv ? kCodeBytes : 0);
  // alignment slack + two down A operands (+ the E4M3 run accumulator)
  const int fixed = 1024 + 2 * pl.hbytes + (a.fp8 ? kRaccBytes : 0);
  // (the static shared memory -- routing, barriers, drain staging -- stays within 16 KB)
  pl.stages = (kSmemLimit - 16384 - fixed) / per_stage;
  if (pl.stages > kMaxStages) pl.stages = kMaxStages;
  if (pl.stages < 2) return cudaErrorInvalidValue;
  // the routing scratch of phase 1 lives in the (not yet used) dynamic region
  const size_t scratch = a.te <= 32 && a.R <= 256
                             ? 128 + (size_t)a.N * a.R * 16   // split routing
                             : (size_t)a.te * 8 + (size_t)((a.te + 31) / 32) * a.E * 4 +
                                   (size_t)a.E * 4 + 160 +
                                   (a.R <= 256 ? 8 + (size_t)a.N * a.R * 16 : 0);
  if (scratch > (size_t)pl.stages * (kTokBytes + kWBytes)) return cudaErrorInvalidValue;
  const size_t sm = (size_t)fixed + (size_t)pl.stages * per_stage;
  const int nthreads = a.nv ? kThreads + 32 * kConvWarps : kThreads;
  auto kern = a.fp8 ? decode_forward_kernel<true, false>
                    : (a.nv ? decode_forward_kernel<false, true> : decode_forward_kernel<false, false>);
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(kern), sm);
  if (e != cudaSuccess) return e;
  // the down phase waits on other blocks' gate/up work: all blocks must be resident (checked
  // once per device and shared-memory size)
  {
    static std::mutex mu;
    static std::set<std::pair<int, size_t>> ok;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    const size_t key = sm * 4 + (a.fp8 ? 1 : 0) + (a.nv ? 2 : 0);
    if (!ok.count({dev, key})) {
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nthreads, sm);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) return cudaErrorInvalidConfiguration;
      ok.insert({dev, key});
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[kDmWg], maps[kDmWu], maps[kDmSg],
                            maps[kDmSu], maps[kDmWd], maps[kDmSd], maps[kDmX], maps[kDmXn],
                            maps[kDmFg], maps[kDmFu], maps[kDmFd], a, pl);
}

}  // namespace moe
