// Decode chain (few tokens): weight-streaming GEMVs over the experts the batch actually
// touches. Each touched expert's gate/up/down weights are read from HBM once, for all the
// tokens routed to it; the shared expert is one more "slot" of the same launches.
//
// Pages: "spark_model/layers/moe/forward.rs" (`forward`: fused gate/up GEMV for the K routed
// experts plus the shared expert, fused SiLU+down GEMV, weighted sum + sigmoid-gated shared
// blend, all on device with no host synchronisation) and
// "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (token-major gate/up for a few rows,
// routed down projections weighted and FP32-atomic-added into a [N,H] accumulator zeroed
// first, then a finalize that casts to BF16 and blends the shared expert).
//
// Both kernels are persistent (one block per SM) and split the work into items: a few
// consecutive weight rows of one slot, contiguous in memory. Warp 0 streams items into a
// shared-memory ring with 1D bulk copies (150-200 KB in flight per SM, enough to keep HBM
// busy); 8 consumer warps take the dot products against the slot's token vectors. Each block
// owns a contiguous range of items, so a slot's token list changes rarely within a block.
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxTok = 16;          // tokens per expert the decode chain handles
constexpr int kConsumers = 8;        // consumer warps
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kSmemBudget = 214 * 1024;   // dynamic part; + RouteMeta, of the 227 KB allowed
constexpr int kMaxPairs = 512;        // N * K of the decode chain (16 tokens x top-32)
constexpr int kMaxStages = 4;
constexpr int kDownRows = 32;        // down-projection rows per item (4 per consumer warp)

// Contiguous, balanced share [i0, i1) of `total` items for this block.
__device__ __forceinline__ void item_range(int total, int& i0, int& i1) {
  const long long G = gridDim.x, b = blockIdx.x;
  i0 = (int)((total * b) / G);
  i1 = (int)((total * (b + 1)) / G);
}

// Routing of the batch, copied to shared memory once per block so the streaming loops
// never wait on a dependent global load: expert, first sorted row and row count of every
// active slot, and the token of every sorted row.
struct RouteMeta {
  int n_active;
  int slot_e[kMaxPairs];
  int slot_r0[kMaxPairs];
  int slot_n[kMaxPairs];
  int row_tok[kMaxPairs];
};

// All threads of the block; routing metadata is read through L2 (an earlier kernel wrote it).
__device__ void load_route_meta(const DecodeArgs& a, RouteMeta& m) {
  const int n_active = (int)__ldcg(&a.hdr->num_active);
  for (int s = threadIdx.x; s < n_active; s += blockDim.x) {
    const int e = (int)__ldcg(a.active + s);
    const int r0 = (int)__ldcg(a.offsets + e);
    m.slot_e[s] = e;
    m.slot_r0[s] = r0;
    m.slot_n[s] = (int)__ldcg(a.offsets + e + 1) - r0;
  }
  for (int r = threadIdx.x; r < a.te; r += blockDim.x)
    m.row_tok[r] = (int)(__ldcg(a.sorted_pairs + r) / (uint32_t)a.K);
  if (threadIdx.x == 0) m.n_active = n_active;
  __syncthreads();
}

// Token list of slot `slot` (-1: the shared expert): lane j < ntok gets the token id and the
// intermediate row of the j-th token.
__device__ __forceinline__ int slot_tokens(const DecodeArgs& a, const RouteMeta& m, int slot,
                                           int lane, int& tok, int& row) {
  if (slot < 0) {
    tok = lane;
    row = a.te + lane;
    return a.N;
  }
  const int r0 = m.slot_r0[slot], ntok = m.slot_n[slot];
  row = r0 + lane;
  tok = lane < ntok ? m.row_tok[r0 + lane] : 0;
  return ntok;
}

// ------------------------------------------------------------------ gate/up

// hd[row_j, i] = SiLU(x_j . Wg[i]) * (x_j . Wu[i]) for every token j of the slot.
// Item = `rp` consecutive row pairs of one slot: rp gate rows then rp up rows in the stage.
__global__ void __launch_bounds__(kThreads, 1)
    decode_gateup_kernel(DecodeArgs a, int rp, int stages, int item_bytes, int xbytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteMeta meta;
  const int H = a.H, N = a.N;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);             // [N, H]
  uint8_t* ring = smem + xbytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)stages * item_bytes);
  uint64_t* empty = full + kMaxStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    fence_mbarrier_init();
  }
  // the block input is not produced by the router: stage it before waiting on the router
  for (int i = threadIdx.x; i < N * H / 8; i += blockDim.x)
    reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(a.x)[i];
  __syncthreads();
  pdl_wait();       // routing of the router kernel
  pdl_trigger();    // the down projection may start streaming its weights
  load_route_meta(a, meta);

  const int per_slot = a.I / rp;
  const int routed = meta.n_active * per_slot;
  const int total = routed + (a.S > 0 ? a.S / rp : 0);
  int i0, i1;
  item_range(total, i0, i1);
  const uint32_t half_bytes = (uint32_t)(rp * H * 2);

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int it = i0; it < i1; ++it, ++issued) {
        const int k = it - i0, s = k % stages;
        if (!mbar_wait(&empty[s], ((k / stages) & 1) ^ 1, a.hdr)) { ok = false; break; }
        const __nv_bfloat16 *g, *u;
        if (it < routed) {
          const int e = meta.slot_e[it / per_slot];
          const size_t r = (size_t)e * a.I + (size_t)(it % per_slot) * rp;
          g = a.wg + r * H;
          u = a.wu + r * H;
        } else {
          const size_t r = (size_t)(it - routed) * rp;
          g = a.sg + r * H;
          u = a.su + r * H;
        }
        uint8_t* dst = ring + (size_t)s * item_bytes;
        mbar_arrive_expect_tx(&full[s], 2 * half_bytes);
        bulk_load(dst, g, half_bytes, &full[s]);
        bulk_load(dst + half_bytes, u, half_bytes, &full[s]);
      }
      if (!ok)   // let the copies already issued land before the block can exit
        for (int k = issued > stages ? issued - stages : 0; k < issued; ++k)
          mbar_wait(&full[k % stages], (k / stages) & 1, nullptr);
    }
  } else {
    const int cw = warp - 1;
    int cur_slot = -2, ntok = 0, tok = 0, orow = 0;
    for (int it = i0; it < i1; ++it) {
      const int k = it - i0, s = k % stages;
      const int slot = it < routed ? it / per_slot : -1;
      const int i = (it < routed ? (it % per_slot) : (it - routed)) * rp + cw;
      if (slot != cur_slot) {
        cur_slot = slot;
        ntok = slot_tokens(a, meta, slot, lane, tok, orow);
      }
      if (!mbar_wait(&full[s], (k / stages) & 1, a.hdr)) break;
      if (cw < rp) {
        const uint8_t* st = ring + (size_t)s * item_bytes + (size_t)cw * H * 2;
        const uint4* gr = reinterpret_cast<const uint4*>(st);
        const uint4* ur = reinterpret_cast<const uint4*>(st + half_bytes);
        float ag[kMaxTok], au[kMaxTok];
        int tks[kMaxTok];     // token ids, gathered while the whole warp is converged
#pragma unroll
        for (int j = 0; j < kMaxTok; ++j) {
          ag[j] = au[j] = 0.0f;
          tks[j] = __shfl_sync(0xffffffffu, tok, j);
        }
        for (int c = lane; c < H / 8; c += 32) {
          float gf[8], uf[8];
          bf16x8_to_f32(gr[c], gf);
          bf16x8_to_f32(ur[c], uf);
#pragma unroll
          for (int j = 0; j < kMaxTok; ++j) {
            if (j < ntok) {
              float xf[8];
              bf16x8_to_f32(reinterpret_cast<const uint4*>(xs + (size_t)tks[j] * H)[c], xf);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                ag[j] = fmaf(gf[q], xf[q], ag[j]);
                au[j] = fmaf(uf[q], xf[q], au[j]);
              }
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kMaxTok; ++j) {
          if (j < ntok) {
            const float gs = warp_sum(ag[j]);
            const float us = warp_sum(au[j]);
            const int rj = __shfl_sync(0xffffffffu, orow, j);
            if (lane == 0) a.hd[(size_t)rj * a.ldh + i] = silu(gs) * us;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// ------------------------------------------------------------------ down

// y_j[r] = h_j . Wd[r] for every token j of the slot. Item = kDownRows consecutive rows of
// Wd_e (or of the shared down weights); routed results go to yd, or are weighted and
// atomically added into acc; shared results go to shy.
__global__ void __launch_bounds__(kThreads, 1)
    decode_down_kernel(DecodeArgs a, int stages, int item_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteMeta meta;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)stages * item_bytes);
  uint64_t* empty = full + kMaxStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    fence_mbarrier_init();
  }
  // Routing metadata comes from the router kernel, which finished before the gate/up kernel
  // passed its own wait, so the weights can stream before this kernel's wait; only the
  // consumers read the SwiGLU outputs and wait for them.
  load_route_meta(a, meta);
  const int per_slot = H / kDownRows;
  const int routed = meta.n_active * per_slot;
  const int total = routed + (a.S > 0 ? per_slot : 0);
  int i0, i1;
  item_range(total, i0, i1);

  if (warp == 0) {
    pdl_trigger();
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int it = i0; it < i1; ++it, ++issued) {
        const int k = it - i0, s = k % stages;
        if (!mbar_wait(&empty[s], ((k / stages) & 1) ^ 1, a.hdr)) { ok = false; break; }
        const __nv_bfloat16* src;
        uint32_t bytes;
        if (it < routed) {
          const int e = meta.slot_e[it / per_slot];
          src = a.wd + ((size_t)e * H + (size_t)(it % per_slot) * kDownRows) * a.I;
          bytes = (uint32_t)(kDownRows * a.I * 2);
        } else {
          src = a.sd + (size_t)(it - routed) * kDownRows * a.S;
          bytes = (uint32_t)(kDownRows * a.S * 2);
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + (size_t)s * item_bytes, src, bytes, &full[s]);
      }
      if (!ok)
        for (int k = issued > stages ? issued - stages : 0; k < issued; ++k)
          mbar_wait(&full[k % stages], (k / stages) & 1, nullptr);
    }
  } else {
    pdl_wait();     // SwiGLU outputs of the gate/up kernel
    pdl_trigger();
    const int cw = warp - 1;
    int cur_slot = -2, ntok = 0, tok = 0, orow = 0;
    float wt = 0.0f;
    for (int it = i0; it < i1; ++it) {
      const int k = it - i0, s = k % stages;
      const bool shared_item = it >= routed;
      const int slot = shared_item ? -1 : it / per_slot;
      const int rbase = (shared_item ? it - routed : it % per_slot) * kDownRows;
      const int L = shared_item ? a.S : a.I;
      if (slot != cur_slot) {
        cur_slot = slot;
        ntok = slot_tokens(a, meta, slot, lane, tok, orow);
        if (!shared_item && a.acc && lane < ntok) wt = a.w[__ldcg(a.sorted_pairs + orow)];
      }
      if (!mbar_wait(&full[s], (k / stages) & 1, a.hdr)) break;
      const uint8_t* stage = ring + (size_t)s * item_bytes;
#pragma unroll 1
      for (int rr = 0; rr < kDownRows / kConsumers; ++rr) {
        const int rl = cw * (kDownRows / kConsumers) + rr;
        const uint4* wr = reinterpret_cast<const uint4*>(stage + (size_t)rl * L * 2);
        float acc[kMaxTok];
        int rws[kMaxTok];     // SwiGLU rows, gathered while the whole warp is converged
#pragma unroll
        for (int j = 0; j < kMaxTok; ++j) {
          acc[j] = 0.0f;
          rws[j] = __shfl_sync(0xffffffffu, orow, j);
        }
        for (int c = lane; c < L / 8; c += 32) {
          float wf[8];
          bf16x8_to_f32(wr[c], wf);
#pragma unroll
          for (int j = 0; j < kMaxTok; ++j) {
            if (j < ntok) {
              const float4* hp =
                  reinterpret_cast<const float4*>(a.hd + (size_t)rws[j] * a.ldh) + 2 * c;
              const float4 h0 = hp[0], h1 = hp[1];
              acc[j] = fmaf(wf[0], h0.x, acc[j]);
              acc[j] = fmaf(wf[1], h0.y, acc[j]);
              acc[j] = fmaf(wf[2], h0.z, acc[j]);
              acc[j] = fmaf(wf[3], h0.w, acc[j]);
              acc[j] = fmaf(wf[4], h1.x, acc[j]);
              acc[j] = fmaf(wf[5], h1.y, acc[j]);
              acc[j] = fmaf(wf[6], h1.z, acc[j]);
              acc[j] = fmaf(wf[7], h1.w, acc[j]);
            }
          }
        }
        const int r = rbase + rl;
#pragma unroll
        for (int j = 0; j < kMaxTok; ++j) {
          if (j < ntok) {
            const float y = warp_sum(acc[j]);
            const int tj = __shfl_sync(0xffffffffu, tok, j);
            const int rj = __shfl_sync(0xffffffffu, orow, j);
            const float wj = __shfl_sync(0xffffffffu, wt, j);
            if (lane == 0) {
              if (shared_item) a.shy[(size_t)tj * H + r] = y;
              else if (a.acc) atomicAdd(a.acc + (size_t)tj * H + r, wj * y);
              else a.yd[(size_t)rj * H + r] = y;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
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

cudaError_t launch_decode_gateup(const DecodeArgs& a, cudaStream_t st) {
  if (a.te > kMaxPairs) return cudaErrorInvalidValue;
  const int xbytes = (a.N * a.H * 2 + 127) & ~127;
  // row pairs per item: the most (<= 8, one per consumer warp) that keep 3 stages in budget
  int rp = 8;
  while (rp > 1 && (a.I % rp || (a.S && a.S % rp) ||
                    (size_t)xbytes + 3 * (size_t)rp * 4 * a.H + 1024 > (size_t)kSmemBudget))
    rp >>= 1;
  const int item = rp * 4 * a.H;
  int stages = (kSmemBudget - 1024 - xbytes) / item;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 1) return cudaErrorInvalidValue;
  const size_t sm = (size_t)xbytes + (size_t)stages * item + 2 * kMaxStages * 8;
  cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_gateup_kernel, dim3(sm_count()), dim3(kThreads), sm, st, a, rp,
                          stages, item, xbytes);
}

cudaError_t launch_decode_down(const DecodeArgs& a, cudaStream_t st) {
  if (a.H % kDownRows || a.te > kMaxPairs) return cudaErrorInvalidValue;
  const int L = a.I > a.S ? a.I : a.S;
  const int item = kDownRows * L * 2;
  int stages = (kSmemBudget - 1024) / item;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 1) return cudaErrorInvalidValue;
  const size_t sm = (size_t)stages * item + 2 * kMaxStages * 8;
  cudaError_t e = cudaFuncSetAttribute(decode_down_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_down_kernel, dim3(sm_count()), dim3(kThreads), sm, st, a, stages,
                          item);
}

}  // namespace moe
