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
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxTok = 16;        // tokens per expert the decode chain handles
constexpr int kGuRowsPerWarp = 2;  // gate/up row pairs per warp
constexpr int kGuRows = 8 * kGuRowsPerWarp;
constexpr int kDnRowsPerWarp = 4;  // down rows per warp
constexpr int kDnRows = 8 * kDnRowsPerWarp;

// Streaming 16-byte load that does not allocate in L1 (weights are read exactly once).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct Slot {
  int ntok;
  const __nv_bfloat16* w0;
  const __nv_bfloat16* w1;
  int nrows;
};

// Resolves block slot `slot`: an active routed expert (slot < n_slots) or the shared expert.
// Fills the token ids and output rows of the slot in shared memory. Returns false if the
// slot has no work.
__device__ bool resolve_slot(const DecodeArgs& a, int slot, int n_slots, bool down, Slot& sl,
                             int* tok_s, int* row_s) {
  if (slot < n_slots) {
    if ((uint32_t)slot >= __ldcg(&a.hdr->num_active)) return false;
    const int e = (int)__ldcg(a.active + slot);
    const int r0 = (int)__ldcg(a.offsets + e), r1 = (int)__ldcg(a.offsets + e + 1);
    sl.ntok = r1 - r0;
    if (down) {
      sl.w0 = a.wd + (size_t)e * a.H * a.I;
      sl.nrows = a.H;
    } else {
      sl.w0 = a.wg + (size_t)e * a.I * a.H;
      sl.w1 = a.wu + (size_t)e * a.I * a.H;
      sl.nrows = a.I;
    }
    for (int j = threadIdx.x; j < sl.ntok; j += blockDim.x) {
      tok_s[j] = (int)(__ldcg(a.sorted_pairs + r0 + j) / (uint32_t)a.K);
      row_s[j] = r0 + j;
    }
  } else {
    if (a.S == 0) return false;
    sl.ntok = a.N;
    if (down) {
      sl.w0 = a.sd;
      sl.nrows = a.H;
    } else {
      sl.w0 = a.sg;
      sl.w1 = a.su;
      sl.nrows = a.S;
    }
    for (int j = threadIdx.x; j < a.N; j += blockDim.x) {
      tok_s[j] = j;
      row_s[j] = a.te + j;
    }
  }
  return sl.ntok > 0;
}

// hd[row_j, i] = SiLU(x_j . Wg[i]) * (x_j . Wu[i]) for every token j of the slot.
__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeArgs a, int n_slots) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int tok_s[kMaxTok], row_s[kMaxTok];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);   // [ntok, H]
  pdl_wait();       // routing of the router kernel
  pdl_trigger();    // the down projection may start issuing its weight loads
  Slot sl;
  if (!resolve_slot(a, blockIdx.y, n_slots, false, sl, tok_s, row_s)) return;
  const int row_base = blockIdx.x * kGuRows;
  if (row_base >= sl.nrows) return;
  __syncthreads();
  const int H = a.H, chunks = H / 8;
  for (int i = threadIdx.x; i < sl.ntok * chunks; i += blockDim.x) {
    int j = i / chunks, c = i % chunks;
    reinterpret_cast<uint4*>(xs)[j * chunks + c] =
        reinterpret_cast<const uint4*>(a.x + (size_t)tok_s[j] * H)[c];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int ntok = sl.ntok;
  for (int rr = 0; rr < kGuRowsPerWarp; ++rr) {
    const int i = row_base + wid * kGuRowsPerWarp + rr;
    if (i >= sl.nrows) break;
    float ag[kMaxTok], au[kMaxTok];
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) ag[j] = au[j] = 0.0f;
    const uint4* g = reinterpret_cast<const uint4*>(sl.w0 + (size_t)i * H);
    const uint4* u = reinterpret_cast<const uint4*>(sl.w1 + (size_t)i * H);
    for (int c0 = 0; c0 < chunks; c0 += 256) {
      uint4 gv[8], uv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = c0 + q * 32 + lane;
        if (c < chunks) {
          gv[q] = ld_stream(g + c);
          uv[q] = ld_stream(u + c);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = c0 + q * 32 + lane;
        if (c < chunks) {
          float gf[8], uf[8];
          bf16x8_to_f32(gv[q], gf);
          bf16x8_to_f32(uv[q], uf);
#pragma unroll
          for (int j = 0; j < kMaxTok; ++j) {
            if (j < ntok) {
              float xf[8];
              bf16x8_to_f32(reinterpret_cast<const uint4*>(xs)[j * chunks + c], xf);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                ag[j] = fmaf(gf[k], xf[k], ag[j]);
                au[j] = fmaf(uf[k], xf[k], au[j]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      if (j < ntok) {
        const float gs = warp_sum(ag[j]);
        const float us = warp_sum(au[j]);
        if (lane == 0) a.hd[(size_t)row_s[j] * a.ldh + i] = silu(gs) * us;
      }
    }
  }
}

// y_j[r] = h_j . Wd[r] for every token j of the slot; routed results go to yd (or are
// weighted and atomically added into acc), shared results to shy.
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a, int n_slots) {
  extern __shared__ __align__(16) float hs[];                   // [ntok, L]
  __shared__ int tok_s[kMaxTok], row_s[kMaxTok];
  __shared__ float wt_s[kMaxTok];
  Slot sl;
  const bool shared_slot = (int)blockIdx.y >= n_slots;
  // Routing metadata comes from the router kernel, which finished before the gate/up kernel
  // passed its own wait; only the SwiGLU outputs need this kernel's wait below.
  const bool active = resolve_slot(a, blockIdx.y, n_slots, true, sl, tok_s, row_s);
  const int row_base = blockIdx.x * kDnRows;
  if (!active || row_base >= sl.nrows) return;
  __syncthreads();
  const int L = shared_slot ? a.S : a.I;        // contraction length
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int ntok = sl.ntok, chunks = L / 8;
  const int r0 = row_base + wid * kDnRowsPerWarp;
  // stream this warp's weight rows first: they do not depend on the gate/up results
  // (contraction <= 1024 elements: each lane holds at most 4 chunks of each of its rows)
  uint4 wv[kDnRowsPerWarp][4];
#pragma unroll
  for (int rr = 0; rr < kDnRowsPerWarp; ++rr) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = q * 32 + lane;
      if (r0 + rr < sl.nrows && c < chunks)
        wv[rr][q] = ld_stream(reinterpret_cast<const uint4*>(sl.w0 + (size_t)(r0 + rr) * L) + c);
    }
  }
  pdl_wait();       // SwiGLU outputs of the gate/up kernel
  pdl_trigger();
  for (int i = threadIdx.x; i < sl.ntok * (L / 4); i += blockDim.x) {
    int j = i / (L / 4), c = i % (L / 4);
    reinterpret_cast<float4*>(hs)[j * (L / 4) + c] =
        __ldcg(reinterpret_cast<const float4*>(a.hd + (size_t)row_s[j] * a.ldh) + c);
  }
  if (!shared_slot && a.acc) {
    for (int j = threadIdx.x; j < sl.ntok; j += blockDim.x)
      wt_s[j] = a.w[a.sorted_pairs[row_s[j]]];
  }
  __syncthreads();
#pragma unroll
  for (int rr = 0; rr < kDnRowsPerWarp; ++rr) {
    const int r = r0 + rr;
    if (r >= sl.nrows) break;
    float acc[kMaxTok];
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) acc[j] = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = q * 32 + lane;
      if (c < chunks) {
        float wf[8];
        bf16x8_to_f32(wv[rr][q], wf);
#pragma unroll
        for (int j = 0; j < kMaxTok; ++j) {
          if (j < ntok) {
            const float4 h0 = reinterpret_cast<const float4*>(hs + j * L)[2 * c];
            const float4 h1 = reinterpret_cast<const float4*>(hs + j * L)[2 * c + 1];
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
    }
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      if (j < ntok) {
        const float y = warp_sum(acc[j]);
        if (lane == 0) {
          if (shared_slot) {
            a.shy[(size_t)tok_s[j] * a.H + r] = y;
          } else if (a.acc) {
            atomicAdd(a.acc + (size_t)tok_s[j] * a.H + r, wt_s[j] * y);
          } else {
            a.yd[(size_t)row_s[j] * a.H + r] = y;
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_decode_gateup(const DecodeArgs& a, cudaStream_t st) {
  const int n_slots = a.te < a.E ? a.te : a.E;
  const int maxrows = a.I > a.S ? a.I : a.S;
  dim3 grid((maxrows + kGuRows - 1) / kGuRows, n_slots + 1);
  const int maxtok = a.N < kMaxTok ? a.N : kMaxTok;
  size_t sm = (size_t)maxtok * a.H * 2;
  if (sm > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(decode_gateup_kernel, grid, dim3(256), sm, st, a, n_slots);
}

cudaError_t launch_decode_down(const DecodeArgs& a, cudaStream_t st) {
  const int n_slots = a.te < a.E ? a.te : a.E;
  dim3 grid((a.H + kDnRows - 1) / kDnRows, n_slots + 1);
  const int maxtok = a.N < kMaxTok ? a.N : kMaxTok;
  const int maxl = a.I > a.S ? a.I : a.S;
  size_t sm = (size_t)maxtok * maxl * 4;
  if (sm > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_down_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(decode_down_kernel, grid, dim3(256), sm, st, a, n_slots);
}

}  // namespace moe
