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
// Both kernels are persistent (one block per SM) and split the work into items: consecutive
// weight rows of one slot, contiguous in memory. Warp 0 streams items into a shared-memory
// ring with 1D bulk copies (up to ~200 KB in flight per SM, enough to keep HBM busy);
// 16 consumer warps take one weight row each per item, with the inner loop specialised on
// the slot's token count, so enough independent warps hide the arithmetic latency. The gate
// kernel writes raw gate and up dot products; the down kernel forms SiLU(gate) * up when it
// stages a slot's intermediate vectors in shared memory. Each block owns a contiguous range
// of items, so a slot changes rarely within a block.
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxTok = 16;          // tokens per expert the decode chain handles
constexpr int kConsumers = 16;       // consumer warps
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kSmemBudget = 212 * 1024;   // dynamic part; + RouteMeta, of the 227 KB allowed
constexpr int kMaxStages = 4;
constexpr int kMaxPairs = 512;       // N * K of the decode chain (16 tokens x top-32)
constexpr int kDownRows = 32;        // down-projection rows per item (2 per consumer warp)

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

// Tokens of slot `slot` (-1: the shared expert): first intermediate row and count.
__device__ __forceinline__ int slot_rows(const DecodeArgs& a, const RouteMeta& m, int slot,
                                         int& r0) {
  if (slot < 0) {
    r0 = a.te;
    return a.N;
  }
  r0 = m.slot_r0[slot];
  return m.slot_n[slot];
}

__device__ __forceinline__ int token_of_row(const DecodeArgs& a, const RouteMeta& m, int row) {
  return row >= a.te ? row - a.te : m.row_tok[row];
}

// Dot products of one bf16 weight row (shared memory) with NT bf16 token rows of x (shared
// memory); only the first `ntok` results are meaningful. Lane-strided 16-byte chunks.
template <int NT>
__device__ __forceinline__ void row_dots(const uint4* w, const __nv_bfloat16* xs, int H,
                                         const int* tk, int lane, float* out) {
  float acc[NT];
  const uint4* xr[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    acc[j] = 0.0f;
    xr[j] = reinterpret_cast<const uint4*>(xs + (size_t)tk[j] * H);
  }
  for (int c = lane; c < H / 8; c += 32) {
    float wf[8];
    bf16x8_to_f32(w[c], wf);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float xf[8];
      bf16x8_to_f32(xr[j][c], xf);
      float p0 = wf[0] * xf[0], p1 = wf[1] * xf[1];
      p0 = fmaf(wf[2], xf[2], p0);
      p1 = fmaf(wf[3], xf[3], p1);
      p0 = fmaf(wf[4], xf[4], p0);
      p1 = fmaf(wf[5], xf[5], p1);
      p0 = fmaf(wf[6], xf[6], p0);
      p1 = fmaf(wf[7], xf[7], p1);
      acc[j] += p0 + p1;
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) out[j] = warp_sum(acc[j]);
}

// Dot products of two bf16 weight rows (shared memory) with NT fp32 vectors hs[j * L ...]
// (shared memory; rows past `ntok` repeat the last valid one and are discarded). Each h chunk
// is loaded once for both rows. out0/out1: results of row 0 / row 1.
template <int NT>
__device__ __forceinline__ void row2_dots_h(const uint4* w0, const uint4* w1, const float* hs,
                                            int L, int ntok, int lane, float* out0,
                                            float* out1) {
  float a0[NT], a1[NT];
  const float4* hr[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    a0[j] = a1[j] = 0.0f;
    hr[j] = reinterpret_cast<const float4*>(hs + (size_t)min(j, ntok - 1) * L);
  }
#pragma unroll 1
  for (int c = lane; c < L / 8; c += 32) {
    float f0[8], f1[8];
    bf16x8_to_f32(w0[c], f0);
    bf16x8_to_f32(w1[c], f1);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float4 h0 = hr[j][2 * c], h1 = hr[j][2 * c + 1];
      const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      float p0 = f0[0] * hv[0], p1 = f1[0] * hv[0];
#pragma unroll
      for (int q = 1; q < 8; ++q) {
        p0 = fmaf(f0[q], hv[q], p0);
        p1 = fmaf(f1[q], hv[q], p1);
      }
      a0[j] += p0;
      a1[j] += p1;
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    out0[j] = warp_sum(a0[j]);
    out1[j] = warp_sum(a1[j]);
  }
}

// ------------------------------------------------------------------ gate/up

// hd[row_j, i] = x_j . Wg[i] and hd[row_j, ldh + i] = x_j . Wu[i] for every token j of the
// slot. Item = `ri` consecutive rows of one slot's gate or up matrix.
__global__ void __launch_bounds__(kThreads, 1)
    decode_gateup_kernel(DecodeArgs a, int ri, int stages, int item_bytes, int xbytes) {
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
  pdl_wait();       // routing of the router kernel
  pdl_trigger();    // the down projection may start streaming its weights
  load_route_meta(a, meta);   // (ends with a block barrier: x is staged too)

  // items per slot: the gate rows in chunks of ri, then the up rows
  const int per_slot = 2 * (a.I / ri);
  const int routed = meta.n_active * per_slot;
  const int total = routed + (a.S > 0 ? 2 * (a.S / ri) : 0);
  int i0, i1;
  item_range(total, i0, i1);
  const uint32_t bytes = (uint32_t)(ri * H * 2);

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int it = i0; it < i1; ++it, ++issued) {
        const int k = it - i0, s = k % stages;
        if (!mbar_wait(&empty[s], ((k / stages) & 1) ^ 1, a.hdr)) { ok = false; break; }
        const __nv_bfloat16* src;
        if (it < routed) {
          const int e = meta.slot_e[it / per_slot];
          const int j = it % per_slot, half = a.I / ri;
          src = (j < half ? a.wg : a.wu) + ((size_t)e * a.I + (size_t)(j % half) * ri) * H;
        } else {
          const int j = it - routed, half = a.S / ri;
          src = (j < half ? a.sg : a.su) + (size_t)(j % half) * ri * H;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + (size_t)s * item_bytes, src, bytes, &full[s]);
      }
      if (!ok)   // let the copies already issued land before the block can exit
        for (int k = issued > stages ? issued - stages : 0; k < issued; ++k)
          mbar_wait(&full[k % stages], (k / stages) & 1, nullptr);
    }
  } else {
    const int cw = warp - 1;
    int cur_slot = -2, ntok = 0, r0 = 0;
    for (int it = i0; it < i1; ++it) {
      const int k = it - i0, s = k % stages;
      const bool routed_item = it < routed;
      const int slot = routed_item ? it / per_slot : -1;
      const int j = routed_item ? it % per_slot : it - routed;
      const int half = (routed_item ? a.I : a.S) / ri;
      const int col = (j < half ? 0 : a.ldh) + (j % half) * ri + cw;   // hd column
      if (slot != cur_slot) {
        cur_slot = slot;
        ntok = slot_rows(a, meta, slot, r0);
      }
      if (!mbar_wait(&full[s], (k / stages) & 1, a.hdr)) break;
      if (cw < ri) {
        const uint4* w = reinterpret_cast<const uint4*>(ring + (size_t)s * item_bytes +
                                                        (size_t)cw * H * 2);
        // groups of up to 4 tokens: each group's results are stored before the next
        for (int j0 = 0; j0 < ntok; j0 += 4) {
          const int nt = min(4, ntok - j0);
          int tg[4];          // the group's tokens; past ntok, repeats of a valid one
#pragma unroll
          for (int u = 0; u < 4; ++u) tg[u] = token_of_row(a, meta, r0 + j0 + min(u, nt - 1));
          float d[4];
          if (nt == 1) row_dots<1>(w, xs, H, tg, lane, d);
          else if (nt == 2) row_dots<2>(w, xs, H, tg, lane, d);
          else row_dots<4>(w, xs, H, tg, lane, d);
          if (lane < nt) {
            float v = d[0];
#pragma unroll
            for (int q = 1; q < 4; ++q)
              if (lane == q) v = d[q];
            a.hd[(size_t)(r0 + j0 + lane) * (2 * a.ldh) + col] = v;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// ------------------------------------------------------------------ down

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// y_j[r] = h_j . Wd[r] for every token j of the slot, h_j = SiLU(gate_j) * up_j. Item =
// kDownRows consecutive rows of Wd_e (or of the shared down weights); routed results go to
// yd, or are weighted and atomically added into acc; shared results go to shy.
__global__ void __launch_bounds__(kThreads, 1)
    decode_down_kernel(DecodeArgs a, int stages, int item_bytes, int hbytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteMeta meta;
  float* hs = reinterpret_cast<float*>(smem);                  // [ntok, L] of the current slot
  uint8_t* ring = smem + hbytes;
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
  // consumers read the gate/up results and wait for them.
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
    pdl_wait();     // gate/up results of the previous kernel
    pdl_trigger();
    const int cw = warp - 1, ct = threadIdx.x - 32;
    int cur_slot = -2, ntok = 0, r0 = 0, L = a.I;
    bool live = true;   // false after a timed-out wait: keep pace (barriers), skip the work
    for (int it = i0; it < i1; ++it) {
      const int k = it - i0, s = k % stages;
      const bool shared_item = it >= routed;
      const int slot = shared_item ? -1 : it / per_slot;
      const int rbase = (shared_item ? it - routed : it % per_slot) * kDownRows;
      if (slot != cur_slot) {
        // every consumer warp walks the same items, so they all change slot together
        named_sync(1, 32 * kConsumers);
        cur_slot = slot;
        ntok = slot_rows(a, meta, slot, r0);
        L = shared_item ? a.S : a.I;
        for (int i = ct; i < ntok * L; i += 32 * kConsumers) {
          const int j = i / L, c = i % L;
          const float* hr = a.hd + (size_t)(r0 + j) * (2 * a.ldh);
          hs[j * L + c] = silu(__ldcg(hr + c)) * __ldcg(hr + a.ldh + c);
        }
        named_sync(1, 32 * kConsumers);
      }
      if (live && !mbar_wait(&full[s], (k / stages) & 1, a.hdr)) live = false;
      if (live) {
        const uint8_t* stage = ring + (size_t)s * item_bytes;
        static_assert(kDownRows == 2 * kConsumers, "two down rows per consumer warp");
        const int rl = 2 * cw;
        const uint4* w0 = reinterpret_cast<const uint4*>(stage + (size_t)rl * L * 2);
        const uint4* w1 = reinterpret_cast<const uint4*>(stage + (size_t)(rl + 1) * L * 2);
        // groups of up to 4 tokens: each group's results are stored before the next
        for (int j0 = 0; j0 < ntok; j0 += 4) {
          const int nt = min(4, ntok - j0);
          float y0[4], y1[4];
          const float* hg = hs + (size_t)j0 * L;
          if (nt == 1) row2_dots_h<1>(w0, w1, hg, L, nt, lane, y0, y1);
          else if (nt == 2) row2_dots_h<2>(w0, w1, hg, L, nt, lane, y0, y1);
          else row2_dots_h<4>(w0, w1, hg, L, nt, lane, y0, y1);
          if (lane < 2 * nt) {
            // lanes 0..nt-1: row rl for token j0+lane; lanes nt..2nt-1: row rl+1
            const int q = lane < nt ? lane : lane - nt;
            float y = 0.0f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (q == u) y = lane < nt ? y0[u] : y1[u];
            const int r = rbase + rl + (lane < nt ? 0 : 1);
            const int j = j0 + q, row = r0 + j;
            if (shared_item) {
              a.shy[(size_t)j * H + r] = y;
            } else if (a.acc) {
              const int t = meta.row_tok[row];
              atomicAdd(a.acc + (size_t)t * H + r, a.w[__ldcg(a.sorted_pairs + row)] * y);
            } else {
              a.yd[(size_t)row * H + r] = y;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0 && live) mbar_arrive(&empty[s]);
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
  // rows per item: the most (<= 16, one per consumer warp) that keep 3 stages in budget
  int ri = kConsumers;
  while (ri > 1 && (a.I % ri || (a.S && a.S % ri) ||
                    (size_t)xbytes + 3 * (size_t)ri * 2 * a.H + 1024 > (size_t)kSmemBudget))
    ri >>= 1;
  const int item = ri * 2 * a.H;
  int stages = (kSmemBudget - 1024 - xbytes) / item;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 1) return cudaErrorInvalidValue;
  const size_t sm = (size_t)xbytes + (size_t)stages * item + 2 * kMaxStages * 8;
  cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_gateup_kernel, dim3(sm_count()), dim3(kThreads), sm, st, a, ri,
                          stages, item, xbytes);
}

cudaError_t launch_decode_down(const DecodeArgs& a, cudaStream_t st) {
  if (a.H % kDownRows || a.te > kMaxPairs) return cudaErrorInvalidValue;
  const int L = a.I > a.S ? a.I : a.S;
  const int maxtok = a.N < kMaxTok ? a.N : kMaxTok;
  const int hbytes = (maxtok * L * 4 + 127) & ~127;
  const int item = kDownRows * L * 2;
  int stages = (kSmemBudget - 1024 - hbytes) / item;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 1) return cudaErrorInvalidValue;
  const size_t sm = (size_t)hbytes + (size_t)stages * item + 2 * kMaxStages * 8;
  cudaError_t e = cudaFuncSetAttribute(decode_down_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_down_kernel, dim3(sm_count()), dim3(kThreads), sm, st, a, stages,
                          item, hbytes);
}

}  // namespace moe
