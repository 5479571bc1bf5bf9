// Decode chain (few tokens): one persistent, cooperatively launched kernel streams the
// weights of every expert the batch touches -- gate and up rows, then down rows -- reading
// each from HBM once for all the tokens routed to it; the shared expert is one more "slot".
//
// Pages: "spark_model/layers/moe/forward.rs" (`forward`: fused gate/up GEMV for the K routed
// experts plus the shared expert, fused SiLU+down GEMV, weighted sum + sigmoid-gated shared
// blend, all on device with no host synchronisation) and
// "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (token-major gate/up for a few rows,
// routed down projections weighted and FP32-atomic-added into a [N,H] accumulator zeroed
// first, then a finalize that casts to BF16 and blends the shared expert).
//
// Work items are consecutive weight rows of one slot (contiguous in memory). Every block
// (one per SM) owns a contiguous range of gate/up items followed by a contiguous range of
// down items; warp 0 streams them into a shared-memory ring with 1D bulk copies (up to
// ~190 KB in flight per SM) and 16 consumer warps take one weight row each. Gate/up
// consumers write raw gate and up dot products and count the rows done per slot; down
// consumers wait for their slot's count (a bounded spin: all blocks are co-resident), stage
// SiLU(gate)*up in shared memory and dot the down rows against it. The producer keeps
// streaming down weights meanwhile, so the two projections share one pipeline.
#include "kernels.h"

namespace moe {

namespace {

constexpr int kConsumers = 16;       // consumer warps
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kSmemBudget = 222 * 1024;   // dynamic part; + RouteMeta, of the 227 KB allowed
constexpr int kMaxStages = 4;

// Contiguous, balanced share [i0, i1) of `total` items for this block.
__device__ __forceinline__ void item_range(int total, int& i0, int& i1) {
  const long long G = gridDim.x, b = blockIdx.x;
  i0 = (int)((total * b) / G);
  i1 = (int)((total * (b + 1)) / G);
}

// Routing of the batch, copied to shared memory once per block so the streaming loops
// never wait on a dependent global load: expert, first sorted row and row count of every
// active slot, and the token of every sorted row (all < 2^16 on the decode chain).
struct RouteMeta {
  int n_active;
  uint16_t slot_e[kDecodeMaxPairs];
  uint16_t slot_r0[kDecodeMaxPairs];
  uint16_t slot_n[kDecodeMaxPairs];
  uint16_t row_tok[kDecodeMaxPairs];
};

// All threads of the block; routing metadata is read through L2 (an earlier kernel wrote it).
__device__ void load_route_meta(const DecodeArgs& a, RouteMeta& m) {
  const int n_active = (int)__ldcg(&a.hdr->num_active);
  for (int s = threadIdx.x; s < n_active; s += blockDim.x) {
    const int e = (int)__ldcg(a.active + s);
    const int r0 = (int)__ldcg(a.offsets + e);
    m.slot_e[s] = (uint16_t)e;
    m.slot_r0[s] = (uint16_t)r0;
    m.slot_n[s] = (uint16_t)((int)__ldcg(a.offsets + e + 1) - r0);
  }
  for (int r = threadIdx.x; r < a.te; r += blockDim.x)
    m.row_tok[r] = (uint16_t)(__ldcg(a.sorted_pairs + r) / (uint32_t)a.K);
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
// memory). Lane-strided 16-byte chunks.
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

// Dot products of one bf16 weight row (shared memory) with NT fp32 vectors hs[j * L ...]
// (shared memory; rows past `ntok` repeat the last valid one and are discarded).
template <int NT>
__device__ __forceinline__ void row_dots_h(const uint4* w, const float* hs, int L, int ntok,
                                           int lane, float* out) {
  float acc[NT];
  const float4* hr[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    acc[j] = 0.0f;
    hr[j] = reinterpret_cast<const float4*>(hs + (size_t)min(j, ntok - 1) * L);
  }
#pragma unroll 1
  for (int c = lane; c < L / 8; c += 32) {
    float f[8];
    bf16x8_to_f32(w[c], f);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float4 h0 = hr[j][2 * c], h1 = hr[j][2 * c + 1];
      float p0 = f[0] * h0.x, p1 = f[1] * h0.y;
      p0 = fmaf(f[2], h0.z, p0);
      p1 = fmaf(f[3], h0.w, p1);
      p0 = fmaf(f[4], h1.x, p0);
      p1 = fmaf(f[5], h1.y, p1);
      p0 = fmaf(f[6], h1.z, p0);
      p1 = fmaf(f[7], h1.w, p1);
      acc[j] += p0 + p1;
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) out[j] = warp_sum(acc[j]);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct Plan {
  int ri;          // gate/up rows per item (one per consumer warp, <= 16)
  int dr;          // down rows per item (a multiple of 16: each consumer warp takes dr/16)
  int stages;
  int slot_bytes;  // ring slot size
  int xbytes;      // x staging
  int hbytes;      // intermediate staging
};

// x[N,H] -> hd (gate/up dots, rows counted in h_cnt) -> y (down dots), in one launch.
__global__ void __launch_bounds__(kThreads, 1) decode_ffn_kernel(DecodeArgs a, Plan pl) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteMeta meta;
  __shared__ int h_ok;
  const int H = a.H, N = a.N;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);              // [N, H]
  float* hs = reinterpret_cast<float*>(smem + pl.xbytes);                    // [ntok, L]
  uint8_t* ring = smem + pl.xbytes + pl.hbytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)pl.stages * pl.slot_bytes);
  uint64_t* empty = full + kMaxStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stages = pl.stages, ri = pl.ri, dr = pl.dr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    fence_mbarrier_init();
  }
  pdl_trigger();   // the combine kernel may launch and wait for this one
  for (int i = threadIdx.x; i < N * H / 8; i += blockDim.x)
    reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(a.x)[i];
  load_route_meta(a, meta);   // (ends with a block barrier: x is staged too)

  // item spaces: gate/up (per slot the gate rows in chunks of ri, then the up rows) and down
  const int gu_slot = 2 * (a.I / ri);
  const int gu_routed = meta.n_active * gu_slot;
  const int gu_total = gu_routed + (a.S > 0 ? 2 * (a.S / ri) : 0);
  const int dn_slot = H / dr;
  const int dn_routed = meta.n_active * dn_slot;
  const int dn_total = dn_routed + (a.S > 0 ? dn_slot : 0);
  int g0, g1, d0, d1;
  item_range(gu_total, g0, g1);
  item_range(dn_total, d0, d1);
  const int ngu = g1 - g0, nitems = ngu + (d1 - d0);

  if (warp == 0) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int k = 0; k < nitems; ++k, ++issued) {
        const int s = k % stages;
        if (!mbar_wait(&empty[s], ((k / stages) & 1) ^ 1, a.hdr)) { ok = false; break; }
        const __nv_bfloat16* src;
        uint32_t bytes;
        if (k < ngu) {
          const int it = g0 + k;
          bytes = (uint32_t)(ri * H * 2);
          if (it < gu_routed) {
            const int e = meta.slot_e[it / gu_slot];
            const int j = it % gu_slot, half = a.I / ri;
            src = (j < half ? a.wg : a.wu) + ((size_t)e * a.I + (size_t)(j % half) * ri) * H;
          } else {
            const int j = it - gu_routed, half = a.S / ri;
            src = (j < half ? a.sg : a.su) + (size_t)(j % half) * ri * H;
          }
        } else {
          const int it = d0 + (k - ngu);
          if (it < dn_routed) {
            const int e = meta.slot_e[it / dn_slot];
            src = a.wd + ((size_t)e * H + (size_t)(it % dn_slot) * dr) * a.I;
            bytes = (uint32_t)(dr * a.I * 2);
          } else {
            src = a.sd + (size_t)(it - dn_routed) * dr * a.S;
            bytes = (uint32_t)(dr * a.S * 2);
          }
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + (size_t)s * pl.slot_bytes, src, bytes, &full[s]);
      }
      if (!ok)   // let the copies already issued land before the block can exit
        for (int k = issued > stages ? issued - stages : 0; k < issued; ++k)
          mbar_wait(&full[k % stages], (k / stages) & 1, nullptr);
    }
    return;
  }

  // ------------------------------------------------ consumers
  const int cw = warp - 1, ct = threadIdx.x - 32;
  bool live = true;    // false after a timed-out wait: keep pace (barriers), skip the work
  int k = 0;
  // gate/up: hd[row_j, i] = x_j . Wg[i], hd[row_j, ldh + i] = x_j . Wu[i]. Rows written are
  // counted per slot and published (fence, then one atomic) when the slot changes, so no fence
  // sits between an item and the release of its ring stage.
  {
    int cur_slot = -2, ntok = 0, r0 = 0, pend = 0;
    auto publish = [&]() {
      if (pend == 0) return;
      __threadfence();
      __syncwarp();
      if (lane == 0)
        atomicAdd(a.h_cnt + (cur_slot < 0 ? kDecodeMaxPairs : cur_slot), (uint32_t)pend);
      pend = 0;
    };
    for (; k < ngu; ++k) {
      const int s = k % stages, it = g0 + k;
      const bool routed_item = it < gu_routed;
      const int slot = routed_item ? it / gu_slot : -1;
      const int j = routed_item ? it % gu_slot : it - gu_routed;
      const int half = (routed_item ? a.I : a.S) / ri;
      const int col = (j < half ? 0 : a.ldh) + (j % half) * ri + cw;   // hd column
      if (slot != cur_slot) {
        publish();
        cur_slot = slot;
        ntok = slot_rows(a, meta, slot, r0);
      }
      if (live && !mbar_wait(&full[s], (k / stages) & 1, a.hdr)) live = false;
      if (live && cw < ri) {
        const uint4* w = reinterpret_cast<const uint4*>(ring + (size_t)s * pl.slot_bytes +
                                                        (size_t)cw * H * 2);
        // groups of up to 4 tokens: each group's results are stored before the next
        for (int j0 = 0; j0 < ntok; j0 += 4) {
          const int nt = min(4, ntok - j0);
          int tg[4];        // the group's tokens; past nt, repeats of a valid one
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
        ++pend;
      }
      __syncwarp();
      if (lane == 0 && live) mbar_arrive(&empty[s]);
    }
    publish();
  }
  // down: y_j[r] = h_j . Wd[r], h_j = SiLU(gate_j) * up_j
  {
    int cur_slot = -2, ntok = 0, r0 = 0, L = a.I;
    for (; k < nitems; ++k) {
      const int s = k % stages, it = d0 + (k - ngu);
      const bool shared_item = it >= dn_routed;
      const int slot = shared_item ? -1 : it / dn_slot;
      const int rbase = (shared_item ? it - dn_routed : it % dn_slot) * dr;
      if (slot != cur_slot) {
        // every consumer warp walks the same items, so they all change slot together
        named_sync(1, 32 * kConsumers);
        cur_slot = slot;
        ntok = slot_rows(a, meta, slot, r0);
        L = shared_item ? a.S : a.I;
        if (ct == 0) {
          // all 2L gate/up rows of this slot written (bounded wait; blocks are co-resident)
          const uint32_t* cnt = a.h_cnt + (slot < 0 ? kDecodeMaxPairs : slot);
          int okv = live ? 1 : 0;
          if (okv && ld_acquire(cnt) < (uint32_t)(2 * L)) {
            const long long t0 = clock64();
            while (ld_acquire(cnt) < (uint32_t)(2 * L)) {
              if (clock64() - t0 > kSpinLimitCycles) {
                report_timeout(a.hdr);
                okv = 0;
                break;
              }
              __nanosleep(64);
            }
          }
          h_ok = okv;
        }
        named_sync(1, 32 * kConsumers);
        live = h_ok != 0;
        if (live) {
          for (int i = ct; i < ntok * L; i += 32 * kConsumers) {
            const int jj = i / L, c = i % L;
            const float* hr = a.hd + (size_t)(r0 + jj) * (2 * a.ldh);
            hs[jj * L + c] = silu(__ldcg(hr + c)) * __ldcg(hr + a.ldh + c);
          }
        }
        named_sync(1, 32 * kConsumers);
      }
      if (live && !mbar_wait(&full[s], (k / stages) & 1, a.hdr)) live = false;
      if (live) {
        const uint8_t* stage = ring + (size_t)s * pl.slot_bytes;
        for (int rl = cw; rl < dr; rl += kConsumers) {
          const uint4* wr = reinterpret_cast<const uint4*>(stage + (size_t)rl * L * 2);
          const int r = rbase + rl;
          for (int j0 = 0; j0 < ntok; j0 += 4) {
            const int nt = min(4, ntok - j0);
            float acc[4];
            const float* hg = hs + (size_t)j0 * L;
            if (nt == 1) row_dots_h<1>(wr, hg, L, nt, lane, acc);
            else if (nt == 2) row_dots_h<2>(wr, hg, L, nt, lane, acc);
            else row_dots_h<4>(wr, hg, L, nt, lane, acc);
            if (lane < nt) {
              float y = acc[0];
#pragma unroll
              for (int q = 1; q < 4; ++q)
                if (lane == q) y = acc[q];
              const int jj = j0 + lane, row = r0 + jj;
              if (shared_item) {
                a.shy[(size_t)jj * H + r] = y;
              } else if (a.acc) {
                atomicAdd(a.acc + (size_t)meta.row_tok[row] * H + r,
                          a.w[__ldcg(a.sorted_pairs + row)] * y);
              } else {
                a.yd[(size_t)row * H + r] = y;
              }
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

cudaError_t launch_decode_ffn(const DecodeArgs& a, cudaStream_t st) {
  if (a.te > kDecodeMaxPairs || a.N > kDecodeMaxTokens || a.H % 16 || !a.h_cnt)
    return cudaErrorInvalidValue;
  const int L = a.I > a.S ? a.I : a.S;
  Plan pl{};
  pl.xbytes = (a.N * a.H * 2 + 127) & ~127;
  pl.hbytes = (a.N * L * 4 + 127) & ~127;
  auto slot = [&](const Plan& p) {
    const int gu = p.ri * a.H * 2, dn = p.dr * L * 2;
    return gu > dn ? gu : dn;
  };
  // the largest items (<= 16 gate/up rows, <= 32 down rows) that keep 3 ring stages
  static const int kChoices[][2] = {{16, 32}, {16, 16}, {8, 16}, {4, 16}, {2, 16}, {1, 16}};
  bool found = false;
  for (const auto& ch : kChoices) {
    pl.ri = ch[0];
    pl.dr = ch[1];
    if (a.I % pl.ri || (a.S && a.S % pl.ri) || a.H % pl.dr) continue;
    if ((size_t)pl.xbytes + pl.hbytes + 3 * (size_t)slot(pl) + 1024 <= (size_t)kSmemBudget) {
      found = true;
      break;
    }
  }
  if (!found) return cudaErrorInvalidValue;
  pl.slot_bytes = slot(pl);
  pl.stages = (int)(((size_t)kSmemBudget - 1024 - pl.xbytes - pl.hbytes) / pl.slot_bytes);
  if (pl.stages > kMaxStages) pl.stages = kMaxStages;
  if (pl.stages < 1 || a.I % pl.ri || (a.S && a.S % pl.ri) || a.H % pl.dr)
    return cudaErrorInvalidValue;
  const size_t sm = (size_t)pl.xbytes + pl.hbytes + (size_t)pl.stages * pl.slot_bytes +
                    2 * kMaxStages * 8;
  cudaError_t e = cudaFuncSetAttribute(decode_ffn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  // the down consumers wait on other blocks' gate/up rows: all blocks must be resident
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_ffn_kernel, kThreads, sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel, a, pl);
}

}  // namespace moe
