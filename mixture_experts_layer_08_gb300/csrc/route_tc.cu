// Fused router for many tokens: the router GEMM on the tensor cores with fp32 scoring, top-K
// and renormalisation in the same launch.
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (the router gate GEMM of the
// prefill forward followed by `moe_topk_softmax_batched` with `norm_topk_prob`) and
// "spark_model/layers/moe/forward.rs" (`forward`: softmax + correction bias for the selection,
// identity experts folded into zero_accum). The decode page rejects a single-CTA fused
// gate+top-K for wide routers as too slow; here the contraction of every 128-token tile is
// split over a cluster of CTAs instead.
//
// Design (grid = ks x ceil(N/128), clusters of ks CTAs along x, 1024 threads per CTA):
//   Each CTA of a cluster owns H/ks of the contraction of one 128-token tile.
//   warp 0      TMA producer: x tile 128 x 64 and router tile R x 64 (bf16, 128-byte swizzle)
//               per stage.
//   warp 1      allocates TMEM (R fp32 columns rounded up to a power of two), one lane issues
//               tcgen05.mma M=128, N=R (two MMAs when R > 256), K=16 x 4 per stage.
//   all warps   once every CTA of the cluster has finished its MMAs (cluster barrier: the
//               partial buffers overlap the stage rings), push the partial logits TMEM ->
//               the shared memory of the CTA that finishes those rows (CTA `rank` owns rows
//               [rank*128/ks, (rank+1)*128/ks); warp w reads lane quadrant w%4, 16 columns at a
//               time; remote stores, no round trip), cluster barrier, sum the ks
//               partials in slot order (the result does not depend on timing), write the fp32
//               logits, then one warp per token: scores, top-K, weights (the scratch rows are
//               the partial slots the sum has freed, so ks >= 2).
#include "kernels.h"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kRtThreads = 1024;
constexpr int kRtWarps = kRtThreads / 32;
constexpr int kRtBM = 128;
constexpr int kRtATile = kRtBM * 128;   // 16 KB: 128 rows of 64 bf16
constexpr int kRtMaxStages = 8;
constexpr int kRtStageBudget = 192 * 1024;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float x, float y, float z, float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y),
               "f"(z), "f"(w)
               : "memory");
}

struct RtGeom {
  int ks;            // CTAs per cluster (contraction split)
  int kb_per;        // 64-wide contraction blocks per CTA
  int nst;           // pipeline stages
  int rb;            // router rows per TMA box
  int stage_bytes;
  int part_ld;       // fp32 row stride of the partial logits in shared memory
  int region;        // bytes of the stage ring / partial buffer (they overlap)
  int tmem_cols;
  size_t smem;
};

__host__ __device__ inline int rt_pow2_cols(int R) {
  int c = 32;
  while (c < R) c <<= 1;
  return c;
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_topk_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_w, const RouteArgs a,
                          const RtGeom geo) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int R = a.R;
  const int nst = geo.nst;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + geo.region);
  uint64_t* empty = full + kRtMaxStages;
  uint64_t* done = empty + kRtMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  float* part = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int m0 = blockIdx.y * kRtBM;
  const int kb0 = (int)rank * geo.kb_per;
  WsHeader* hdr = a.hdr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, geo.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    long long issued = 0;
    bool ok = true;
    for (int kb = 0; kb < geo.kb_per; ++kb) {
      const int s = kb % nst;
      const uint32_t ph = (uint32_t)((kb / nst) & 1);
      if (!mbar_wait(&empty[s], ph ^ 1, hdr)) { ok = false; break; }
      uint8_t* st = smem + s * geo.stage_bytes;
      mbar_arrive_expect_tx(&full[s], (uint32_t)geo.stage_bytes);
      tma_load_2d(st, &tm_x, (kb0 + kb) * 64, m0, &full[s]);
      for (int r0 = 0; r0 < R; r0 += geo.rb)
        tma_load_2d(st + kRtATile + r0 * 128, &tm_w, (kb0 + kb) * 64, r0, &full[s]);
      ++issued;
    }
    if (!ok) {
      // let the copies already issued land before the CTA can exit
      for (long long i = issued > nst ? issued - nst : 0; i < issued; ++i)
        mbar_wait(&full[i % nst], (uint32_t)((i / nst) & 1), nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    for (int kb = 0; kb < geo.kb_per; ++kb) {
      const int s = kb % nst;
      if (!mbar_wait(&full[s], (uint32_t)((kb / nst) & 1), hdr)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + s * geo.stage_bytes);
      const uint32_t b0 = a0 + kRtATile;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        for (int n0 = 0; n0 < R; n0 += 256) {
          const int nn = R - n0 < 256 ? R - n0 : 256;
          tc_mma_bf16(tmem_base + n0, sdesc_k_sw128(a0 + k * 32),
                      sdesc_k_sw128(b0 + n0 * 128 + k * 32), idesc_make(kRtBM, nn, 1, 1),
                      (kb | k) != 0 ? 1u : 0u);
        }
      }
      tc_commit(&empty[s]);
    }
    // `done` completes once every MMA above has (or at once when none was issued)
    tc_commit(done);
  }

  // the producer and MMA warps' other lanes wait here (not spinning beside their lane 0)
  __syncwarp();

  // ------------------------------------------------ partial logits TMEM -> owner CTA
  // Row `row` of the tile is finished by CTA row / tr; this CTA's partial of it lands in slot
  // `rank` of that CTA's buffer (rows [rank*tr, (rank+1)*tr)). Remote stores: no round trip.
  // The buffer overlaps the stage ring, so the pushes wait for every CTA's MMAs to finish.
  const int tr = kRtBM / geo.ks;           // token rows each CTA finishes
  const int ld = geo.part_ld;
  const int t0 = m0 + (int)rank * tr;
  const bool have = __all_sync(0xffffffffu, mbar_wait(done, 0, hdr));
  tc_fence_after();
  cluster_arrive();
  cluster_wait();
  __syncwarp();   // tcgen05.ld is warp-collective: the lanes leave the barrier together
  if (have) {
    const uint32_t part_s = smem_u32(part);
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t owner = (uint32_t)(row / tr);
    const uint32_t dst_row = rank * (uint32_t)tr + (uint32_t)(row % tr);
    for (int c = (warp >> 2) * 16; c < R; c += 16 * (kRtWarps / 4)) {
      float v[16];
      tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + c, v);
      const uint32_t dst =
          dsmem_addr(part_s + (dst_row * (uint32_t)ld + (uint32_t)c) * 4u, owner);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_dsmem_f4(dst + 16u * j, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, geo.tmem_cols);
  }
  // every partial has landed in its owner's buffer
  cluster_arrive();
  cluster_wait();

  // ------------------------------------------------ sum of the ks partials, slot order
  const int c4n = R / 4;
  for (int i = threadIdx.x; i < tr * c4n; i += kRtThreads) {
    const int lr = i / c4n;
    const int c4 = i % c4n;
    float4 acc = *reinterpret_cast<const float4*>(part + (size_t)lr * ld + c4 * 4);
    for (int c = 1; c < geo.ks; ++c) {
      const float4 v =
          *reinterpret_cast<const float4*>(part + ((size_t)c * tr + lr) * ld + c4 * 4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int t = t0 + lr;
    if (t < a.N) reinterpret_cast<float4*>(a.logits + (size_t)t * R)[c4] = acc;
  }
  __syncthreads();   // the logits rows are complete (and slots 1.. are free: the scratch)

  // ------------------------------------------------ scoring + top-K, one warp per token
  float* scratch = part + (size_t)tr * ld + (size_t)warp * 2 * R;
  for (int lr = warp; lr < tr; lr += kRtWarps) {
    const int t = t0 + lr;
    if (t >= a.N) break;
    route_token_warp(a.logits + (size_t)t * R, a.logit_bias, a.corr_bias, R, a.E, a.K,
                     a.scoring, a.norm, a.scale,
                     a.forced ? a.forced + (size_t)t * a.K : nullptr, scratch, scratch + R,
                     a.idx + (size_t)t * a.K, a.w + (size_t)t * a.K, a.zsum + t, nullptr);
  }
}

bool rt_geometry(int N, int H, int R, int num_sms, RtGeom* g) {
  if (R < 32 || R > 384 || R % 32 != 0 || H % 64 != 0) return false;
  if (R > 256 && R % 128 != 0) return false;
  const int mt = (N + kRtBM - 1) / kRtBM;
  const int nkb = H / 64;
  int ks = 1;
  while (ks < 8 && (long long)mt * ks * 2 <= num_sms && nkb % (ks * 2) == 0) ks *= 2;
  g->ks = ks;
  g->kb_per = nkb / ks;
  g->rb = R <= 256 ? R : 128;
  g->stage_bytes = kRtATile + R * 128;
  int nst = kRtStageBudget / g->stage_bytes;
  if (nst > kRtMaxStages) nst = kRtMaxStages;
  if (nst > g->kb_per) nst = g->kb_per;
  if (nst < 1) return false;
  g->nst = nst;
  g->part_ld = R + 4;
  const int ring = nst * g->stage_bytes;
  const int part = kRtBM * g->part_ld * 4;
  g->region = ((ring > part ? ring : part) + 7) & ~7;
  g->tmem_cols = rt_pow2_cols(R);
  // scratch of the per-token routing (two rows of R floats per warp) in the slot rows the
  // sum frees: needs ks >= 2
  if ((kRtBM - kRtBM / ks) * g->part_ld < kRtWarps * 2 * R) return false;
  g->smem = (size_t)g->region + 1024 + (2 * kRtMaxStages + 2) * 8;
  return g->smem <= 227 * 1024;
}

}  // namespace

bool router_topk_tc_supported(int N, int H, int R, int num_sms) {
  RtGeom g;
  return rt_geometry(N, H, R, num_sms, &g);
}

cudaError_t launch_router_topk_tc(const RouteArgs& a, const CUtensorMap& tm_x,
                                  const CUtensorMap& tm_w, int num_sms, cudaStream_t st) {
  RtGeom geo;
  if (!rt_geometry(a.N, a.H, a.R, num_sms, &geo)) return cudaErrorInvalidValue;
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(router_topk_tc_kernel), geo.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(geo.ks, (a.N + kRtBM - 1) / kRtBM, 1);
  cfg.blockDim = dim3(kRtThreads, 1, 1);
  cfg.dynamicSmemBytes = geo.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = geo.ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_topk_tc_kernel, tm_x, tm_w, a, geo);
}

}  // namespace moe
