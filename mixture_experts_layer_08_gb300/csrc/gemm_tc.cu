// Grouped GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// D[rows of expert e, n-tile] = A[rows, K] . B_e[n-tile rows, K]^T over the expert-sorted
// rows, with the epilogue fused: SiLU(gate) * up -> bf16 (gate/up projection), plain bf16
// store (down projection), or fp32 store (router logits). One launch may carry two problems
// (the shared expert's dense FFN and the routed experts), so both fill the same persistent
// grid.
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (`run_routed_grouped_gemm`:
// grouped gate/up GEMM, activation and grouped down GEMM over the rows sorted by expert,
// the sorted result left for the unpermute; `run_shared_expert_prefill`: the shared expert
// as a dense FFN on all rows).
//
// Design (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: A tile 128 x 64 and B tile BN x 64 (bf16, 128-byte swizzle)
//               per stage into a ring of kStages stages. (A 4-row TMA gather straight from
//               the token rows measured 3x slower than reading an expert-sorted copy.)
//   warp 1      allocates TMEM (2 x BN fp32 columns: two accumulators), one lane issues
//               tcgen05.mma (M=128, N=BN, K=16) x 4 per stage and commits stage releases.
//   warps 2-5   epilogue: tcgen05.ld of the finished accumulator (warp w reads TMEM lanes
//               32*(w%4)...), fused activation, masked stores (the down projection's bf16
//               rows staged in shared memory so that every store instruction writes whole
//               128-byte lines); releases the accumulator so the MMA of the next tile overlaps
//               this epilogue.
// Tiles are (m-tile, n-tile) pairs, m-tiles taken from the device-built list of 128-row
// windows of each expert; n is the fastest index so the CTAs working at the same time share
// A rows and the same expert's weights in L2.
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;                 // bf16 elements per 128-byte swizzle row
constexpr int kATileBytes = kBM * 128;  // 16 KB
constexpr int kEpiWarps = 4;
constexpr int kStageRowsBytes = 32 * 128;   // one epilogue warp: 32 rows x 64 bf16 outputs

template <int BN>
struct Cfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kBTileBytes = BN * 128;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes;
  static constexpr int kTmemCols = 2 * BN;
};

// Ring, barrier block (256 B), the epilogue warps' staging rows (bf16 store only), alignment
// slack.
template <int BN, int MODE>
constexpr size_t smem_bytes() {
  return (size_t)Cfg<BN>::kStages * Cfg<BN>::kStageBytes + 256 +
         (MODE == kGemmStoreBF16 ? kEpiWarps * kStageRowsBytes : 0) + 1024;
}

// Per-tile view of the problem it belongs to (selected without dynamic param indexing).
struct Tile {
  int p, e, row0, row1, n, num_kb, b_rows_per_expert;
  void* out;
  int ldo, n_valid;
};

__device__ __forceinline__ int problem_mtiles(const GemmProblem& q) {
  return q.tiles ? (int)q.count->num_mtiles : (q.dense_m + kBM - 1) / kBM;
}

__device__ __forceinline__ void tile_of(const GemmArgs& g, int tot0, int tile, Tile& t) {
  const bool second = tile >= tot0;
  const GemmProblem& q0 = g.p[0];
  const GemmProblem& q1 = g.p[1];
  const int local = second ? tile - tot0 : tile;
  const int n_tiles = second ? q1.n_tiles : q0.n_tiles;
  const int4* tiles = second ? q1.tiles : q0.tiles;
  const int m = local / n_tiles;
  t.p = second ? 1 : 0;
  t.n = local % n_tiles;
  if (tiles) {
    const int4 v = tiles[m];
    t.e = v.x;
    t.row0 = v.y;
    t.row1 = v.z;
  } else {
    t.e = 0;
    t.row0 = m * kBM;
    t.row1 = min(second ? q1.dense_m : q0.dense_m, t.row0 + kBM);
  }
  t.num_kb = second ? q1.num_kb : q0.num_kb;
  t.b_rows_per_expert = second ? q1.b_rows_per_expert : q0.b_rows_per_expert;
  t.out = second ? q1.out : q0.out;
  t.ldo = second ? q1.ldo : q0.ldo;
  t.n_valid = second ? q1.n_valid : q0.n_valid;
}

template <int BN, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a0,
                     const __grid_constant__ CUtensorMap tm_b00,
                     const __grid_constant__ CUtensorMap tm_b01,
                     const __grid_constant__ CUtensorMap tm_a1,
                     const __grid_constant__ CUtensorMap tm_b10,
                     const __grid_constant__ CUtensorMap tm_b11, const GemmArgs g) {
  using C = Cfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = g.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_a0);
    tma_prefetch_desc(&tm_b00);
    if (MODE == kGemmSwiGLU) tma_prefetch_desc(&tm_b01);
    if (g.nprob > 1) {
      tma_prefetch_desc(&tm_a1);
      tma_prefetch_desc(&tm_b10);
      if (MODE == kGemmSwiGLU) tma_prefetch_desc(&tm_b11);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();   // (launched as a programmatic dependent: the previous kernel's results)

  const int tot0 = problem_mtiles(g.p[0]) * g.p[0].n_tiles;
  const int total = tot0 + (g.nprob > 1 ? problem_mtiles(g.p[1]) * g.p[1].n_tiles : 0);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    constexpr int b_rows = MODE == kGemmSwiGLU ? BN / 2 : BN;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      Tile t;
      tile_of(g, tot0, tile, t);
      const CUtensorMap* ma = t.p ? &tm_a1 : &tm_a0;
      const CUtensorMap* mb0 = t.p ? &tm_b10 : &tm_b00;
      const CUtensorMap* mb1 = t.p ? &tm_b11 : &tm_b01;
      const int brow = t.e * t.b_rows_per_expert + t.n * b_rows;
      for (int kb = 0; kb < t.num_kb; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1, hdr)) { ok = false; break; }
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        tma_load_2d(sA + s * kATileBytes, ma, kb * kBK, t.row0, &full[s]);
        tma_load_2d(sB + s * C::kBTileBytes, mb0, kb * kBK, brow, &full[s]);
        if (MODE == kGemmSwiGLU)
          tma_load_2d(sB + s * C::kBTileBytes + (BN / 2) * 128, mb1, kb * kBK, brow, &full[s]);
        ++issued;
        if (++s == S) { s = 0; ph ^= 1; }
      }
    }
    if (!ok) {
      // let the copies already issued land before the CTA can exit
      for (long long i = issued > S ? issued - S : 0; i < issued; ++i)
        mbar_wait(&full[i % S], (uint32_t)((i / S) & 1), nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_make(kBM, BN, 1, 1);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int it = 0;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      Tile t;
      tile_of(g, tot0, tile, t);
      const int acc = it & 1;
      if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, hdr)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d = tmem_base + acc * BN;
      for (int kb = 0; kb < t.num_kb; ++kb) {
        if (!mbar_wait(&full[s], ph, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kATileBytes);
        const uint32_t b0 = smem_u32(sB + s * C::kBTileBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          tc_mma_bf16(d, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                      (kb | k) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
        if (++s == S) { s = 0; ph ^= 1; }
      }
      if (ok) tc_commit(&tfull[acc]);
    }
    // all MMAs of this thread complete before TMEM can be released
    tc_commit(drain);
    mbar_wait(drain, 0, hdr);
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quadrant of this warp
    const int r_local = q * 32 + lane;
    uint8_t* stg = smem + S * C::kStageBytes + 256 + (warp - 2) * kStageRowsBytes;
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      Tile t;
      tile_of(g, tot0, tile, t);
      const int acc = it & 1;
      if (!mbar_wait(&tfull[acc], (it >> 1) & 1, hdr)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      const int row = t.row0 + r_local;
      const bool valid = row < t.row1;
      if (MODE == kGemmSwiGLU) {
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(t.out) + (size_t)row * t.ldo + t.n * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          float gv[32], uv[32];
          tmem_ld32(taddr + c, gv);
          tmem_ld32(taddr + BN / 2 + c, uv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              o.x = pack_bf16x2(silu(gv[8 * v + 0]) * uv[8 * v + 0], silu(gv[8 * v + 1]) * uv[8 * v + 1]);
              o.y = pack_bf16x2(silu(gv[8 * v + 2]) * uv[8 * v + 2], silu(gv[8 * v + 3]) * uv[8 * v + 3]);
              o.z = pack_bf16x2(silu(gv[8 * v + 4]) * uv[8 * v + 4], silu(gv[8 * v + 5]) * uv[8 * v + 5]);
              o.w = pack_bf16x2(silu(gv[8 * v + 6]) * uv[8 * v + 6], silu(gv[8 * v + 7]) * uv[8 * v + 7]);
              dst[v] = o;
            }
          }
        }
      } else if (MODE == kGemmStoreBF16) {
        // 64 output columns at a time through the warp's staging rows: whole 128-byte row
        // segments per store instruction
        uint8_t* obase = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(t.out) +
                                                    (size_t)(t.row0 + q * 32) * t.ldo + t.n * BN);
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          uint4 pk[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[32];
            tmem_ld32(taddr + c + 32 * h, v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              pk[4 * h + j].x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
              pk[4 * h + j].y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
              pk[4 * h + j].z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
              pk[4 * h + j].w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
            }
          }
          warp_store_rows<8>(stg, pk, obase + c * 2, (size_t)t.ldo * 2, t.row1 - t.row0 - q * 32);
        }
      } else {
        float* orow = static_cast<float*>(t.out) + (size_t)row * t.ldo;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(taddr + c, v);
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = t.n * BN + c + j;
              if (col < t.n_valid) orow[col] = v[j];
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, int MODE>
cudaError_t launch_t(const CUtensorMap maps[2][3], const GemmArgs& g, int num_sms,
                     cudaStream_t st) {
  using C = Cfg<BN>;
  auto kern = gemm_bf16_kernel<BN, MODE>;
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(kern), smem_bytes<BN, MODE>());
  if (e != cudaSuccess) return e;
  int max_tiles = g.p[0].max_mtiles * g.p[0].n_tiles;
  if (g.nprob > 1) max_tiles += g.p[1].max_mtiles * g.p[1].n_tiles;
  int grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  const int j = g.nprob > 1 ? 1 : 0;   // unused maps of a one-problem launch repeat problem 0's
  return launch_dependent(kern, dim3(grid), dim3(kThreads), smem_bytes<BN, MODE>(), st, maps[0][0],
                          maps[0][1], maps[0][2], maps[j][0], maps[j][1], maps[j][2], g);
}

}  // namespace

cudaError_t launch_gemm_bf16(int mode, int bn, const CUtensorMap maps[2][3], const GemmArgs& g,
                             int num_sms, cudaStream_t st) {
  if (g.nprob < 1 || g.nprob > 2) return cudaErrorInvalidValue;
  if (bn == 256) {
    if (mode == kGemmSwiGLU) return launch_t<256, kGemmSwiGLU>(maps, g, num_sms, st);
    if (mode == kGemmStoreBF16) return launch_t<256, kGemmStoreBF16>(maps, g, num_sms, st);
  } else if (bn == 128) {
    if (mode == kGemmSwiGLU) return launch_t<128, kGemmSwiGLU>(maps, g, num_sms, st);
    if (mode == kGemmStoreBF16) return launch_t<128, kGemmStoreBF16>(maps, g, num_sms, st);
    if (mode == kGemmStoreF32) return launch_t<128, kGemmStoreF32>(maps, g, num_sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
