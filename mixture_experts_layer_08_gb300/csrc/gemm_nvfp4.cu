// Grouped GEMM with NVFP4 expert weights on the 5th-generation tensor cores (sm_103a).
//
// D[rows of expert e, n-tile] = A[rows, K] . dequant(B_e)[n-tile rows, K]^T over the
// expert-sorted rows, where B is packed E2M1 codes (two per byte, element 2j in the low
// nibble) with one E4M3 scale per 16 elements along K and one fp32 scale2 per expert
// matrix. Epilogue: scale2 on the fp32 accumulators, then SiLU(gate) * up to f16 (gate/up),
// or a bf16 store (down).
//
// Pages: "spark_model/layers/moe/forward.rs" (NVFP4 arm of the decode forward: packed expert
// weights with a per-group scale table and one scale2 value per expert matrix,
// `moe_expert_gate_up_shared` / `moe_expert_silu_down_shared`) and
// "metrale_model_layers/layers/moe/forward_prefill.rs" (`run_routed_grouped_gemm` over the
// expert-sorted rows).
//
// The block-scaled tcgen05 MMA kinds take E4M3 scales only with both operands in FP4
// (kind::mxf4nvf4), and an FP8 x FP4 product (kind::mxf8f6f4) only with power-of-two scales.
// The activations keep 16 bits here (the pages' w4a16), so the weights are dequantised in
// shared memory instead, exactly: an E2M1 value times an E4M3 scale has at most 5 significant
// bits and lies in [2^-10, 2688], so it is an f16 (and the hardware converts both formats to
// f16 in one instruction per pair). The MMA is kind::f16 with f16 operands: the activations
// are the gathered token rows (or the SwiGLU intermediate) in f16, exact for the bf16 inputs
// in f16's normal range. HBM carries 0.5 + 1/16 bytes per weight.
//
// Design (one persistent CTA per SM, 448 threads; a ring of 4 loads and a ring of 3
// converted B tiles):
//   warp 0      TMA producer, per step: the A tile 128 x 64 (f16, 128-byte swizzle), the
//               packed codes of the BN weight rows (BN x 32 bytes) and their scale codes
//               (BN x 16 bytes: the 4 groups of this step and of the 3 steps after it,
//               reloaded with each step so the box stays 16 bytes wide), all completing on
//               the load slot's barrier.
//   warp 1      TMEM allocation and the MMA issuer (M=128, N=BN, K=16 x 4 per step); each
//               step's commit frees its load slot and its B slot.
//   warps 2-5   epilogue (TMEM lane quadrant warp % 4): scale2, then SwiGLU or bf16 store.
//   warps 6-13  converters: one weight row per thread, 8 chunks of 8 elements each: 4 code
//               bytes -> 4 f16 pairs (cvt e2m1x2), times the group's scale (exact), one
//               16-byte store into the 128-byte-swizzled B tile; then a proxy fence and one
//               arrival per warp on the B slot's barrier, which the MMA waits on (the
//               converters saw the load -- the A tile too -- land first).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kNvThreads = 448;
constexpr int kNvConvWarps = 8;
constexpr int kNvConvBase = 192;          // first converter thread
constexpr int kNvBM = 128;
constexpr int kNvATile = kNvBM * 128;     // 16 KB

template <int BN>
struct NvCfg {
  static constexpr int kStages = 4;     // load ring: A tile + codes + scale codes
  static constexpr int kBStages = 3;    // converted B tiles
  static constexpr int kBTile = BN * 128;   // bf16, 64 elements per row
  static constexpr int kCTile = BN * 32;    // packed codes, 64 elements per row
  static constexpr int kSTile = BN * 16;    // scale codes, 16 groups per row
  static constexpr int kTmemCols = 2 * BN;
  static constexpr size_t kRingBytes =
      (size_t)kStages * (kNvATile + kCTile + kSTile) + (size_t)kBStages * kBTile;
};

constexpr int kNvStageRows = 32 * 128;   // bf16 store: one epilogue warp's staging rows

// Rings, barrier block (256 B), the down projection's staging rows, alignment slack.
template <int BN, int MODE>
constexpr size_t nv_smem_bytes() {
  return NvCfg<BN>::kRingBytes + 256 + (MODE == kGemmSwiGLU ? 0 : 4 * kNvStageRows) + 1024;
}

struct NvTile {
  int e, row0, row1, n;
};

__device__ __forceinline__ void nv_tile_of(const NvGemmArgs& g, int tile, NvTile& t) {
  const int m = tile / g.n_tiles;
  t.n = tile % g.n_tiles;
  const int4 v = g.tiles[m];
  t.e = v.x;
  t.row0 = v.y;
  t.row1 = v.z;
}

template <int BN, int MODE>
__global__ void __launch_bounds__(kNvThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_c0,
                      const __grid_constant__ CUtensorMap tm_c1,
                      const __grid_constant__ CUtensorMap tm_s0,
                      const __grid_constant__ CUtensorMap tm_s1, const NvGemmArgs g) {
  using C = NvCfg<BN>;
  constexpr int S = C::kStages;
  constexpr int SB = C::kBStages;
  constexpr bool kGlu = MODE == kGemmSwiGLU;
  constexpr int b_rows = kGlu ? BN / 2 : BN;   // rows per weight matrix in one tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kNvATile;
  uint8_t* sC = sB + SB * C::kBTile;
  uint8_t* sS = sC + S * C::kCTile;
  uint64_t* lfull = reinterpret_cast<uint64_t*>(sS + S * C::kSTile);   // load landed
  uint64_t* lempty = lfull + S;      // load slot free (its MMA done)
  uint64_t* bfull = lempty + S;      // B tile converted
  uint64_t* bempty = bfull + SB;     // B slot free (its MMA done)
  uint64_t* tfull = bempty + SB;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint8_t* stg_all = smem + C::kRingBytes + 256;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = g.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&lfull[s], 1);    // A tile, codes and scale codes landed
      mbar_init(&lempty[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&bfull[s], kNvConvWarps);
      mbar_init(&bempty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_c0);
    tma_prefetch_desc(&tm_s0);
    if (kGlu) {
      tma_prefetch_desc(&tm_c1);
      tma_prefetch_desc(&tm_s1);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();   // (launched as a programmatic dependent: the previous kernel's results)
  const int total = (int)g.hdr->num_mtiles * g.n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      NvTile t;
      nv_tile_of(g, tile, t);
      const int brow = t.e * g.b_rows_per_expert + t.n * b_rows;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(&lempty[s], ph ^ 1, hdr)) { ok = false; break; }
        mbar_arrive_expect_tx(&lfull[s], kNvATile + C::kCTile + C::kSTile);
        tma_load_2d(sA + s * kNvATile, &tm_a, kb * 64, t.row0, &lfull[s]);
        uint8_t* cs = sC + s * C::kCTile;
        uint8_t* ss = sS + s * C::kSTile;
        tma_load_2d(cs, &tm_c0, kb * 32, brow, &lfull[s]);
        tma_load_2d(ss, &tm_s0, (kb >> 2) * 16, brow, &lfull[s]);
        if (kGlu) {
          tma_load_2d(cs + b_rows * 32, &tm_c1, kb * 32, brow, &lfull[s]);
          tma_load_2d(ss + b_rows * 16, &tm_s1, (kb >> 2) * 16, brow, &lfull[s]);
        }
        ++issued;
        if (++s == S) { s = 0; ph ^= 1; }
      }
    }
    if (!ok) {
      // let the copies already issued land before the CTA can exit
      for (long long i = issued > S ? issued - S : 0; i < issued; ++i) {
        mbar_wait(&lfull[i % S], (uint32_t)((i / S) & 1), nullptr);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_make(kNvBM, BN, 0, 0);   // f16 x f16
    int s = 0, sb = 0;
    uint32_t ph = 0, phb = 0;
    bool ok = true;
    int it = 0;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, hdr)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d = tmem_base + acc * BN;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        // the converters saw this step's load land before they finished its B tile
        if (!mbar_wait(&bfull[sb], phb, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kNvATile);
        const uint32_t b0 = smem_u32(sB + sb * C::kBTile);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_bf16(d, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                      (kb | k) != 0 ? 1u : 0u);
        tc_commit(&lempty[s]);
        tc_commit(&bempty[sb]);
        if (++s == S) { s = 0; ph ^= 1; }
        if (++sb == SB) { sb = 0; phb ^= 1; }
      }
      if (ok) tc_commit(&tfull[acc]);
    }
    tc_commit(drain);
    mbar_wait(drain, 0, hdr);
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r_local = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      NvTile t;
      nv_tile_of(g, tile, t);
      const int acc = it & 1;
      if (!mbar_wait(&tfull[acc], (it >> 1) & 1, hdr)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      const int row = t.row0 + r_local;
      const bool valid = row < t.row1;
      const float s2a = g.s2_0[t.e];
      if (kGlu) {
        const float s2u = g.s2_1[t.e];
        __half* orow = static_cast<__half*>(g.out) + (size_t)row * g.ldo + t.n * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          float gv[32], uv[32];
          tmem_ld32(taddr + c, gv);
          tmem_ld32(taddr + BN / 2 + c, uv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float h[8];
#pragma unroll
              for (int j = 0; j < 8; ++j)
                h[j] = silu(gv[8 * v + j] * s2a) * (uv[8 * v + j] * s2u);
              uint4 o;
              o.x = pack_f16x2(h[0], h[1]);
              o.y = pack_f16x2(h[2], h[3]);
              o.z = pack_f16x2(h[4], h[5]);
              o.w = pack_f16x2(h[6], h[7]);
              dst[v] = o;
            }
          }
        }
      } else {
        // 64 output columns at a time through the warp's staging rows: whole 128-byte row
        // segments per store instruction
        uint8_t* stg = stg_all + (warp - 2) * kNvStageRows;
        uint8_t* obase = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(g.out) +
                                                    (size_t)(t.row0 + q * 32) * g.ldo + t.n * BN);
#pragma unroll 1
        for (int c = 0; c < BN; c += 64) {
          uint4 pk[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[32];
            tmem_ld32(taddr + c + 32 * h, v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              pk[4 * h + j].x = pack_bf16x2(v[8 * j + 0] * s2a, v[8 * j + 1] * s2a);
              pk[4 * h + j].y = pack_bf16x2(v[8 * j + 2] * s2a, v[8 * j + 3] * s2a);
              pk[4 * h + j].z = pack_bf16x2(v[8 * j + 4] * s2a, v[8 * j + 5] * s2a);
              pk[4 * h + j].w = pack_bf16x2(v[8 * j + 6] * s2a, v[8 * j + 7] * s2a);
            }
          }
          warp_store_rows<8>(stg, pk, obase + c * 2, (size_t)g.ldo * 2, t.row1 - t.row0 - q * 32);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  } else if (warp >= kNvConvBase / 32) {
    // ------------------------------------------------ converters
    const int r = threadIdx.x - kNvConvBase;   // B-tile row of this thread
    int s = 0, sb = 0;
    uint32_t ph = 0, phb = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(&lfull[s], ph, hdr) || !mbar_wait(&bempty[sb], phb ^ 1, hdr)) {
          ok = false;
          break;
        }
        if (r < BN) {
          const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(sS + s * C::kSTile + r * 16 +
                                                                  (kb & 3) * 4);
          nvfp4_row_to_f16(sC + s * C::kCTile + r * 32, sc4, sB + sb * C::kBTile + r * 128, r);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bfull[sb]);
        if (++s == S) { s = 0; ph ^= 1; }
        if (++sb == SB) { sb = 0; phb ^= 1; }
      }
      if (!ok) break;
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
cudaError_t launch_nv(const CUtensorMap maps[5], const NvGemmArgs& g, int num_sms,
                      cudaStream_t st) {
  using C = NvCfg<BN>;
  auto kern = gemm_nvfp4_kernel<BN, MODE>;
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(kern), nv_smem_bytes<BN, MODE>());
  if (e != cudaSuccess) return e;
  const int max_tiles = g.max_mtiles * g.n_tiles;
  int grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  return launch_dependent(kern, dim3(grid), dim3(kNvThreads), nv_smem_bytes<BN, MODE>(), st, maps[0],
                          maps[1], maps[2], maps[3], maps[4], g);
}

}  // namespace

cudaError_t launch_gemm_nvfp4(int mode, int bn, const CUtensorMap maps[5], const NvGemmArgs& g,
                              int num_sms, cudaStream_t st) {
  if (mode == kGemmSwiGLU && bn == 256) return launch_nv<256, kGemmSwiGLU>(maps, g, num_sms, st);
  if (mode == kGemmStoreBF16 && bn == 256)
    return launch_nv<256, kGemmStoreBF16>(maps, g, num_sms, st);
  if (mode == kGemmStoreBF16 && bn == 128)
    return launch_nv<128, kGemmStoreBF16>(maps, g, num_sms, st);
  return cudaErrorInvalidValue;
}

}  // namespace moe
