// FP8 (E4M3) grouped GEMM with block scales on the tcgen05 tensor cores (sm_103a).
//
// Operands: A rows quantised per 1x128 along K (one fp32 scale per row and 128-wide K block),
// B = expert weights quantised per 128x128 block (one fp32 scale per block). Because every
// 128-wide K block carries its own pair of scales, each K block's product is formed in TMEM
// on its own (kind::f8f6f4, M=128, N=256, 4 x K=32) and promoted into fp32 registers as
//   acc += (sa[row, kb] * sb[nblk, kb]) * partial_kb,
// with two TMEM partial buffers so the tensor cores run one K block ahead of the promotion.
//
// Epilogues: SwiGLU -> the intermediate quantised per 1x128 to E4M3 (codes + fp32 scales, the
// A operand of the down projection), or a plain bf16 store (down projection).
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (`forward_prefill_fp8` /
// `moe_fp8_grouped_gemm_k`: FP8 experts take the grouped GEMM over the expert-sorted rows),
// "spark_model/layers/moe/forward.rs" (FP8 experts carry per-expert weight and scale tables;
// FP8 experts reach a per-layer cosine of about 0.989 against BF16).
//
// Threads: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2-9 promotion and
// epilogue (two warps per TMEM lane quadrant, each owning half of the 256 columns).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 320;
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;                    // fp8 elements = bytes per swizzle row
constexpr int kStages = 3;
constexpr int kMaxKb = 32;                  // K blocks of 128 per tile (K <= 4096)
constexpr int kEpi = 256;                   // promotion / epilogue threads
constexpr int kATile = kBM * kBK;           // 16 KB
constexpr int kBTile = kBN * kBK;           // 32 KB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kTmemCols = 2 * kBN;          // two partial buffers
constexpr size_t kScaleBytes = (size_t)kMaxKb * kEpi * 4 + (size_t)8 * kMaxKb * 2 * 4;
constexpr size_t kSmemBytes =
    (size_t)kStages * kStageBytes + 1024 + 256 + 2 * 2 * 128 * 4 + kScaleBytes;

// Hands this thread's row amax to the warp that owns the other column half of the same row
// and returns the partner's; `seq` tags the tile so values of different tiles never mix.
// The wait is bounded: on expiry it reports a timeout and returns -1.
__device__ __forceinline__ float exchange_amax(volatile float* am_s, volatile uint32_t* seq_s,
                                              int half, int r, float am, uint32_t seq,
                                              WsHeader* hdr) {
  am_s[half * 128 + r] = am;
  __threadfence_block();
  seq_s[half * 128 + r] = seq;
  const int o = (1 - half) * 128 + r;
  const long long t0 = clock64();
  while (seq_s[o] != seq) {
    if (clock64() - t0 > kSpinLimitCycles) {
      report_timeout(hdr);
      return -1.0f;
    }
  }
  __threadfence_block();
  return am_s[o];
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b0,
                    const __grid_constant__ CUtensorMap tm_b1, const Fp8GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kATile;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* pfull = empty + kStages;
  uint64_t* pempty = pfull + 2;
  uint64_t* drain = pempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* amax_s = reinterpret_cast<float*>(smem + kStages * kStageBytes + 256);  // [2][128]
  uint32_t* seq_s = reinterpret_cast<uint32_t*>(amax_s + 2 * 128);                  // [2][128]
  // per tile: each promotion thread's row scale for every K block ([kb][thread]), and each
  // epilogue warp's weight-block scales ([warp][kb][gate/up])
  float* sa_s = reinterpret_cast<float*>(seq_s + 2 * 128);
  float* sb_s = sa_s + kMaxKb * kEpi;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = g.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], 256);
    }
    mbar_init(drain, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b0);
    if (MODE == 0) tma_prefetch_desc(&tm_b1);
  }
  for (int i = threadIdx.x; i < 2 * 128; i += blockDim.x) seq_s[i] = 0;
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_m = (int)g.hdr->num_mtiles;
  const int total = num_m * g.n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    int s = 0;
    uint32_t ph = 0;
    long long issued = 0;
    bool ok = true;
    constexpr int b_rows = MODE == 0 ? kBN / 2 : kBN;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const int m = tile / g.n_tiles, n = tile % g.n_tiles;
      const int4 t = g.tiles[m];
      const int brow = t.x * g.b_rows_per_expert + n * b_rows;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1, hdr)) { ok = false; break; }
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(sA + s * kATile, &tm_a, kb * kBK, t.y, &full[s]);
        tma_load_2d(sB + s * kBTile, &tm_b0, kb * kBK, brow, &full[s]);
        if (MODE == 0) tma_load_2d(sB + s * kBTile + (kBN / 2) * kBK, &tm_b1, kb * kBK, brow, &full[s]);
        ++issued;
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
    }
    if (!ok) {
      for (long long i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        mbar_wait(&full[i % kStages], (uint32_t)((i / kStages) & 1), nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer: one partial per K block
    constexpr uint32_t idesc = idesc_make(kBM, kBN, 0, 0);   // E4M3 x E4M3 -> fp32
    int s = 0;
    uint32_t ph = 0;
    uint32_t pc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < g.num_kb; ++kb, ++pc) {
        const uint32_t slot = pc & 1;
        if (!mbar_wait(&pempty[slot], ((pc >> 1) & 1) ^ 1, hdr)) { ok = false; break; }
        if (!mbar_wait(&full[s], ph, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kATile);
        const uint32_t b0 = smem_u32(sB + s * kBTile);
        const uint32_t d = tmem_base + slot * kBN;
#pragma unroll
        for (int k = 0; k < kBK / 32; ++k)
          tc_mma_fp8(d, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                     k != 0 ? 1u : 0u);
        tc_commit(&empty[s]);
        tc_commit(&pfull[slot]);
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
    }
    tc_commit(drain);
    mbar_wait(drain, 0, hdr);
  } else if (warp >= 2) {
    // ------------------------------------------------ promotion + epilogue
    const int q = warp & 3;                   // TMEM lane quadrant
    const int half = (warp - 2) >> 2;         // column half of this warp
    const int r_local = q * 32 + lane;
    uint32_t pc = 0;
    uint32_t tseq = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      ++tseq;
      const int m = tile / g.n_tiles, n = tile % g.n_tiles;
      const int4 t = g.tiles[m];
      const int e = t.x;
      const int row = t.y + r_local;
      const bool valid = row < t.z;
      // this tile's scales into shared memory, loads in flight together: every promotion
      // step below then reads them without a global round trip
      const int et = threadIdx.x - 64, ew = et >> 5;
      for (int kb = 0; kb < g.num_kb; ++kb)
        sa_s[kb * kEpi + et] = valid ? __ldg(g.sa + (size_t)kb * g.sa_stride + row) : 0.0f;
      if (lane < g.num_kb) {
        float b0, b1;
        if (MODE == 0) {
          const size_t bi = ((size_t)e * g.b_blocks_per_expert + n) * g.num_kb + lane;
          b0 = __ldg(g.sb0 + bi);
          b1 = __ldg(g.sb1 + bi);
        } else {
          const size_t bi =
              ((size_t)e * g.b_blocks_per_expert + 2 * n + half) * g.num_kb + lane;
          b0 = b1 = __ldg(g.sb0 + bi);
        }
        sb_s[(ew * kMaxKb + lane) * 2] = b0;
        sb_s[(ew * kMaxKb + lane) * 2 + 1] = b1;
      }
      __syncwarp();
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < g.num_kb; ++kb, ++pc) {
        const uint32_t slot = pc & 1;
        const float sa = sa_s[kb * kEpi + et];
        const float s0 = sa * sb_s[(ew * kMaxKb + kb) * 2];
        const float s1 = sa * sb_s[(ew * kMaxKb + kb) * 2 + 1];
        if (!mbar_wait(&pfull[slot], (pc >> 1) & 1, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + slot * kBN;
        // columns: SwiGLU -> gate [half*64, +64) and up [128 + half*64, +64); down -> [half*128, +128)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = MODE == 0 ? (c < 2 ? half * 64 + c * 32 : 128 + half * 64 + (c - 2) * 32)
                                    : half * 128 + c * 32;
          float v[32];
          tmem_ld32(taddr + col, v);
          const float sc = (MODE == 0 && c >= 2) ? s1 : s0;
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[c * 32 + j] = fmaf(sc, v[j], acc[c * 32 + j]);
        }
        tc_fence_before();
        mbar_arrive(&pempty[slot]);
      }
      __syncwarp();     // the next tile rewrites this warp's scales
      if (!ok) break;
      if (MODE == 0) {
        // h = SiLU(gate) * up for 64 columns; quantise each row's 128-wide group (two warps)
        float am = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = silu(acc[j]) * acc[64 + j];
          am = fmaxf(am, fabsf(acc[j]));
        }
        const float other = exchange_amax(amax_s, seq_s, half, r_local, am, tseq, hdr);
        if (other < 0.0f) break;
        am = fmaxf(am, other);
        const float scale = am > 0.0f ? __fdiv_rn(am, 448.0f) : 1.0f;
        if (valid) {
          uint8_t* orow = static_cast<uint8_t*>(g.out) + (size_t)row * g.ldo + n * 128 + half * 64;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = v * 16 + i * 4;
              const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                  make_float2(__fdiv_rn(acc[j], scale), __fdiv_rn(acc[j + 1], scale)),
                  __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                  make_float2(__fdiv_rn(acc[j + 2], scale), __fdiv_rn(acc[j + 3], scale)),
                  __NV_SATFINITE, __NV_E4M3);
              w[i] = lo | (hi << 16);
            }
            reinterpret_cast<uint4*>(orow)[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (half == 0) g.out_scales[(size_t)n * g.out_scale_stride + row] = scale;
        }
      } else if (valid) {
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(g.out) + (size_t)row * g.ldo +
                              n * kBN + half * 128;
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          uint4 o;
          o.x = pack_bf16x2(acc[8 * v + 0], acc[8 * v + 1]);
          o.y = pack_bf16x2(acc[8 * v + 2], acc[8 * v + 3]);
          o.z = pack_bf16x2(acc[8 * v + 4], acc[8 * v + 5]);
          o.w = pack_bf16x2(acc[8 * v + 6], acc[8 * v + 7]);
          reinterpret_cast<uint4*>(orow)[v] = o;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int MODE>
cudaError_t launch_t(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                     const Fp8GemmArgs& g, int num_sms, cudaStream_t st) {
  auto kern = gemm_fp8_kernel<MODE>;
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(kern), kSmemBytes);
  if (e != cudaSuccess) return e;
  const int max_tiles = g.max_mtiles * g.n_tiles;
  int grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  kern<<<grid, kThreads, kSmemBytes, st>>>(a, b0, b1, g);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_fp8(int mode, const CUtensorMap& a, const CUtensorMap& b0,
                            const CUtensorMap& b1, const Fp8GemmArgs& g, int num_sms,
                            cudaStream_t st) {
  if (mode == 0) return launch_t<0>(a, b0, b1, g, num_sms, st);
  return launch_t<1>(a, b0, b1, g, num_sms, st);
}

}  // namespace moe
