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
// Threads: three warpgroups (384 threads, one CTA per SM).
//   warpgroup 0  warp 0 TMA producer; warp 1 TMEM owner + MMA issuer; warps 2-3 stage the
//                scales (A row scales and B block scales), eight K blocks at a time, into one
//                of two shared-memory buffers ahead of the promotion.
//   warpgroups 1-2  promotion + epilogue: two warps per TMEM lane quadrant, each owning one
//                half of the 256 columns of its 32 rows (128 fp32 accumulators per thread).
// Registers: the launch gives every thread 168; warpgroup 0 hands most of its share to the
// promotion warpgroups (setmaxnreg: 56 vs 224 per thread, 128*56 + 256*224 = 384*168), so the
// 128 accumulators and a 64-column TMEM read stay in registers. The host checks the launch
// register count before the first launch (a split that asked for more than the launch holds
// would never complete).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;            // 65536 / 384, rounded down to a multiple of 8
constexpr int kRegsWg0 = 56;
constexpr int kRegsPromo = 224;
static_assert(128 * kRegsWg0 + 256 * kRegsPromo <= kThreads * kLaunchRegs, "register split");
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;                    // fp8 elements = bytes per swizzle row
constexpr int kStages = 4;
constexpr int kMaxKb = 32;                  // K blocks of 128 per tile (K <= 4096)
constexpr int kPromoWarps = 8;              // promotion / epilogue warps
constexpr int kStagerWarps = 2;             // scale staging warps
constexpr int kATile = kBM * kBK;           // 16 KB
constexpr int kBTile = kBN * kBK;           // 32 KB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kTmemCols = 2 * kBN;          // two partial buffers
// Scales are staged in chunks of kScKb K blocks through two buffers: A row scales [kb][128]
// and B block scales [half][kb][2] (gate, up) of the chunk.
constexpr int kScKb = 8;
constexpr int kSaFloats = kScKb * kBM;
constexpr int kSbFloats = 2 * kScKb * 2;
constexpr int kScaleBufFloats = kSaFloats + kSbFloats;
constexpr size_t kSmemBase = 1024 + (size_t)kStages * kStageBytes + 256 + 2 * 2 * 128 * 4 +
                             (size_t)2 * kScaleBufFloats * 4;
constexpr int kStageRowBytes = 32 * 64;     // down: one promotion warp's staging rows
// (the down projection adds the promotion warps' staging rows)
template <int MODE>
constexpr size_t smem_bytes() {
  return kSmemBase + (MODE == 1 ? (size_t)kPromoWarps * kStageRowBytes : 0);
}
static_assert(smem_bytes<1>() <= 227 * 1024, "shared memory");

__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsPromo));
}
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWg0));
}

// SiLU(z) = z * sigmoid(z) with sigmoid(z) = (1 + tanh(z/2)) / 2 from the hardware tanh
// approximation (relative error about 2^-11): one special-function op per element instead of
// an exponential and a reciprocal. The result is quantised to E4M3 (3 mantissa bits) next.
__device__ __forceinline__ float silu_tanh(float z) {
  const float hz = 0.5f * z;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hz));
  return fmaf(hz, t, hz);
}

// q = v / s for a run of values sharing one divisor, by Markstein's method (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): r = 1/s correctly rounded once, then per value the product q0 = v * r,
// its exact residual e = v - q0 * s (one fused multiply-add) and the corrected quotient
// q0 + e * r -- the correctly rounded quotient for normal operands. Two values per
// instruction (fp32x2).
__device__ __forceinline__ float2 div_by(float2 v, float s, float r) {
  const float2 r2 = make_float2(r, r);
  const float2 q0 = __fmul2_rn(v, r2);
  const float2 e = __ffma2_rn(make_float2(-q0.x, -q0.y), make_float2(s, s), v);
  return __ffma2_rn(e, r2, q0);
}

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

// acc[0..31] += s * v[0..31], two lanes of fp32 per instruction.
__device__ __forceinline__ void fma_block32(float* acc, const float* v, float s) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 r = __ffma2_rn(s2, make_float2(v[j], v[j + 1]), make_float2(acc[j], acc[j + 1]));
    acc[j] = r.x;
    acc[j + 1] = r.y;
  }
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
  uint64_t* pfull = empty + kStages;      // [2] K block partial in TMEM
  uint64_t* pempty = pfull + 2;           // [2] partial read back by every promotion thread
  uint64_t* sfull = pempty + 2;           // [2] a chunk of scales staged
  uint64_t* sempty = sfull + 2;           // [2] that chunk no longer needed
  uint64_t* drain = sempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* amax_s = reinterpret_cast<float*>(smem + kStages * kStageBytes + 256);  // [2][128]
  uint32_t* seq_s = reinterpret_cast<uint32_t*>(amax_s + 2 * 128);                // [2][128]
  float* scale_s = reinterpret_cast<float*>(seq_s + 2 * 128);                     // [2][buf]
  uint8_t* stg_all = reinterpret_cast<uint8_t*>(scale_s + 2 * kScaleBufFloats);    // down only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = g.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], 1);
      // one arrival per warp (lane 0, after the warp's lanes are done)
      mbar_init(&pempty[i], kPromoWarps);
      mbar_init(&sfull[i], kStagerWarps);
      mbar_init(&sempty[i], kPromoWarps);
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
  pdl_wait();   // (launched as a programmatic dependent: the previous kernel's results)

  const int num_m = (int)g.hdr->num_mtiles;
  const int total = num_m * g.n_tiles;

  if (warp < 4) {
    setmaxnreg_dec();
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
          if (MODE == 0)
            tma_load_2d(sB + s * kBTile + (kBN / 2) * kBK, &tm_b1, kb * kBK, brow, &full[s]);
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
      // ------------------------------------------------ scale stager (64 threads)
      const int st = threadIdx.x - 64;
      const int half = st >> 5;
      uint32_t cc = 0;   // chunks staged so far (all tiles)
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const int m = tile / g.n_tiles, n = tile % g.n_tiles;
        const int4 t = g.tiles[m];
        const int r0 = t.y + st, r1 = t.y + st + 64;
        const bool v0 = r0 < t.z, v1 = r1 < t.z;
        for (int kc = 0; kc < g.num_kb; kc += kScKb, ++cc) {
          const int b = cc & 1;
          if (!mbar_wait(&sempty[b], ((cc >> 1) & 1) ^ 1, hdr)) { ok = false; break; }
          float* sa_s = scale_s + b * kScaleBufFloats;
          float* sb_s = sa_s + kSaFloats;
          // A row scales: rows st and st + 64 of the tile, four K blocks in flight at a time
#pragma unroll
          for (int u0 = 0; u0 < kScKb; u0 += 4) {
            float a[4], c[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int kb = kc + u0 + u;
              const float* col = g.sa + (size_t)kb * g.sa_stride;
              a[u] = (kb < g.num_kb && v0) ? __ldg(col + r0) : 0.0f;
              c[u] = (kb < g.num_kb && v1) ? __ldg(col + r1) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              sa_s[(u0 + u) * kBM + st] = a[u];
              sa_s[(u0 + u) * kBM + st + 64] = c[u];
            }
          }
          // B block scales of this warp's column half: [half][kb][gate, up] (down: one)
          if (lane < kScKb && kc + lane < g.num_kb) {
            const int kb = kc + lane;
            float b0, b1;
            if (MODE == 0) {
              const size_t bi = ((size_t)t.x * g.b_blocks_per_expert + n) * g.num_kb + kb;
              b0 = __ldg(g.sb0 + bi);
              b1 = __ldg(g.sb1 + bi);
            } else {
              const size_t bi =
                  ((size_t)t.x * g.b_blocks_per_expert + 2 * n + half) * g.num_kb + kb;
              b0 = b1 = __ldg(g.sb0 + bi);
            }
            sb_s[(half * kScKb + lane) * 2] = b0;
            sb_s[(half * kScKb + lane) * 2 + 1] = b1;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfull[b]);   // (release: the warp's stores are seen)
        }
      }
    }
  } else {
    setmaxnreg_inc();
    // ------------------------------------------------ promotion + epilogue
    const int q = warp & 3;                   // TMEM lane quadrant
    const int half = (warp - 4) >> 2;        // column half of this warp
    const int r_local = q * 32 + lane;
    uint32_t pc = 0;
    uint32_t cc = 0;   // scale chunks consumed so far
    uint32_t tseq = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      ++tseq;
      const int m = tile / g.n_tiles, n = tile % g.n_tiles;
      const int4 t = g.tiles[m];
      const int row = t.y + r_local;
      const bool valid = row < t.z;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < g.num_kb; ++kb, ++pc) {
        const uint32_t slot = pc & 1;
        // this K block's scales, from the chunk buffer of the stager
        const int u = kb % kScKb;
        const int b = cc & 1;
        if (u == 0 && !mbar_wait(&sfull[b], (cc >> 1) & 1, hdr)) { ok = false; break; }
        const float* sa_s = scale_s + b * kScaleBufFloats;
        const float* sb_s = sa_s + kSaFloats + half * kScKb * 2;
        const float sa = sa_s[u * kBM + r_local];
        const float s0 = sa * sb_s[u * 2];
        const float s1 = MODE == 0 ? sa * sb_s[u * 2 + 1] : s0;
        if (u == kScKb - 1 || kb == g.num_kb - 1) {   // the chunk's last K block: release it
          __syncwarp();
          if (lane == 0) mbar_arrive(&sempty[b]);
          ++cc;
        }
        if (!mbar_wait(&pfull[slot], (pc >> 1) & 1, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + slot * kBN;
        // columns: SwiGLU -> gate [half*64, +64) and up [128 + half*64, +64);
        // down -> [half*128, +128)
        const uint32_t c0 = MODE == 0 ? half * 64 : half * 128;
        const uint32_t c1 = MODE == 0 ? 128 + half * 64 : half * 128 + 64;
        // two 32-column register buffers: each is promoted, then refilled with the next
        // 32 columns while the other one is promoted, so the slot is released after the
        // fourth read, with half of the promotion still to do
        float v0[32], v1[32];
        tmem_ld32_nowait(taddr + c0, v0);
        tmem_ld32_nowait(taddr + c0 + 32, v1);
        tmem_wait_ld_tied(v0);
        tmem_tie(v1);
        fma_block32(acc, v0, s0);
        tmem_ld32_nowait(taddr + c1, v0);
        fma_block32(acc + 32, v1, s0);
        tmem_ld32_nowait(taddr + c1 + 32, v1);
        tmem_wait_ld_tied(v0);
        tmem_tie(v1);
        // the partial is in registers: the MMA may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[slot]);
        fma_block32(acc + 64, v0, s1);
        fma_block32(acc + 96, v1, s1);
      }
      if (!ok) break;
      if (MODE == 0) {
        // h = SiLU(gate) * up for 64 columns; quantise each row's 128-wide group (two warps)
        float am = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = silu_tanh(acc[j]) * acc[64 + j];
          am = fmaxf(am, fabsf(acc[j]));
        }
        const float other = exchange_amax(amax_s, seq_s, half, r_local, am, tseq, hdr);
        if (other < 0.0f) break;
        am = fmaxf(am, other);
        const float scale = am > 0.0f ? __fdiv_rn(am, 448.0f) : 1.0f;
        const float rcp = __frcp_rn(scale);
        if (valid) {
          uint8_t* orow = static_cast<uint8_t*>(g.out) + (size_t)row * g.ldo + n * 128 + half * 64;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = v4 * 16 + i * 4;
              const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                  div_by(make_float2(acc[j], acc[j + 1]), scale, rcp), __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                  div_by(make_float2(acc[j + 2], acc[j + 3]), scale, rcp), __NV_SATFINITE,
                  __NV_E4M3);
              w[i] = lo | (hi << 16);
            }
            reinterpret_cast<uint4*>(orow)[v4] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (half == 0) g.out_scales[(size_t)n * g.out_scale_stride + row] = scale;
        }
      } else {
        // 32 columns at a time through the warp's staging rows: 64-byte row segments, 8 rows
        // per store instruction
        uint8_t* stg = stg_all + (warp - 4) * kStageRowBytes;
        uint8_t* obase = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(g.out) +
                                                    (size_t)(t.y + q * 32) * g.ldo + n * kBN +
                                                    half * 128);
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint4 pk[4];
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            pk[v8].x = pack_bf16x2(acc[c + 8 * v8 + 0], acc[c + 8 * v8 + 1]);
            pk[v8].y = pack_bf16x2(acc[c + 8 * v8 + 2], acc[c + 8 * v8 + 3]);
            pk[v8].z = pack_bf16x2(acc[c + 8 * v8 + 4], acc[c + 8 * v8 + 5]);
            pk[v8].w = pack_bf16x2(acc[c + 8 * v8 + 6], acc[c + 8 * v8 + 7]);
          }
          warp_store_rows<4>(stg, pk, obase + c * 2, (size_t)g.ldo * 2, t.z - t.y - q * 32);
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

// The register split above assumes the launch gives every thread exactly kLaunchRegs.
template <int MODE>
cudaError_t check_launch_regs() {
  static int ok[64];   // per device: 0 unknown, 1 checked
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && ok[dev]) return cudaSuccess;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, gemm_fp8_kernel<MODE>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidDeviceFunction;
  if (dev >= 0 && dev < 64) ok[dev] = 1;
  return cudaSuccess;
}

template <int MODE>
cudaError_t launch_t(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                     const Fp8GemmArgs& g, int num_sms, cudaStream_t st) {
  auto kern = gemm_fp8_kernel<MODE>;
  cudaError_t e = check_launch_regs<MODE>();
  if (e != cudaSuccess) return e;
  e = ensure_dyn_smem(reinterpret_cast<const void*>(kern), smem_bytes<MODE>());
  if (e != cudaSuccess) return e;
  const int max_tiles = g.max_mtiles * g.n_tiles;
  int grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  return launch_dependent(kern, dim3(grid), dim3(kThreads), smem_bytes<MODE>(), st, a, b0, b1, g);
}

}  // namespace

cudaError_t launch_gemm_fp8(int mode, const CUtensorMap& a, const CUtensorMap& b0,
                            const CUtensorMap& b1, const Fp8GemmArgs& g, int num_sms,
                            cudaStream_t st) {
  if (g.num_kb > kMaxKb) return cudaErrorInvalidValue;
  if (mode == 0) return launch_t<0>(a, b0, b1, g, num_sms, st);
  return launch_t<1>(a, b0, b1, g, num_sms, st);
}

}  // namespace moe
