// Decode chain (few tokens): the expert projections of the whole batch as skinny GEMMs on the
// 5th-generation tensor cores, in one persistent, cooperatively launched kernel that streams
// the weights of every expert the batch touches -- gate and up rows, then down rows -- from
// HBM once, for all the tokens routed to it. The shared expert is one more slot.
//
// Pages: "spark_model/layers/moe/forward.rs" (`forward`: fused gate/up projection for the K
// routed experts plus the shared expert, fused SiLU and down projection, weighted sum and
// sigmoid-gated shared blend, all on device with no host synchronisation) and
// "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (few-row decode: routed down
// projections weighted and FP32-atomic-added into an [N,H] accumulator zeroed first, then a
// finalize that casts to BF16 and blends the shared expert).
//
// Shape of the work. A weight tile is 128 rows of one projection of one slot (the A operand,
// M = 128); the batch is the B operand (N = 16, tokens zero-padded): x itself for gate/up,
// SiLU(gate)*up of the slot's tokens for down. A work item is one tile times 128 of its
// contraction columns (32 KB of weights). Items are numbered slot-major; every block takes a
// contiguous, balanced range of the gate/up items and then of the down items, so a block's
// consecutive items of one tile form a run that accumulates in TMEM. The grid of each phase is
// capped so that no tile is split over more than two blocks: the two fp32 partial sums then
// meet in a zeroed buffer through atomic adds, and a + b == b + a makes the result
// independent of their order.
//
// Roles (192 threads, one block per SM, all blocks resident):
//   warp 0     TMA producer: per item two 128x64 weight boxes (+ two 16x64 x boxes on gate/up)
//              into a ring of 36 KB stages.
//   warp 1     allocates 32 TMEM columns (two 16-column accumulators); one lane issues
//              tcgen05.mma (M=128, N=16, K=16) x 8 per item and commits stage releases and
//              finished runs.
//   warps 2-5  epilogue: tcgen05.ld of a finished run, fp32 atomic adds of each token's column
//              into the gate/up buffer (then one count per run for the slot) or into the down
//              output; before the first down run of a slot, wait for the slot's gate/up count
//              (other blocks; bounded spin) and build SiLU(gate)*up in shared memory as the
//              bf16 B operand (128-byte swizzle).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 192;
constexpr int kM = 128;                  // weight rows per tile (MMA M)
constexpr int kNB = 16;                  // MMA N: the batch's tokens, zero-padded
constexpr int kKC = 128;                 // contraction columns per item (two 64-column boxes)
constexpr int kABytes = kM * kKC * 2;    // 32 KB
constexpr int kXBytes = kNB * kKC * 2;   // 4 KB
constexpr int kStageBytes = kABytes + kXBytes;
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 32;            // two accumulators of kNB columns
constexpr int kEpiThreads = 128;
constexpr int kSmemLimit = 227 * 1024;

struct Plan {
  int stages;
  int hbytes;   // B operand of the down projection: [16 rows, max(I, S)] bf16, swizzled
};

// Routing of the batch, copied to shared memory once per block: expert, first sorted row and
// row count of every active slot, and the token of every sorted row.
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

// Item numbering of both phases.
struct Geo {
  int nIt, nSt;     // 128-row tiles of one gate (or up) projection: routed, shared
  int Pg;           // items per gate/up tile (H / 128)
  int nHt;          // 128-row tiles of a down projection (H / 128)
  int Pdr, Pds;     // items per down tile: routed (I / 128), shared (S / 128)
  int na;           // active routed slots
  int g_rt, g_items, d_ritems, d_items;
  __device__ void init(const DecodeArgs& a, int n_active) {
    nIt = a.I / kM;
    nSt = a.S / kM;
    Pg = a.H / kKC;
    nHt = a.H / kM;
    Pdr = a.I / kKC;
    Pds = a.S / kKC;
    na = n_active;
    g_rt = na * 2 * nIt;
    g_items = (g_rt + (a.S ? 2 * nSt : 0)) * Pg;
    d_ritems = na * nHt * Pdr;
    d_items = d_ritems + (a.S ? nHt * Pds : 0);
  }
  // slot: active slot index, or -1 for the shared expert; lt: tile within the slot's
  // projection(s) (gate/up: gate tiles first, then up tiles)
  __device__ void item(bool down, int it, int& tile, int& kc, int& slot, int& lt) const {
    if (!down) {
      tile = it / Pg;
      kc = it - tile * Pg;
      if (tile < g_rt) {
        slot = tile / (2 * nIt);
        lt = tile - slot * 2 * nIt;
      } else {
        slot = -1;
        lt = tile - g_rt;
      }
    } else if (it < d_ritems) {
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
};

// Contiguous share [i0, i1) of `total` items for this block. At most total / per_tile blocks
// take part, so every block holds at least one tile's worth of items and no tile is split over
// more than two blocks.
__device__ __forceinline__ void phase_range(int total, int per_tile, int& i0, int& i1) {
  int G = gridDim.x;
  int cap = total / per_tile;
  if (cap < 1) cap = 1;
  if (G > cap) G = cap;
  const int b = blockIdx.x;
  if (b >= G) {
    i0 = i1 = 0;
    return;
  }
  i0 = (int)((long long)total * b / G);
  i1 = (int)((long long)total * (b + 1) / G);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// v[c] for a warp-uniform column c < 16 (no dynamic register indexing).
__device__ __forceinline__ float pick16(const float* v, int c) {
  float r = v[0];
#pragma unroll
  for (int i = 1; i < 16; ++i)
    if (c == i) r = v[i];
  return r;
}

__device__ __forceinline__ int slot_rows(const DecodeArgs& a, const RouteMeta& m, int slot,
                                         int& r0) {
  if (slot < 0) {
    r0 = a.te;
    return a.N;
  }
  r0 = m.slot_r0[slot];
  return m.slot_n[slot];
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_ffn_kernel(const __grid_constant__ CUtensorMap tm_wg,
                      const __grid_constant__ CUtensorMap tm_wu,
                      const __grid_constant__ CUtensorMap tm_sg,
                      const __grid_constant__ CUtensorMap tm_su,
                      const __grid_constant__ CUtensorMap tm_wd,
                      const __grid_constant__ CUtensorMap tm_sd,
                      const __grid_constant__ CUtensorMap tm_x, const DecodeArgs a, const Plan pl) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ RouteMeta meta;
  __shared__ uint64_t bars[2 * kMaxStages + 6];
  __shared__ uint32_t tmem_slot;
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stages = pl.stages;
  uint8_t* ring = smem;
  uint8_t* hb = smem + (size_t)stages * kStageBytes;   // down-projection B operand
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* afull = bars + 2 * kMaxStages;             // [2] run accumulated
  uint64_t* aempty = afull + 2;                        // [2] run drained
  uint64_t* bfull = aempty + 2;                        // down B operand built
  uint64_t* drain = bfull + 1;                         // every MMA complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = a.hdr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 4);   // lane 0 of each epilogue warp
    }
    mbar_init(bfull, 1);
    mbar_init(drain, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wu);
    tma_prefetch_desc(&tm_wd);
    tma_prefetch_desc(&tm_x);
    if (a.S) {
      tma_prefetch_desc(&tm_sg);
      tma_prefetch_desc(&tm_su);
      tma_prefetch_desc(&tm_sd);
    }
  }
  pdl_trigger();   // the combine kernel may launch and wait for this one
  if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  load_route_meta(a, meta);   // (ends with a block barrier)
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;

  Geo geo;
  geo.init(a, meta.n_active);
  int g0, g1, d0, d1;
  phase_range(geo.g_items, geo.Pg, g0, g1);
  phase_range(geo.d_items, geo.Pdr > geo.Pds ? geo.Pdr : geo.Pds, d0, d1);
  const int ng = g1 - g0, nitems = ng + (d1 - d0);

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int k = 0; k < nitems; ++k) {
        if (!mbar_wait(&empty[s], ph ^ 1, hdr)) { ok = false; break; }
        const bool down = k >= ng;
        int tile, kc, slot, lt;
        geo.item(down, down ? d0 + (k - ng) : g0 + k, tile, kc, slot, lt);
        uint8_t* st = ring + (size_t)s * kStageBytes;
        const CUtensorMap* m;
        int row;
        if (!down) {
          const int nt = slot >= 0 ? geo.nIt : geo.nSt;
          const bool up = lt >= nt;
          const int r = (up ? lt - nt : lt) * kM;
          if (slot >= 0) {
            m = up ? &tm_wu : &tm_wg;
            row = (int)meta.slot_e[slot] * a.I + r;
          } else {
            m = up ? &tm_su : &tm_sg;
            row = r;
          }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          tma_load_2d(st + kABytes, &tm_x, kc * kKC, 0, &full[s]);
          tma_load_2d(st + kABytes + kXBytes / 2, &tm_x, kc * kKC + 64, 0, &full[s]);
        } else {
          m = slot >= 0 ? &tm_wd : &tm_sd;
          row = (slot >= 0 ? (int)meta.slot_e[slot] * a.H : 0) + lt * kM;
          mbar_arrive_expect_tx(&full[s], kABytes);
        }
        tma_load_2d(st, m, kc * kKC, row, &full[s]);
        tma_load_2d(st + kABytes / 2, m, kc * kKC + 64, row, &full[s]);
        ++issued;
        if (++s == stages) { s = 0; ph ^= 1; }
      }
      if (!ok)   // let the copies already issued land before the block can exit
        for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
          mbar_wait(&full[i % stages], (uint32_t)((i / stages) & 1), nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(kM, kNB, 1, 1);
      int s = 0, run = -1, prev_tile = -1, bslot = -2, nb = 0;
      uint32_t ph = 0;
      bool prev_down = false, ok = true, first = false;
      const uint32_t hb_addr = smem_u32(hb);
      for (int k = 0; k < nitems && ok; ++k) {
        const bool down = k >= ng;
        int tile, kc, slot, lt;
        geo.item(down, down ? d0 + (k - ng) : g0 + k, tile, kc, slot, lt);
        if (run < 0 || down != prev_down || tile != prev_tile) {
          if (run >= 0) tc_commit(&afull[run & 1]);
          ++run;
          prev_down = down;
          prev_tile = tile;
          if (!mbar_wait(&aempty[run & 1], (((uint32_t)run >> 1) & 1) ^ 1, hdr)) { ok = false; break; }
          if (down && slot != bslot) {
            if (!mbar_wait(bfull, (uint32_t)nb & 1, hdr)) { ok = false; break; }
            ++nb;
            bslot = slot;
          }
          tc_fence_after();
          first = true;
        }
        if (!mbar_wait(&full[s], ph, hdr)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)((run & 1) * kNB);
        const uint32_t a0 = smem_u32(ring + (size_t)s * kStageBytes);
        const uint32_t b0 = down ? hb_addr + (uint32_t)kc * 2 * 2048 : a0 + kABytes;
#pragma unroll
        for (int kk = 0; kk < kKC / 16; ++kk) {
          const uint32_t ka = (uint32_t)(kk >> 2) * (kM * 128) + (uint32_t)(kk & 3) * 32;
          const uint32_t kb = (uint32_t)(kk >> 2) * (kNB * 128) + (uint32_t)(kk & 3) * 32;
          tc_mma_bf16(d, sdesc_k_sw128(a0 + ka), sdesc_k_sw128(b0 + kb), idesc,
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
  } else {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row_l = q * 32 + lane;        // weight row within the tile
    const int et = threadIdx.x - 64;        // 0..127
    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
    int run = -1, prev_tile = -1, bslot = -2;
    bool prev_down = false;
    // the run being accumulated: phase, slot, tile within the slot, items
    bool r_down = false;
    int r_slot = 0, r_lt = 0, r_len = 0;
    bool ok = true;
    auto drain_run = [&]() {
      if (!ok) return;
      if (!mbar_wait(&afull[run & 1], ((uint32_t)run >> 1) & 1, hdr)) { ok = false; return; }
      tc_fence_after();
      float v[16];
      tmem_ld16(tq + (uint32_t)((run & 1) * kNB), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[run & 1]);
      int r0;
      const int ntok = slot_rows(a, meta, r_slot, r0);
      if (!r_down) {
        const int nt = r_slot >= 0 ? geo.nIt : geo.nSt;
        const int col = (r_lt < nt ? 0 : a.ldh) + (r_lt < nt ? r_lt : r_lt - nt) * kM + row_l;
        for (int jj = 0; jj < ntok; ++jj) {
          const int row = r0 + jj;
          const int t = row >= a.te ? row - a.te : (int)meta.row_tok[row];
          atomicAdd(a.hd + (size_t)row * (2 * a.ldh) + col, pick16(v, t));
        }
        // publish: the slot's count moves only after every partial sum of the run landed
        __threadfence();
        named_sync(1, kEpiThreads);
        if (et == 0) {
          __threadfence();
          atomicAdd(a.h_cnt + (r_slot < 0 ? kDecodeMaxPairs : r_slot), (uint32_t)r_len);
        }
      } else {
        const int r = r_lt * kM + row_l;
        for (int jj = 0; jj < ntok; ++jj) {
          const float y = pick16(v, jj);
          const int row = r0 + jj;
          if (r_slot < 0) {
            atomicAdd(a.shy + (size_t)jj * a.H + r, y);
          } else if (a.acc) {
            const uint32_t pair = __ldcg(a.sorted_pairs + row);
            atomicAdd(a.acc + (size_t)meta.row_tok[row] * a.H + r, a.w[pair] * y);
          } else {
            atomicAdd(a.yd + (size_t)row * a.H + r, y);
          }
        }
      }
    };
    // SiLU(gate) * up of the slot's tokens as the bf16 B operand [16 rows, L], 128-byte swizzle:
    // row j's 16-byte chunk c of K-block kb at kb * 2048 + j * 128 + ((c ^ (j & 7)) * 16).
    auto build_b = [&](int slot) {
      const uint32_t target =
          (uint32_t)((slot >= 0 ? 2 * geo.nIt : 2 * geo.nSt) * geo.Pg);
      if (et == 0) {
        const uint32_t* cnt = a.h_cnt + (slot < 0 ? kDecodeMaxPairs : slot);
        if (ld_acquire(cnt) < target) {
          const long long t0 = clock64();
          while (ld_acquire(cnt) < target) {
            if (clock64() - t0 > kSpinLimitCycles) {   // (the result is then not used)
              report_timeout(hdr);
              break;
            }
            __nanosleep(64);
          }
        }
      }
      named_sync(1, kEpiThreads);
      int r0;
      const int ntok = slot_rows(a, meta, slot, r0);
      const int L = slot >= 0 ? a.I : a.S;
      const int cpr = L / 8;   // 16-byte chunks per row
      for (int id = et; id < kNB * cpr; id += kEpiThreads) {
        const int j = id / cpr, c = id - j * cpr;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (j < ntok) {
          const float* hr = a.hd + (size_t)(r0 + j) * (2 * a.ldh) + c * 8;
          const float4 g0v = __ldcg(reinterpret_cast<const float4*>(hr));
          const float4 g1v = __ldcg(reinterpret_cast<const float4*>(hr + 4));
          const float4 u0 = __ldcg(reinterpret_cast<const float4*>(hr + a.ldh));
          const float4 u1 = __ldcg(reinterpret_cast<const float4*>(hr + a.ldh + 4));
          o.x = pack_bf16x2(silu(g0v.x) * u0.x, silu(g0v.y) * u0.y);
          o.y = pack_bf16x2(silu(g0v.z) * u0.z, silu(g0v.w) * u0.w);
          o.z = pack_bf16x2(silu(g1v.x) * u1.x, silu(g1v.y) * u1.y);
          o.w = pack_bf16x2(silu(g1v.z) * u1.z, silu(g1v.w) * u1.w);
        }
        *reinterpret_cast<uint4*>(hb + (size_t)(c >> 3) * 2048 + j * 128 +
                                  (((c & 7) ^ (j & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      named_sync(1, kEpiThreads);
      if (et == 0) mbar_arrive(bfull);
    };
    for (int k = 0; k < nitems; ++k) {
      const bool down = k >= ng;
      int tile, kc, slot, lt;
      geo.item(down, down ? d0 + (k - ng) : g0 + k, tile, kc, slot, lt);
      if (run < 0 || down != prev_down || tile != prev_tile) {
        if (run >= 0) drain_run();
        ++run;
        prev_down = down;
        prev_tile = tile;
        r_down = down;
        r_slot = slot;
        r_lt = lt;
        r_len = 0;
        // the MMAs of every earlier run are complete (drained): the B buffer is free
        if (down && slot != bslot) {
          build_b(slot);
          bslot = slot;
        }
      }
      ++r_len;
    }
    if (run >= 0) drain_run();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
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

cudaError_t launch_decode_ffn(const DecodeArgs& a, const CUtensorMap* maps, cudaStream_t st) {
  if (a.te > kDecodeMaxPairs || a.N > kDecodeMaxTokens || a.N < 1 || !a.h_cnt ||
      a.H % kKC || a.I % kKC || a.S % kKC)
    return cudaErrorInvalidValue;
  const int L = a.I > a.S ? a.I : a.S;
  Plan pl{};
  pl.hbytes = L * kNB * 2;
  const int fixed = 1024 + pl.hbytes;   // alignment slack + B operand
  // (the static shared memory -- routing metadata, barriers -- stays within the 8 KB margin)
  pl.stages = (kSmemLimit - 8192 - fixed) / kStageBytes;
  if (pl.stages > kMaxStages) pl.stages = kMaxStages;
  if (pl.stages < 2) return cudaErrorInvalidValue;
  const size_t sm = (size_t)fixed + (size_t)pl.stages * kStageBytes;
  cudaError_t e =
      cudaFuncSetAttribute(decode_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  // the down phase waits on other blocks' gate/up work: all blocks must be resident
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
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel, maps[kDmWg], maps[kDmWu], maps[kDmSg],
                            maps[kDmSu], maps[kDmWd], maps[kDmSd], maps[kDmX], a, pl);
}

}  // namespace moe
