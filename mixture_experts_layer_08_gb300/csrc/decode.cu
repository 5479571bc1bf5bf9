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
// Shape of the work. The weights are the wide B operand: a tile is BN (256, or 128 when a
// dimension is not a multiple of 256) rows of one projection of one slot, so every MMA reads
// its weights at the full-rate N. The batch is the A operand (M = 128): rows 0..15 hold the
// tokens (x for gate/up, SiLU(gate)*up of the slot's tokens for down), rows 16..127 read
// whatever shared memory follows and only produce accumulator rows that are never read. A
// work item is one tile times one 64-column swizzle box of its contraction (BN x 128 bytes).
// Items are numbered slot-major; every block takes a contiguous, balanced range of the gate/up
// items and then of the down items, so a block's consecutive items of one tile form a run
// that accumulates in TMEM. The grid of each phase is capped so that no tile is split over
// more than two blocks: the two fp32 partial sums then meet in a zeroed buffer through atomic
// adds, and a + b == b + a makes the result independent of their order.
//
// Roles (192 threads, one block per SM, all blocks resident):
//   warp 0     TMA producer: per item one BN x 64 weight box (+ one 16 x 64 box of x on
//              gate/up) into a ring of stages.
//   warp 1     allocates all 512 TMEM columns (two accumulators of up to 256 columns); one
//              lane issues tcgen05.mma (M=128, N=BN, K=16) x 4 per item and commits stage
//              releases and finished runs.
//   warps 2-5  epilogue. Warp 4 (TMEM lanes 0..31 = the token rows) drains a finished run:
//              fp32 atomic adds of each token's row into the gate/up buffer (then one count
//              per run for the slot) or into the down output. Before the first down run of a
//              slot, all four wait for the slot's gate/up count (other blocks; bounded spin)
//              and build SiLU(gate)*up of its tokens as the bf16 A operand (128-byte swizzle).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 192;
constexpr int kBox = 64;                  // contraction columns per item (one 128-byte row)
constexpr int kMaxBN = 256;
constexpr int kWBytes = kMaxBN * 128;     // weight box of a stage, 32 KB
constexpr int kTokBytes = 16 * 128;       // token rows of one contraction box, 2 KB
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 512;            // two accumulators of up to 256 columns
constexpr int kEpiThreads = 128;
constexpr int kDrainWarp = 4;             // warp % 4 == 0: TMEM lanes 0..31
constexpr int kStageLd = 68;              // drain staging row stride (floats; 16-byte rows)
constexpr int kSmemLimit = 227 * 1024;

struct Plan {
  int stages;
  int bn_g, bn_d;   // weight rows per tile: gate/up, down
  int hbytes;       // down-projection A operand: max(I, S) / 64 boxes of 16 rows x 128 bytes
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
  int nIt, nSt;     // weight tiles of one gate (or up) projection: routed, shared
  int Pg;           // items per gate/up tile (H / 64)
  int nHt;          // weight tiles of a down projection
  int Pdr, Pds;     // items per down tile: routed (I / 64), shared (S / 64)
  int na;           // active routed slots
  int g_rt, g_items, d_ritems, d_items;
  __device__ void init(const DecodeArgs& a, const Plan& pl, int n_active) {
    nIt = a.I / pl.bn_g;
    nSt = a.S / pl.bn_g;
    Pg = a.H / kBox;
    nHt = a.H / pl.bn_d;
    Pdr = a.I / kBox;
    Pds = a.S / kBox;
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
  __shared__ __align__(16) float stage_rows[16 * kStageLd];   // drain staging, 16 rows x 64
  // 1024-byte alignment for the 128-byte swizzle atoms. Layout: token boxes of the stages,
  // the down-projection A operand, the weight ring (the A descriptors' rows 16..127 read on
  // into what follows, always inside this allocation).
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stages = pl.stages;
  uint8_t* xtok = smem;                                   // [stages][16 x 128 B]
  uint8_t* hb = xtok + (size_t)stages * kTokBytes;        // [max(I,S)/64][16 x 128 B]
  uint8_t* ring = hb + pl.hbytes;                         // [stages][BN x 128 B]
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* afull = bars + 2 * kMaxStages;                // [2] run accumulated
  uint64_t* aempty = afull + 2;                           // [2] run drained
  uint64_t* bfull = aempty + 2;                           // down A operand built
  uint64_t* drain = bfull + 1;                            // every MMA complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = a.hdr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);   // the draining warp's lane 0
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
  geo.init(a, pl, meta.n_active);
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
        uint8_t* wst = ring + (size_t)s * kWBytes;
        if (!down) {
          const int nt = slot >= 0 ? geo.nIt : geo.nSt;
          const bool up = lt >= nt;
          const int r = (up ? lt - nt : lt) * pl.bn_g;
          const CUtensorMap* m;
          int row;
          if (slot >= 0) {
            m = up ? &tm_wu : &tm_wg;
            row = (int)meta.slot_e[slot] * a.I + r;
          } else {
            m = up ? &tm_su : &tm_sg;
            row = r;
          }
          mbar_arrive_expect_tx(&full[s], (uint32_t)(pl.bn_g * 128 + kTokBytes));
          tma_load_2d(xtok + (size_t)s * kTokBytes, &tm_x, kc * kBox, 0, &full[s]);
          tma_load_2d(wst, m, kc * kBox, row, &full[s]);
        } else {
          const CUtensorMap* m = slot >= 0 ? &tm_wd : &tm_sd;
          const int row = (slot >= 0 ? (int)meta.slot_e[slot] * a.H : 0) + lt * pl.bn_d;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(pl.bn_d * 128));
          tma_load_2d(wst, m, kc * kBox, row, &full[s]);
        }
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
      const uint32_t idesc_g = idesc_make(128, pl.bn_g, 1, 1);
      const uint32_t idesc_d = idesc_make(128, pl.bn_d, 1, 1);
      int s = 0, run = -1, prev_tile = -1, bslot = -2, nb = 0;
      uint32_t ph = 0;
      bool prev_down = false, ok = true, first = false;
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
        const uint32_t d = tmem_base + (uint32_t)((run & 1) * kMaxBN);
        const uint32_t a0 = down ? smem_u32(hb) + (uint32_t)kc * kTokBytes
                                 : smem_u32(xtok) + (uint32_t)s * kTokBytes;
        const uint32_t b0 = smem_u32(ring) + (uint32_t)s * kWBytes;
        const uint32_t idesc = down ? idesc_d : idesc_g;
#pragma unroll
        for (int kk = 0; kk < kBox / 16; ++kk)
          tc_mma_bf16(d, sdesc_k_sw128(a0 + kk * 32), sdesc_k_sw128(b0 + kk * 32), idesc,
                      (first && kk == 0) ? 0u : 1u);
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
    const int et = threadIdx.x - 64;        // 0..127
    const bool drainer = warp == kDrainWarp;
    int run = -1, prev_tile = -1, bslot = -2;
    bool prev_down = false;
    // the run being accumulated: phase, slot, tile within the slot, items
    bool r_down = false;
    int r_slot = 0, r_lt = 0, r_len = 0;
    bool ok = true;
    // Warp 4 drains a finished run: TMEM lane j < 16 holds accumulator row j (token j of x on
    // gate/up, the slot's j-th token on down) across the tile's BN columns. 64 columns at a
    // time go through shared memory so that every row's partial sums leave as coalesced
    // 32-lane atomic adds.
    auto drain_run = [&]() {
      if (!ok) return;
      if (!mbar_wait(&afull[run & 1], ((uint32_t)run >> 1) & 1, hdr)) { ok = false; return; }
      tc_fence_after();
      int r0;
      const int ntok = slot_rows(a, meta, r_slot, r0);
      const uint32_t tacc = tmem_base + (uint32_t)((run & 1) * kMaxBN);
      float* dst = nullptr;      // output row of accumulator row `lane` (lanes < 16)
      float scale = 1.0f;
      int bn;
      if (!r_down) {
        bn = pl.bn_g;
        int row = -1;            // sorted row of (slot, token lane)
        if (r_slot < 0) {
          if (lane < a.N) row = a.te + lane;
        } else {
          for (int j = 0; j < ntok; ++j)
            if ((int)meta.row_tok[r0 + j] == lane) row = r0 + j;
        }
        const int nt = r_slot >= 0 ? geo.nIt : geo.nSt;
        const int col = (r_lt < nt ? 0 : a.ldh) + (r_lt < nt ? r_lt : r_lt - nt) * bn;
        if (row >= 0) dst = a.hd + (size_t)row * (2 * a.ldh) + col;
      } else {
        bn = pl.bn_d;
        const int c0 = r_lt * bn;
        if (lane < ntok) {
          const int row = r0 + lane;
          if (r_slot < 0) {
            dst = a.shy + (size_t)lane * a.H + c0;
          } else if (a.acc) {
            scale = a.w[__ldcg(a.sorted_pairs + row)];
            dst = a.acc + (size_t)meta.row_tok[row] * a.H + c0;
          } else {
            dst = a.yd + (size_t)row * a.H + c0;
          }
        }
      }
      const uint32_t rows = __ballot_sync(0xffffffffu, dst != nullptr);
#pragma unroll 1
      for (int c = 0; c < bn; c += 64) {
        float v[64];
        tmem_ld32_nowait(tacc + (uint32_t)c, v);
        tmem_ld32_nowait(tacc + (uint32_t)c + 32, v + 32);
        tmem_wait_ld();
        if (lane < 16 && dst) {
          float4* st = reinterpret_cast<float4*>(stage_rows + lane * kStageLd);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        __syncwarp();
        for (uint32_t m = rows; m; m &= m - 1) {
          const int j = __ffs(m) - 1;
          float* dj = reinterpret_cast<float*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), j));
          const float sj = __shfl_sync(0xffffffffu, scale, j);
          atomicAdd(dj + c + lane, sj * stage_rows[j * kStageLd + lane]);
          atomicAdd(dj + c + 32 + lane, sj * stage_rows[j * kStageLd + 32 + lane]);
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[run & 1]);
      if (!r_down) {
        // publish: the slot's count moves only after every partial sum of the run landed
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(a.h_cnt + (r_slot < 0 ? kDecodeMaxPairs : r_slot), (uint32_t)r_len);
        }
      }
    };
    // SiLU(gate) * up of the slot's tokens as the bf16 A operand, 16 rows per 64-column box
    // with the 128-byte swizzle: row j's 16-byte chunk c of box kb at
    // kb * 2048 + j * 128 + ((c ^ (j & 7)) * 16).
    auto build_a = [&](int slot) {
      const uint32_t target = (uint32_t)((slot >= 0 ? 2 * geo.nIt : 2 * geo.nSt) * geo.Pg);
      if (drainer && lane == 0) {   // (after this warp published the block's own gate/up runs)
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
      for (int id = et; id < 16 * cpr; id += kEpiThreads) {
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
        *reinterpret_cast<uint4*>(hb + (size_t)(c >> 3) * kTokBytes + j * 128 +
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
        if (run >= 0 && drainer) drain_run();
        ++run;
        prev_down = down;
        prev_tile = tile;
        r_down = down;
        r_slot = slot;
        r_lt = lt;
        r_len = 0;
        // the MMAs of every earlier run are complete (drained): the A buffer is free
        if (down && slot != bslot) {
          build_a(slot);
          bslot = slot;
        }
      }
      ++r_len;
    }
    if (run >= 0 && drainer) drain_run();
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

// Weight rows per tile of each phase; the tensor maps of the weights use them as box rows.
void decode_tile_rows(int H, int I, int S, int* bn_g, int* bn_d) {
  *bn_g = (I % 256 == 0 && S % 256 == 0) ? 256 : 128;
  *bn_d = H % 256 == 0 ? 256 : 128;
}

cudaError_t launch_decode_ffn(const DecodeArgs& a, const CUtensorMap* maps, cudaStream_t st) {
  if (a.te > kDecodeMaxPairs || a.N > kDecodeMaxTokens || a.N < 1 || !a.h_cnt ||
      a.H % 128 || a.I % 128 || a.S % 128)
    return cudaErrorInvalidValue;
  const int L = a.I > a.S ? a.I : a.S;
  Plan pl{};
  decode_tile_rows(a.H, a.I, a.S, &pl.bn_g, &pl.bn_d);
  pl.hbytes = (L / kBox) * kTokBytes;
  const int per_stage = kTokBytes + kWBytes;
  const int fixed = 1024 + pl.hbytes;   // alignment slack + down A operand
  // (the static shared memory -- routing metadata, barriers -- stays within the 8 KB margin)
  pl.stages = (kSmemLimit - 8192 - fixed) / per_stage;
  if (pl.stages > kMaxStages) pl.stages = kMaxStages;
  if (pl.stages < 2) return cudaErrorInvalidValue;
  const size_t sm = (size_t)fixed + (size_t)pl.stages * per_stage;
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
