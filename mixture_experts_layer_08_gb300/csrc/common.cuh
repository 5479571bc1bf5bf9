// Shared device helpers of the MoE kernels: bf16/fp32 packing, warp reductions, bounded
// mbarrier waits, TMA tile loads and the tcgen05 (5th-generation tensor core) primitives
// for sm_103a, written as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Workspace header: the first 256 bytes of every workspace.
struct WsHeader {
  int32_t status;          // MOE_OK or MOE_ERR_DEVICE_TIMEOUT, written by kernels
  uint32_t done_blocks;    // "last block" counter of the small router's fused tail; grid
                           // barrier counter of the fused decode kernel
  uint32_t num_active;     // distinct experts with at least one routed row
  uint32_t num_mtiles;     // 128-row tiles of the grouped GEMM (sum over experts)
  float gate_dot[16];      // fused decode kernel: x[t] . g of the shared-expert gate, t < 16
  uint32_t pad[44];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr uint32_t kNoRow = 0xFFFFFFFFu;

// Roughly a second at 2 GHz: no healthy wait in these kernels lasts a millisecond.
constexpr long long kSpinLimitCycles = 2000000000ll;

__device__ __forceinline__ void report_timeout(WsHeader* hdr) {
  if (hdr) atomicExch(&hdr->status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 8 bf16 packed in a uint4 -> 8 floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// SiLU(z) = z / (1 + e^-z) with the fast exponential and the fast (approximate-reciprocal)
// divide: a few ulp, far below the bf16 rounding of the result, and a short dependency chain
// for the epilogues that apply it to every accumulator (an IEEE divide there kept the
// epilogue, not the tensor cores, on the critical path of compute-bound tiles). For z below
// about -87 the result is -0 instead of a value under 1e-36 in magnitude.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ------------------------------------------------------------------ NVFP4 -> f16

// Two E2M1 codes (one byte, element 2j in the low nibble) -> f16x2 (element 2j in the low
// half), by the hardware conversion.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(d)
      : "r"(byte));
  return d;
}

// Two E4M3 codes (low 16 bits, the first in the low byte) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(d)
      : "r"(two));
  return d;
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  __half2 y = *reinterpret_cast<__half2*>(&b);
  __half2 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One weight row of a 64-element NVFP4 box -> f16, written as row `r` of a 128-byte-swizzled
// tile at `brow` (16-byte chunk c at ((c ^ (r % 8)) * 16)): 32 code bytes `crow` (element 2j
// in the low nibble), the 4 group scale codes `sc4` (first group in the low byte). Exact: an
// E2M1 value times an E4M3 scale has at most 5 significant bits and fits f16.
__device__ __forceinline__ void nvfp4_row_to_f16(const uint8_t* crow, uint32_t sc4, uint8_t* brow,
                                                 int r) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(crow);
  const uint4 c1 = *reinterpret_cast<const uint4*>(crow + 16);
  const uint32_t s01 = e4m3x2_to_f16x2(sc4), s23 = e4m3x2_to_f16x2(sc4 >> 16);
  const uint32_t scl[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232),
                           __byte_perm(s23, 0, 0x1010), __byte_perm(s23, 0, 0x3232)};
  const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t w = words[c];
    const uint32_t sc = scl[c >> 1];
    uint4 o;
    o.x = f16x2_mul(e2m1x2_to_f16x2(w), sc);
    o.y = f16x2_mul(e2m1x2_to_f16x2(w >> 8), sc);
    o.z = f16x2_mul(e2m1x2_to_f16x2(w >> 16), sc);
    o.w = f16x2_mul(e2m1x2_to_f16x2(w >> 24), sc);
    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = o;
  }
}

// ------------------------------------------------------------------ programmatic dependent launch

// Blocks until the preceding kernel of the stream has completed and its writes are visible
// (a no-op when this kernel was not launched as a programmatic dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel of the stream start launching once every block of this one got here.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ shared-memory addresses

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up after `limit` cycles,
// reports MOE_ERR_DEVICE_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, WsHeader* hdr,
                                          long long limit = kSpinLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      report_timeout(hdr);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled bulk-tensor load (x = innermost element coordinate, y = row) into shared memory,
// completing transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 1D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16), completing
// transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Allocates `ncols` TMEM columns (power of two >= 32); the base address is written to
// `*dst_smem`. Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart (stride byte offset), the
// leading byte offset unused for this layout, descriptor version 1, layout code 2.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);          // start address
  d |= (uint64_t)(16 >> 4) << 16;                       // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;                     // stride byte offset
  d |= (uint64_t)1 << 46;                               // descriptor version
  d |= (uint64_t)2 << 61;                               // 128-byte swizzle
  return d;
}

// Instruction descriptor: dense, fp32 accumulator, K-major A and B, shape M x N.
// a_fmt/b_fmt: kind::f16 -> 1 = bf16; kind::f8f6f4 -> 0 = E4M3.
__host__ __device__ constexpr uint32_t idesc_make(int M, int N, uint32_t a_fmt, uint32_t b_fmt) {
  return (1u << 4)                         // D format fp32
         | (a_fmt << 7) | (b_fmt << 10)    // operand formats
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma_fp8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma previously issued by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the async proxy (operands
// that tcgen05.mma will read through a shared-memory descriptor).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Each thread of the warp reads 16 consecutive fp32 columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Issues a read of 32 consecutive fp32 columns of this thread's TMEM lane; the values are
// valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tmem_wait_ld() that also ties the 32 registers a tmem_ld32_nowait() filled to the wait, so
// the compiler cannot move a use of them above it.
__device__ __forceinline__ void tmem_wait_ld_tied(float* v) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]),
        "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]),
        "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]),
        "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]), "+f"(v[24]),
        "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]), "+f"(v[30]),
        "+f"(v[31])
      :
      : "memory");
}

// Ties the 32 registers to an earlier wait without waiting again (no loads are outstanding).
__device__ __forceinline__ void tmem_tie(float* v) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                 "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                 "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                 "+f"(v[30]), "+f"(v[31])
               :
               : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Stores CHUNKS 16-byte chunks (8: 128 bytes, 4: 64 bytes) of each of the warp's 32 rows,
// lane l holding row l's chunks in pk, through the warp's staging area stg (32 * CHUNKS * 16
// bytes of shared memory): the rows are written there with their chunks XOR-swizzled (no bank
// conflicts either way), then every store instruction writes 32 / CHUNKS whole row segments.
// Row r goes to gcol + r * ld_bytes; rows r >= nvalid are skipped.
template <int CHUNKS>
__device__ __forceinline__ int staged_swizzle(int r) {
  return CHUNKS == 8 ? (r & 7) : ((r >> 1) & 3);
}

template <int CHUNKS>
__device__ __forceinline__ void warp_store_rows(uint8_t* stg, const uint4 (&pk)[CHUNKS],
                                                uint8_t* gcol, size_t ld_bytes, int nvalid) {
  static_assert(CHUNKS == 8 || CHUNKS == 4, "row segment of 64 or 128 bytes");
  constexpr int kRowBytes = CHUNKS * 16;
  constexpr int kRowsPerStore = 32 / CHUNKS;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < CHUNKS; ++j)
    *reinterpret_cast<uint4*>(stg + lane * kRowBytes + ((j ^ staged_swizzle<CHUNKS>(lane)) << 4)) =
        pk[j];
  __syncwarp();
  const int jj = lane % CHUNKS;
#pragma unroll
  for (int i = 0; i < CHUNKS; ++i) {
    const int r = i * kRowsPerStore + lane / CHUNKS;
    const uint4 v = *reinterpret_cast<const uint4*>(
        stg + r * kRowBytes + ((jj ^ staged_swizzle<CHUNKS>(r)) << 4));
    if (r < nvalid) *reinterpret_cast<uint4*>(gcol + (size_t)r * ld_bytes + jj * 16) = v;
  }
  __syncwarp();
}

}  // namespace moe
