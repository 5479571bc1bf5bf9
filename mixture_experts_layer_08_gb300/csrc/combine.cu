// Unpermute + weighted reduce + identity-expert add + shared-expert blend, one pass over
// the output.
//
// Pages: "metrale_model_layers/layers/moe/forward_prefill.rs" (`moe_unpermute_reduce_indexed`:
// out[t] = sum_k w[t,k] * y[token_to_perm[t*K+k]]; `moe_batched_blend`: out += sigmoid(input .
// gate) * shared, weight 1 without a gate), "spark_model/layers/moe/forward.rs"
// (`apply_zero_expert`: out[t,:] += zero_accum[t] * x[t,:] after the routed blend;
// `moe_weighted_sum_blend` computes the gate scalar inline in every block) and
// "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (finalize: bf16(accumulator + shared)).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kCombThreads = 256;

template <bool F32>
struct Row8;      // 8 consecutive outputs of one row, loaded raw then widened

template <>
struct Row8<false> {
  uint4 v;
  __device__ __forceinline__ void load(const void* base, size_t off) {
    v = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
  }
  __device__ __forceinline__ void widen(float* f) const { bf16x8_to_f32(v, f); }
};

template <>
struct Row8<true> {
  float4 a, b;
  __device__ __forceinline__ void load(const void* base, size_t off) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    a = p[0];
    b = p[1];
  }
  __device__ __forceinline__ void widen(float* f) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

// Block (t, part): 8 consecutive outputs per thread of token t. YF32 / SF32: the expert rows
// and the shared-expert row are fp32 (decode chain) or bf16 (grouped chain).
template <bool YF32, bool SF32>
__global__ void __launch_bounds__(kCombThreads) combine_kernel(CombineArgs a) {
  __shared__ float red[kCombThreads / 32];
  const int t = blockIdx.x;
  const int H = a.H;
  const __nv_bfloat16* xt = a.x + (size_t)t * H;
  float gamma = 1.0f;
  if (a.shy && a.sh_gate_vec) {
    // blend weight sigmoid(x[t] . g), recomputed by every block of the token
    float d = 0.0f;
    for (int c = threadIdx.x; c < H / 8; c += kCombThreads) {
      float xf[8], gf[8];
      bf16x8_to_f32(reinterpret_cast<const uint4*>(xt)[c], xf);
      bf16x8_to_f32(reinterpret_cast<const uint4*>(a.sh_gate_vec)[c], gf);
#pragma unroll
      for (int i = 0; i < 8; ++i) d = fmaf(xf[i], gf[i], d);
    }
    d = warp_sum(d);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = d;
    __syncthreads();
    d = 0.0f;
#pragma unroll
    for (int i = 0; i < kCombThreads / 32; ++i) d += red[i];
    gamma = 1.0f / (1.0f + expf(-d));
  }
  const int c = blockIdx.y * kCombThreads + threadIdx.x;    // chunk of 8 outputs
  const bool on = c < H / 8;
  const size_t h0 = (size_t)c * 8;
  // Everything produced before the expert projections (routing, x) is read before waiting on
  // the previous kernel: it finished at least two launches back.
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  if (a.zsum) {   // (null without identity experts: no x read)
    const float z = a.zsum[t];
    float xf[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xf[i] = 0.0f;
    if (on) bf16x8_to_f32(reinterpret_cast<const uint4*>(xt)[c], xf);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = z * xf[i];
  }
  pdl_wait();     // expert outputs of the previous kernel
  if (!on) return;
  if (a.acc) {
    Row8<true> r;
    r.load(a.acc, (size_t)t * H + h0);
    float f[8];
    r.widen(f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  if (a.y) {
    // 4 expert rows in flight per round, loaded before any of them is used
    for (int k0 = 0; k0 < a.K; k0 += 4) {
      Row8<YF32> rows[4];
      float wk[4];
      bool live[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + u;
        const uint32_t row = k < a.K ? a.pair_to_row[t * a.K + k] : kNoRow;
        live[u] = row != kNoRow;     // identity-expert slots have no expert row
        wk[u] = live[u] ? a.w[t * a.K + k] : 0.0f;
        if (live[u]) rows[u].load(a.y, (size_t)row * H + h0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (live[u]) {
          float yf[8];
          rows[u].widen(yf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wk[u], yf[i], acc[i]);
        }
      }
    }
  }
  if (a.shy) {
    Row8<SF32> r;
    r.load(a.shy, (size_t)t * H + h0);
    float sf[8];
    r.widen(sf);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(gamma, sf[i], acc[i]);
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(a.out + (size_t)t * H)[c] = o;
}

// One thread waits, with the library's bounded wait, on an mbarrier nothing arrives on.
__global__ void bounded_wait_selftest_kernel(WsHeader* hdr, long long limit_cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbarrier_init();
  mbar_wait(&bar, 0, hdr, limit_cycles);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(WsHeader* hdr, long long limit_cycles, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(hdr, limit_cycles);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  dim3 grid(a.N, (a.H / 8 + kCombThreads - 1) / kCombThreads);
  if (a.y_is_f32 != a.shy_is_f32 && a.shy) return cudaErrorInvalidValue;
  if (a.y_is_f32) return launch_dependent(combine_kernel<true, true>, grid, dim3(kCombThreads), 0, st, a);
  return launch_dependent(combine_kernel<false, false>, grid, dim3(kCombThreads), 0, st, a);
}

}  // namespace moe
