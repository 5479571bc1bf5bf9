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

__device__ __forceinline__ void load8(const void* base, int is_f32, size_t off, float* f) {
  if (is_f32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = p[0], b = p[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off),
                  f);
  }
}

// Block (t, part): 8 consecutive outputs per thread of token t.
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
  if (c >= H / 8) return;
  const size_t h0 = (size_t)c * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  if (a.acc) {
    load8(a.acc, 1, (size_t)t * H + h0, acc);
  }
  if (a.y) {
    // all of the token's expert rows in flight at once: 8 slots per round
    for (int k0 = 0; k0 < a.K; k0 += 8) {
      float yf[8][8];
      float wk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u;
        const uint32_t row = k < a.K ? a.pair_to_row[t * a.K + k] : kNoRow;
        wk[u] = row != kNoRow ? a.w[t * a.K + k] : 0.0f;
        if (row != kNoRow) load8(a.y, a.y_is_f32, (size_t)row * H + h0, yf[u]);
        else
#pragma unroll
          for (int i = 0; i < 8; ++i) yf[u][i] = 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wk[u], yf[u][i], acc[i]);
    }
  }
  {
    const float z = a.zsum[t];
    float xf[8];
    bf16x8_to_f32(reinterpret_cast<const uint4*>(xt)[c], xf);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(z, xf[i], acc[i]);
  }
  if (a.shy) {
    float sf[8];
    load8(a.shy, a.shy_is_f32, (size_t)t * H + h0, sf);
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
  combine_kernel<<<grid, kCombThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
