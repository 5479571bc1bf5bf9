/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts block forward.
 *
 * The operation is the MoE block forward of LLM serving, as dispatched by the pages
 * "metrale_model_layers/layers/moe/forward_prefill.rs" (`MoeLayer::forward_prefill`: shared
 * expert, router gate GEMM, top-K, sort by expert, grouped gate/up GEMM + activation, grouped
 * down GEMM, unpermute + weighted reduce, shared blend), "spark_model/layers/moe/forward.rs"
 * (`forward` single-token decode, softmax + correction-bias routing, `apply_zero_expert`) and
 * "metrale_model_layers/layers/moe/forward_atomic_c4.rs" (4-row decode with FP32 atomic
 * accumulation of the routed down projections, then a finalize that casts to BF16 and blends
 * the shared expert):
 *
 *   L[t,:]   = x[t,:] . Wr^T (+ router_logit_bias)                       fp32 accumulate
 *   p[t,:]   = softmax(L[t,:]) over all R router columns                  fp32
 *              (MOE_SCORING_SIGMOID_BIAS: p[t,r] = sigmoid(L[t,r]))
 *   idx[t,:] = top-K of p (or of p + correction_bias), ties to the lower id
 *   w[t,k]   = p[t,idx] (/ sum_k if norm_topk_prob) * routed_scaling_factor
 *   out[t,:] = sum_{k: idx<E} w[t,k] * (SiLU(x Wg_e^T) * (x Wu_e^T)) Wd_e^T
 *                                   (x = its pre-expert RMSNorm here when pre_expert_norm)
 *            + (sum_{k: idx>=E} w[t,k]) * x[t,:]            identity ("zero-computation") experts
 *            + gamma_t * (SiLU(x Sg^T) * (x Su^T)) Sd^T      shared expert, gamma_t = sigmoid(x.g)
 *                                                             or 1 when g is NULL
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major, with the contraction dim contiguous
 *    ([out_features, in_features], like an nn.Linear weight). bf16 is IEEE bfloat16; FP8 is
 *    OCP E4M3 ("e4m3fn").
 *  - The caller owns every buffer. The library allocates nothing, keeps no state between
 *    calls (apart from a per-process cache of CUDA device attributes), and never
 *    synchronises the host: all work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream), so a call can be captured into a CUDA graph.
 *  - Errors are returned as moe_status_t, never thrown; on a non-OK return nothing has been
 *    enqueued unless the status is MOE_ERR_CUDA (a launch failed part-way).
 *  - Device-side waits are bounded: a kernel that gives up writes MOE_ERR_DEVICE_TIMEOUT into
 *    the workspace status word (read it with moe_read_device_status) and returns.
 *  - Sizes: hidden, inter and shared_inter must be multiples of 128; 1 <= top_k <= 32,
 *    top_k <= router_width <= 1024, num_experts <= router_width, num_experts <= 1024.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_SCORING_SOFTMAX = 0,      /* p = softmax(L); select by p */
  MOE_SCORING_SOFTMAX_BIAS = 1, /* p = softmax(L); select by p + correction_bias; weights from p
                                   ("spark_model/layers/moe/forward.rs", LongCat arm) */
  MOE_SCORING_SIGMOID_BIAS = 2  /* p = sigmoid(L) per column; select by p + correction_bias;
                                   weights from p, renormalised over the K chosen when
                                   norm_topk_prob, times routed_scaling_factor (same page,
                                   DeepSeek-V3 / MiniMax-M2 arm); router_width == num_experts */
} moe_scoring_t;

typedef enum {
  MOE_W_BF16 = 0,               /* routed expert weights bf16 */
  MOE_W_FP8_E4M3_B128 = 1,      /* routed expert weights E4M3 + one fp32 scale per 128x128 block;
                                   expert inputs and the SwiGLU intermediate are quantised per
                                   1x128 (along the contraction) to E4M3, scale = amax/448 */
  MOE_W_NVFP4 = 2               /* routed expert weights NVFP4: E2M1 codes packed two per byte
                                   (element 2j in the low nibble), one E4M3 scale per 16
                                   consecutive elements along the contraction (sf_*), one fp32
                                   scale2 per expert matrix; weight = e2m1 * sf * scale2.
                                   Activations are not quantised: the experts read x (or xn)
                                   and the SwiGLU intermediate as f16, exact for bf16 values
                                   of magnitude in [2^-14, 65504] (larger overflow). Needs
                                   hidden and inter multiples of 256; both chains
                                   ("spark_model/layers/moe/forward.rs", NVFP4 decode arm:
                                   packed, scale and scale2 tables) */
} moe_wdtype_t;

typedef enum {
  MOE_PATH_AUTO = 0,            /* decode chain for num_tokens <= 16 (inter and shared_inter
                                   <= 1024; E4M3 and NVFP4 experts: hidden % 256 == 0) when the
                                   weights the batch may touch -- min(num_experts, num_tokens *
                                   top_k) experts' three matrices plus the shared expert's --
                                   come to at least 8 MiB; else grouped */
  MOE_PATH_DECODE = 1,          /* one cooperative kernel: routing, tcgen05 projections streaming
                                   each touched expert's weights once, combine (bf16, E4M3 or
                                   NVFP4 experts, num_tokens <= 16, inter and shared_inter <=
                                   1024) */
  MOE_PATH_GROUPED = 2          /* sort + tcgen05 grouped GEMM chain (any num_tokens) */
} moe_path_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* NULL where a pointer is required, negative size, ... */
  MOE_ERR_UNSUPPORTED = 2,          /* valid but not implemented (e.g. hidden % 128 != 0) */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < moe_workspace_size() */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_TIMEOUT = 5        /* a bounded device wait gave up (reported on device) */
} moe_status_t;

typedef struct {
  int32_t num_tokens;    /* N >= 0 */
  int32_t hidden;        /* H */
  int32_t num_experts;   /* E: SwiGLU experts, ids 0..E-1 */
  int32_t router_width;  /* R >= E: router columns; ids E..R-1 are identity experts.
                            R > E requires MOE_SCORING_SOFTMAX_BIAS (the pages wire identity
                            experts only on that arm); otherwise MOE_ERR_UNSUPPORTED */
  int32_t top_k;         /* K */
  int32_t inter;         /* I: routed expert intermediate size */
  int32_t shared_inter;  /* S: shared expert intermediate size, 0 = no shared expert */
  int32_t scoring;       /* moe_scoring_t */
  int32_t norm_topk_prob;          /* nonzero: renormalise the K weights to sum 1 */
  float routed_scaling_factor;     /* multiplies every routing weight */
  int32_t weight_dtype;  /* moe_wdtype_t */
  int32_t deterministic; /* nonzero: bitwise run-to-run reproducible (slot-ordered reduction;
                            partial sums meet pairwise, a + b == b + a); 0: the decode chain
                            accumulates the weighted routed down projections into [N,H] with
                            FP32 atomics in any order */
  int32_t path;          /* moe_path_t */
  int32_t pre_expert_norm; /* nonzero: the routed experts read RMSNorm(x) (weights
                              pre_expert_norm_w), xn = bf16(x * g / sqrt(mean(x^2) + eps)),
                              while the router, the shared expert and its gate and the identity
                              experts read x ("metrale_model_layers/layers/moe/
                              forward_prefill.rs", `pre_expert_norm`) */
  float rms_norm_eps;      /* eps of that norm (>= 0) */
} moe_config_t;

typedef struct {
  const void *router_w;            /* bf16 [R,H] */
  const float *router_logit_bias;  /* nullable fp32 [R], added to the logits before softmax */
  const float *correction_bias;    /* fp32 [R], required by the *_BIAS scorings (selection only),
                                      ignored with MOE_SCORING_SOFTMAX */
  const void *w_gate;              /* [E,I,H] bf16 or E4M3; NVFP4: packed [E,I,H/2] */
  const void *w_up;                /* [E,I,H] bf16 or E4M3; NVFP4: packed [E,I,H/2] */
  const void *w_down;              /* [E,H,I] bf16 or E4M3; NVFP4: packed [E,H,I/2] */
  const float *s_gate;             /* FP8 only: fp32 [E,I/128,H/128] */
  const float *s_up;               /* FP8 only: fp32 [E,I/128,H/128] */
  const float *s_down;             /* FP8 only: fp32 [E,H/128,I/128] */
  const void *sh_gate;             /* bf16 [S,H]; NULL iff S == 0 */
  const void *sh_up;               /* bf16 [S,H] */
  const void *sh_down;             /* bf16 [H,S] */
  const void *sh_gate_vec;         /* nullable bf16 [H]: shared blend weight sigmoid(x . g);
                                      NULL = weight 1 */
  const void *pre_expert_norm_w;   /* bf16 [H], required iff pre_expert_norm */
  const void *sf_gate;             /* NVFP4 only: E4M3 codes [E,I,H/16] */
  const void *sf_up;               /* NVFP4 only: E4M3 codes [E,I,H/16] */
  const void *sf_down;             /* NVFP4 only: E4M3 codes [E,H,I/16] */
  const float *scale2_gate;        /* NVFP4 only: fp32 [E] */
  const float *scale2_up;          /* NVFP4 only: fp32 [E] */
  const float *scale2_down;        /* NVFP4 only: fp32 [E] */
} moe_weights_t;

/* Bytes of device workspace moe_forward / moe_route need for `cfg` (path resolved as in
 * moe_forward). Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a config they reject. */
MOE_API moe_status_t moe_workspace_size(const moe_config_t *cfg, size_t *bytes);

/* The whole block forward (all steps above) on `stream`.
 *  x          bf16 [N,H] device, read only; must not overlap `out`.
 *  out        bf16 [N,H] device, fully overwritten (FP32 accumulation, one rounding to bf16).
 *  workspace  device scratch of >= moe_workspace_size() bytes, 256-byte aligned; its contents
 *             on entry do not matter; it must not be used by another call still in flight.
 *  topk_idx_out / topk_w_out  nullable uint32 / fp32 [N,K]: the routing actually used.
 *  forced_idx nullable uint32 [N,K] expert ids (< router_width) that replace the top-K
 *             selection (test hook; the weights are then the probabilities of those ids,
 *             renormalised as configured).
 * Pages: forward_prefill.rs `forward_prefill` (prefill chain), forward.rs `forward`
 * (decode), forward_atomic_c4.rs (atomic decode accumulation), forward.rs `apply_zero_expert`. */
MOE_API moe_status_t moe_forward(const moe_config_t *cfg, const moe_weights_t *weights, const void *x,
                         void *out, void *workspace, size_t workspace_bytes, void *stream,
                         uint32_t *topk_idx_out, float *topk_w_out, const uint32_t *forced_idx);

/* Routing steps only (router GEMM, scoring + top-K + weights, identity-expert sum, and the
 * stable sort of the (token, slot) pairs by expert), for inspection and tests. Each output
 * pointer is a nullable device buffer:
 *  idx_out uint32 [N,K], w_out fp32 [N,K], zsum_out fp32 [N] (summed identity-expert weight),
 *  offsets_out uint32 [E+1] (row offset of each expert in the sorted order),
 *  sorted_pairs_out uint32 [N*K] (flat pair index t*K+k of each sorted row; entries past
 *  offsets[E] are unspecified), pair_to_row_out uint32 [N*K] (sorted row of each pair,
 *  0xFFFFFFFF for identity-expert pairs). Within an expert, rows keep the pair order.
 * Pages: forward_prefill.rs gate GEMM / top-K / `moe_sort_by_expert`. */
MOE_API moe_status_t moe_route(const moe_config_t *cfg, const moe_weights_t *weights, const void *x,
                       void *workspace, size_t workspace_bytes, void *stream,
                       uint32_t *idx_out, float *w_out, float *zsum_out, uint32_t *offsets_out,
                       uint32_t *sorted_pairs_out, uint32_t *pair_to_row_out);

/* Stages of one forward, in launch order, for moe_forward_profiled. The decode chain is one
 * kernel: its ROUTE stage is the memset of the workspace header, its GATE_UP stage the kernel
 * (routing, both projections, the shared expert and the combine), the other stages empty. */
typedef enum {
  MOE_STAGE_ROUTE = 0,     /* router GEMM, scoring + top-K, sort (+ gather of expert rows) */
  MOE_STAGE_SHARED = 1,    /* shared expert gate/up + down (grouped chain) */
  MOE_STAGE_GATE_UP = 2,   /* routed gate/up projection with fused SiLU(gate) * up */
  MOE_STAGE_DOWN = 3,      /* routed down projection */
  MOE_STAGE_COMBINE = 4,   /* unpermute + weighted reduce + identity add + shared blend */
  MOE_NUM_STAGES = 5
} moe_stage_t;

/* moe_forward that also records `events[2*s]` before and `events[2*s+1]` after stage s on
 * `stream` (events: MOE_NUM_STAGES*2 cudaEvent_t handles created by the caller; NULL entries
 * are skipped). For measuring per-kernel durations; results are identical to moe_forward. */
MOE_API moe_status_t moe_forward_profiled(const moe_config_t *cfg, const moe_weights_t *weights,
                                          const void *x, void *out, void *workspace,
                                          size_t workspace_bytes, void *stream, void **events);

/* The decode chain of moe_forward (bf16 experts, num_tokens <= 16) for callers that cannot
 * allocate device memory: a plugin hosted by another runtime that owns every allocation and
 * offers no allocator, or a latency-critical loop that may not call cudaMalloc because it can
 * synchronise the whole device. The pages have no counterpart; it exists for such callers.
 * Instead of a caller workspace it uses one 4 MiB scratch array that the CUDA driver places in
 * device memory when it loads this library's device code (every GPU that loads it holds the
 * array until the process exits). It allocates nothing and calls no allocating routine.
 *  - cfg->path must be MOE_PATH_AUTO or MOE_PATH_DECODE; the decode chain is always used.
 *  - Configurations whose scratch would exceed 4 MiB return MOE_ERR_WORKSPACE_TOO_SMALL
 *    (moe_workspace_size() with path = MOE_PATH_DECODE gives the bytes needed); grouped-only
 *    configurations return MOE_ERR_UNSUPPORTED.
 *  - The first call on each device looks up the array's device address (with that device
 *    current); make that first call before any stream capture. The address is kept for the
 *    life of the process: do not use this entry point on a device after cudaDeviceReset()
 *    (the library's device code is then loaded anew and the kept address is stale).
 *  - Every call shares the array and clears what must start at zero itself; calls that
 *    overlap on the GPU (unordered streams or host threads) race on it.
 *  - There is no caller workspace: moe_noalloc_read_device_status() reads this call's device
 *    status word (a device wait that times out still ends its kernel).
 * x, out, stream and the weights are as for moe_forward. */
MOE_API moe_status_t moe_forward_decode_noalloc(const moe_config_t *cfg,
                                                const moe_weights_t *weights, const void *x,
                                                void *out, void *stream);

/* Synchronises `stream` and reads the device status word of `workspace` into *status
 * (MOE_OK or MOE_ERR_DEVICE_TIMEOUT). For tests and debugging; it blocks the host. */
MOE_API moe_status_t moe_read_device_status(const void *workspace, void *stream, int32_t *status);

/* The same for moe_forward_decode_noalloc: synchronises `stream` and reads the status word of
 * the library's 4 MiB array on the current device, i.e. of the last no-alloc call there
 * (each call clears it first, so read it before the next call). */
MOE_API moe_status_t moe_noalloc_read_device_status(void *stream, int32_t *status);

/* Failure-detection self test: clears the workspace status word, then one device thread waits
 * (with the same bounded wait every kernel here uses) on a barrier that nothing completes,
 * giving up after `limit_cycles` SM clock cycles (1 <= limit_cycles <= 2e9). Afterwards
 * moe_read_device_status() reports MOE_ERR_DEVICE_TIMEOUT and the CUDA context stays usable.
 * workspace: >= 256 bytes, 256-byte aligned. */
MOE_API moe_status_t moe_selftest_bounded_wait(void *workspace, long long limit_cycles,
                                               void *stream);

/* After MOE_ERR_CUDA: the failing CUDA call and its error text, for the calling thread
 * (empty string if none failed). The pointer stays valid until the thread's next call. */
MOE_API const char *moe_last_error_detail(void);

/* Static description of a status code. */
MOE_API const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
