/*
 * CPU oracle of the Mixture-of-Experts block forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 restatement of what the MoE block computes, used to check the CUDA
 * library. Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * it. It shares no code, header or table with the CUDA path.
 *
 * Sources (pages of MoE dispatch code from two LLM inference engines):
 *  - "metrale_model_layers/layers/moe/forward_prefill.rs" (`forward_prefill`): router GEMM
 *    with fixed accumulation order; softmax top-K; sort by expert; grouped gate/up,
 *    activation, grouped down; unpermute + weighted reduce (`moe_unpermute_reduce_indexed`);
 *    shared-expert blend `output += sigmoid(input . gate) * shared`, weight 1 without a gate
 *    (`moe_batched_blend`).
 *  - "spark_model/layers/moe/forward.rs" (`forward`, `apply_zero_expert`): softmax +
 *    correction bias used for SELECTION only, unbiased softmax x scaling for the weights;
 *    selected identity experts fold their weight into `zero_accum`, then
 *    `out[t,:] += zero_accum[t] * x[t,:]`; sigmoid+bias arm shows `topk(scores + bias)`,
 *    `scores[idx] / sum(scores[idx])` with `norm_topk_prob` toggling the divide.
 *  - "spark_model/layers/moe/forward_batched.rs": the router width is routed + zero
 *    experts ("the router also scores the zero-computation experts").
 *  - "spark_model/layers/moe/forward.rs" decode gate/up/down: SiLU(gate) * up, then down.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - softmax runs over all R router columns; ids E..R-1 are the identity experts;
 *  - top-K order: score descending, lower index first on equal scores;
 *  - the renormalising sum runs over all K selected slots, identity experts included;
 *  - the routing weight multiplies after the down projection;
 *  - SiLU(z) = z / (1 + exp(-z)); no clamp;
 *  - FP8 experts: input rows and the SwiGLU intermediate are quantised per 1x128 group along
 *    the contraction dim to E4M3 with scale = amax/448 (1 if amax == 0), the quantisation
 *    decided in fp32 (the kernel's precision); weights arrive as E4M3 codes with one fp32
 *    scale per 128x128 block. Everything after the quantisation is fp64.
 *  - NVFP4 experts (the decode page's packed weights + `scale_ptrs` + `scale2_vals` tables,
 *    "spark_model/layers/moe/forward.rs", NVFP4 decode arm): weight = E2M1 code x E4M3 scale
 *    of its group of 16 consecutive elements along the contraction x the matrix's fp32
 *    scale2; codes packed two per byte, element 2j in the low nibble. Activations stay bf16
 *    (the pages' w4a16 GEMV): nothing is quantised, everything is fp64.
 *
 * Parity pins: see the oracle tests (brute-force top-K, closed forms, dense SwiGLU through a
 * library matmul, exact identity-expert results, E4M3 against torch's float8 type, and a
 * second independent dense formulation).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- number formats */

double orc_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E2M1 (OCP MX FP4): bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa; exponent 0
 * encodes the subnormals 0 and 0.5; no infinities or NaN. */
double orc_e2m1_decode(uint8_t nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (OCP FP8, "fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; exponent 0 encodes subnormals m/8 * 2^-6. */
double orc_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to the nearest E4M3 value, ties to the even code (mantissa lsb 0), saturating to
 * +-448. Exhaustive over the 127 non-negative finite codes: slow and obviously right. */
uint8_t orc_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x80 : 0;
    double a = fabs(v);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            bestd = d;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

void orc_e4m3_encode_array(const double *v, long n, uint8_t *codes) {
    for (long i = 0; i < n; ++i) codes[i] = orc_e4m3_encode(v[i]);
}

/* Per-1x128 activation quantisation of `n` (multiple of 128) fp32 values: returns the
 * dequantised values (code * scale, exact in fp64). amax, the scale and the scaled value are
 * formed in fp32, as the kernel does. Writes the codes/scales if the pointers are given. */
static void quant_1x128(const float *v, int n, double *deq, uint8_t *codes, float *scales) {
    for (int g = 0; g < n / 128; ++g) {
        float amax = 0.0f;
        for (int j = 0; j < 128; ++j) {
            float a = fabsf(v[g * 128 + j]);
            if (a > amax) amax = a;
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        if (scales) scales[g] = s;
        for (int j = 0; j < 128; ++j) {
            float q = v[g * 128 + j] / s;
            uint8_t c = orc_e4m3_encode((double)q);
            if (codes) codes[g * 128 + j] = c;
            deq[g * 128 + j] = orc_e4m3_decode(c) * (double)s;
        }
    }
}

void orc_quant_1x128(const float *v, int n, uint8_t *codes, float *scales, double *deq) {
    quant_1x128(v, n, deq, codes, scales);
}

/* ---------------------------------------------------------------- routing */

typedef struct {
    int32_t num_tokens, hidden, num_experts, router_width, top_k, inter, shared_inter;
    int32_t scoring;          /* 0 softmax, 1 softmax + selection-only correction bias,
                                 2 sigmoid + selection-only correction bias */
    int32_t norm_topk_prob;
    double routed_scaling_factor;
    int32_t weight_dtype;     /* 0 bf16, 1 E4M3 + fp32 128x128 block scales, 2 NVFP4 */
    double rms_norm_eps;      /* with pre_expert_norm_w: epsilon of the pre-expert RMSNorm */
} orc_config_t;

typedef struct {
    const uint16_t *router_w;         /* bf16 [R,H] */
    const float *router_logit_bias;   /* [R] or NULL, added to the logits */
    const float *correction_bias;     /* [R] or NULL, selection only */
    const void *w_gate, *w_up, *w_down; /* bf16 or E4M3 [E,I,H], [E,I,H], [E,H,I] */
    const float *s_gate, *s_up, *s_down; /* [E,I/128,H/128], [E,I/128,H/128], [E,H/128,I/128] */
    const uint16_t *sh_gate, *sh_up, *sh_down; /* bf16 [S,H], [S,H], [H,S] */
    const uint16_t *sh_gate_vec;      /* bf16 [H] or NULL */
    const uint16_t *pre_expert_norm_w; /* bf16 [H] or NULL: RMSNorm of the routed experts' input */
    const uint8_t *sf_gate, *sf_up, *sf_down; /* NVFP4: E4M3 scale codes [E,rows,cols/16] */
    const float *scale2_gate, *scale2_up, *scale2_down; /* NVFP4: fp32 [E] */
} orc_weights_t;

/* Router logits of one token, fp64: L[r] = sum_h x[h] * Wr[r,h] (+ logit bias[r]). */
static void router_logits(const orc_config_t *c, const orc_weights_t *w, const double *x,
                          double *L) {
    int H = c->hidden, R = c->router_width;
    for (int r = 0; r < R; ++r) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h) acc += x[h] * orc_bf16_to_f64(w->router_w[(size_t)r * H + h]);
        if (w->router_logit_bias) acc += (double)w->router_logit_bias[r];
        L[r] = acc;
    }
}

/* Does candidate a rank before b? Higher selection score first, lower index on a tie. */
static int ranks_before(const double *sel, int a, int b) {
    return sel[a] > sel[b] || (sel[a] == sel[b] && a < b);
}

/* Scoring, top-K and weights of one token.
 * p = softmax(L) over all R columns (scoring 2: p[r] = sigmoid(L[r]) = 1 / (1 + e^-L[r]),
 * each column on its own, the decode page's sigmoid + correction-bias arm);
 * sel = p (+ correction bias); idx = K best by sel;
 * w = p[idx] (/ sum if norm_topk_prob) * routed_scaling_factor; zsum = sum of w on ids >= E.
 * gap = sel of the K-th choice minus sel of the (K+1)-th (INFINITY when K == R). */
static void route_token(const orc_config_t *c, const orc_weights_t *w, const double *L,
                        const int32_t *forced, int32_t *idx, double *wt, double *zsum,
                        double *gap, double *p, double *sel, char *taken) {
    int R = c->router_width, K = c->top_k, E = c->num_experts;
    if (c->scoring == 2) {
        for (int r = 0; r < R; ++r) p[r] = 1.0 / (1.0 + exp(-L[r]));
    } else {
        double mx = L[0];
        for (int r = 1; r < R; ++r) if (L[r] > mx) mx = L[r];
        double den = 0.0;
        for (int r = 0; r < R; ++r) { p[r] = exp(L[r] - mx); den += p[r]; }
        for (int r = 0; r < R; ++r) p[r] /= den;
    }
    for (int r = 0; r < R; ++r) {
        sel[r] = p[r];
        if ((c->scoring == 1 || c->scoring == 2) && w->correction_bias)
            sel[r] += (double)w->correction_bias[r];
    }
    for (int r = 0; r < R; ++r) taken[r] = 0;
    for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int r = 0; r < R; ++r)
            if (!taken[r] && (best < 0 || ranks_before(sel, r, best))) best = r;
        taken[best] = 1;
        idx[k] = best;
    }
    if (gap) {
        int next = -1;
        for (int r = 0; r < R; ++r)
            if (!taken[r] && (next < 0 || ranks_before(sel, r, next))) next = r;
        *gap = next < 0 ? INFINITY : sel[idx[K - 1]] - sel[next];
    }
    if (forced) for (int k = 0; k < K; ++k) idx[k] = forced[k];
    double sum = 0.0;
    for (int k = 0; k < K; ++k) { wt[k] = p[idx[k]]; sum += wt[k]; }
    for (int k = 0; k < K; ++k) {
        if (c->norm_topk_prob) wt[k] /= sum;
        wt[k] *= c->routed_scaling_factor;
    }
    double z = 0.0;
    for (int k = 0; k < K; ++k) if (idx[k] >= E) z += wt[k];
    *zsum = z;
}

/* ---------------------------------------------------------------- experts */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert weight matrix [E, rows, cols] and its scales (by weight dtype). */
typedef struct {
    const void *w;
    const float *s;        /* FP8: fp32 [E, rows/128, cols/128] */
    const uint8_t *sf;     /* NVFP4: E4M3 codes [E, rows, cols/16] */
    const float *scale2;   /* NVFP4: fp32 [E] */
} orc_mat_t;

/* Weight element (row, col) of expert e of a [E, rows, cols] matrix, decoded to fp64. */
static double wget(const orc_config_t *c, orc_mat_t m, int e, int rows, int cols, int row,
                   int col) {
    if (c->weight_dtype == 2) {
        uint8_t byte = ((const uint8_t *)m.w)[((size_t)e * rows + row) * (cols / 2) + col / 2];
        uint8_t nib = (col & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        uint8_t sc = m.sf[((size_t)e * rows + row) * (cols / 16) + col / 16];
        return orc_e2m1_decode(nib) * orc_e4m3_decode(sc) * (double)m.scale2[e];
    }
    size_t off = ((size_t)e * rows + row) * cols + col;
    if (c->weight_dtype == 0) return orc_bf16_to_f64(((const uint16_t *)m.w)[off]);
    double s = (double)m.s[((size_t)e * (rows / 128) + row / 128) * (cols / 128) + col / 128];
    return orc_e4m3_decode(((const uint8_t *)m.w)[off]) * s;
}

/* y[H] = (SiLU(xe . Wg_e^T) * (xe . Wu_e^T)) . Wd_e^T for routed expert e. `xe` is the
 * expert input (the token row, or its 1x128-quantised copy for FP8 experts). */
static void expert_ffn(const orc_config_t *c, const orc_weights_t *w, int e, const double *xe,
                       double *hbuf, float *hbuf32, double *y) {
    int H = c->hidden, I = c->inter;
    orc_mat_t mg = {w->w_gate, w->s_gate, w->sf_gate, w->scale2_gate};
    orc_mat_t mu = {w->w_up, w->s_up, w->sf_up, w->scale2_up};
    orc_mat_t md = {w->w_down, w->s_down, w->sf_down, w->scale2_down};
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += xe[h] * wget(c, mg, e, I, H, i, h);
            u += xe[h] * wget(c, mu, e, I, H, i, h);
        }
        hbuf[i] = silu(g) * u;
    }
    if (c->weight_dtype == 1) {
        /* the intermediate is quantised before the down projection, decided in fp32 */
        for (int i = 0; i < I; ++i) hbuf32[i] = (float)hbuf[i];
        quant_1x128(hbuf32, I, hbuf, NULL, NULL);
    }
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += hbuf[i] * wget(c, md, e, H, I, h, i);
        y[h] = acc;
    }
}

/* Shared expert: sh[H] = (SiLU(x . Sg^T) * (x . Su^T)) . Sd^T on the raw block input. */
static void shared_ffn(const orc_config_t *c, const orc_weights_t *w, const double *x,
                       double *hbuf, double *y) {
    int H = c->hidden, S = c->shared_inter;
    for (int s = 0; s < S; ++s) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += x[h] * orc_bf16_to_f64(w->sh_gate[(size_t)s * H + h]);
            u += x[h] * orc_bf16_to_f64(w->sh_up[(size_t)s * H + h]);
        }
        hbuf[s] = silu(g) * u;
    }
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int s = 0; s < S; ++s) acc += hbuf[s] * orc_bf16_to_f64(w->sh_down[(size_t)h * S + s]);
        y[h] = acc;
    }
}

/* ---------------------------------------------------------------- pre-expert norm */

/* Nearest bf16 (ties to even) of v taken to fp32 first: the normed copy of the pages is a
 * bf16 buffer written from fp32 arithmetic. */
static double round_bf16_via_f32(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Routed experts' input with a pre-expert norm ("metrale_model_layers/layers/moe/
 * forward_prefill.rs", `pre_expert_norm`: after routing, before expert dispatch; the router
 * and the shared-expert blend keep reading the un-normed input):
 * xn[h] = bf16( x[h] * g[h] / sqrt(mean_h x^2 + eps) ). */
static void pre_expert_rms_norm(const orc_config_t *c, const uint16_t *g, const double *x,
                                double *xn) {
    int H = c->hidden;
    double ss = 0.0;
    for (int h = 0; h < H; ++h) ss += x[h] * x[h];
    double inv = 1.0 / sqrt(ss / (double)H + c->rms_norm_eps);
    for (int h = 0; h < H; ++h) xn[h] = round_bf16_via_f32(x[h] * orc_bf16_to_f64(g[h]) * inv);
}

/* ---------------------------------------------------------------- the block forward */

/* Forward of the tokens listed in `tokens` (n_sel of them; NULL = all N in order).
 * x: bf16 [N,H]. forced_idx: NULL, or [N,K] expert ids that replace the selection (the
 * weights are then the (renormalised) probabilities of those ids).
 * Outputs, per listed token j: out[j,H] fp64, idx[j,K], w[j,K], zsum[j], gap[j], gamma[j],
 * sel[j,R] (the selection score of every router column).
 * Any output pointer may be NULL. Returns 0, or -1 on a bad argument. */
int orc_moe_forward(const orc_config_t *c, const orc_weights_t *w, const uint16_t *x,
                    int n_sel, const int32_t *tokens, const int32_t *forced_idx,
                    double *out, int32_t *idx_out, double *w_out, double *zsum_out,
                    double *gap_out, double *gamma_out, double *sel_out, int routing_only) {
    int N = c->num_tokens, H = c->hidden, R = c->router_width, K = c->top_k;
    int E = c->num_experts, I = c->inter, S = c->shared_inter;
    if (N < 0 || H <= 0 || E <= 0 || R < E || K <= 0 || K > R || K > 64 || I <= 0 || S < 0)
        return -1;
    if (c->weight_dtype == 1 && (H % 128 || I % 128)) return -1;
    if (c->weight_dtype == 2 && (H % 16 || I % 16 || !w->sf_gate || !w->sf_up || !w->sf_down ||
                                 !w->scale2_gate || !w->scale2_up || !w->scale2_down))
        return -1;
    if (c->weight_dtype < 0 || c->weight_dtype > 2) return -1;
    if (tokens == NULL) n_sel = N;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n_sel; ++j) {
        int t = tokens ? tokens[j] : j;
        if (t < 0 || t >= N) { bad = 1; continue; }
        int mx = H > R ? H : R;
        mx = mx > I ? mx : I;
        mx = mx > S ? mx : S;
        double *xt = malloc(sizeof(double) * H);
        double *xe = malloc(sizeof(double) * H);
        float *x32 = malloc(sizeof(float) * (size_t)mx);
        double *L = malloc(sizeof(double) * R), *p = malloc(sizeof(double) * R);
        double *sel = malloc(sizeof(double) * R);
        char *taken = malloc((size_t)R);
        double *hbuf = malloc(sizeof(double) * (size_t)mx);
        double *y = malloc(sizeof(double) * H);
        double *acc = malloc(sizeof(double) * H);
        int32_t idx[64];
        double wt[64], zsum = 0.0, gap = 0.0, gamma = 1.0;
        for (int h = 0; h < H; ++h) xt[h] = orc_bf16_to_f64(x[(size_t)t * H + h]);
        router_logits(c, w, xt, L);
        route_token(c, w, L, forced_idx ? forced_idx + (size_t)t * K : NULL, idx, wt, &zsum,
                    &gap, p, sel, taken);
        if (!routing_only) {
            /* the routed experts' input: x, or its pre-expert RMSNorm */
            if (w->pre_expert_norm_w) pre_expert_rms_norm(c, w->pre_expert_norm_w, xt, xe);
            else memcpy(xe, xt, sizeof(double) * H);
            if (c->weight_dtype == 1) {
                for (int h = 0; h < H; ++h) x32[h] = (float)xe[h];
                quant_1x128(x32, H, xe, NULL, NULL);
            }
            for (int h = 0; h < H; ++h) acc[h] = 0.0;
            for (int k = 0; k < K; ++k) {
                if (idx[k] >= E) continue;   /* identity expert: folded into zsum */
                expert_ffn(c, w, idx[k], xe, hbuf, x32, y);
                for (int h = 0; h < H; ++h) acc[h] += wt[k] * y[h];
            }
            for (int h = 0; h < H; ++h) acc[h] += zsum * xt[h];
            if (S > 0) {
                if (w->sh_gate_vec) {
                    double d = 0.0;
                    for (int h = 0; h < H; ++h) d += xt[h] * orc_bf16_to_f64(w->sh_gate_vec[h]);
                    gamma = 1.0 / (1.0 + exp(-d));
                }
                shared_ffn(c, w, xt, hbuf, y);
                for (int h = 0; h < H; ++h) acc[h] += gamma * y[h];
            }
            if (out) memcpy(out + (size_t)j * H, acc, sizeof(double) * H);
        }
        if (idx_out) memcpy(idx_out + (size_t)j * K, idx, sizeof(int32_t) * K);
        if (w_out) memcpy(w_out + (size_t)j * K, wt, sizeof(double) * K);
        if (zsum_out) zsum_out[j] = zsum;
        if (gap_out) gap_out[j] = gap;
        if (gamma_out) gamma_out[j] = gamma;
        if (sel_out) {
            /* route_token marks taken columns only in `taken`; sel itself is intact */
            memcpy(sel_out + (size_t)j * R, sel, sizeof(double) * R);
        }
        free(xt); free(xe); free(x32); free(L); free(p); free(sel); free(taken);
        free(hbuf); free(y); free(acc);
    }
    return bad ? -1 : 0;
}
