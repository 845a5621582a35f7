/*
 * moe_oracle.c -- plain, slow CPU oracle for the DeepSeek-style MoE FFN forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: it exists so that tests, the smoke check and the CPU-baseline leg of the bench
 * can check the CUDA library against an independent statement of what the layer
 * computes.  It shares no code, header, table or constant with the CUDA sources.
 *
 * Sources (page title, section):
 *   [gate]  "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)",
 *           sections "API" and "Algorithm (mlx-lm group_expert_select)", and the review
 *           sections "What looks solid" 1-2 and "Non-issues".
 *   [epic]  "Epic: Engine Inference Core Stage E - MoE + hybrid families", the first
 *           paragraph (expert dispatch through gather_mm / gather_qmm) and "Decision 5"
 *           (target checkpoint is 4-bit affine-quantised).
 *   [arch]  the same PR, review section "Architecture and design" (route -> switch_glu ->
 *           combine with an always-active, ungated shared expert checked against a manual
 *           SwiGLU reference).
 *
 * Precision: the gate works in fp32 because the algorithm casts the router logits to f32
 * before the sigmoid ([gate] Algorithm, first line).  The expert FFN, whose precision the
 * pages leave open, is evaluated in double on bf16-exact (or dequantised) operands; the
 * intermediate h is not rounded.
 *
 * Readings where the pages are silent, named R<n> where the code below applies them:
 *   R1 order within the K selected experts: descending biased score, ties to the lower
 *      expert index (the reference's argpartition leaves the order unspecified);
 *   R2 group-drop ties: among groups of equal group score the lower group index is kept;
 *   R3 NaN is the lowest value in every comparison; -0.0 compares equal to +0.0;
 *   R4 SwiGLU form: FFN(v) = W_down (silu(W_gate v) * (W_up v)), silu(a) = a / (1 + e^-a);
 *   R5 4-bit packing: element j of a row lives in 32-bit word j/8, bits 4*(j%8) .. +3
 *      (low nibble first); w = scale * q + bias with the fp16 scale and bias of element j's
 *      group of consecutive inputs (64 unless the weights say 32 or 128);
 *   R6 the permutation lists the pairs p = t*K + k sorted by (expert, p);
 *   R19 softmax route: the K largest logits are selected (ties as R1) and their weights are
 *      the softmax over the selected logits only, i.e. always renormalised;
 *   R25 8-bit packing: element j of a row lives in 32-bit word j/4, bits 8*(j%4) .. +7 (low
 *      byte first); groups of 32, 64 or 128 inputs share one fp16 scale and bias.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* scalar conversions                                                                   */
/* ------------------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32 pattern. */
float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary16 -> binary32, written out from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
float oracle_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 / 2^10 */
    } else if (exp == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)frac / 1024.0, exp - 15);
    }
    return (float)(sign ? -v : v);
}

/* ------------------------------------------------------------------------------------ */
/* route ([gate] Algorithm)                                                             */
/* ------------------------------------------------------------------------------------ */

/* "a is preferred over b" for values with indices (R1/R3): larger value first, NaN last,
 * equal values go to the lower index. */
static int route_better(float a, int ia, float b, int ib) {
    int an = isnan(a), bn = isnan(b);
    if (an || bn) {
        if (an && bn) return ia < ib;
        return bn; /* a is a number and b is NaN */
    }
    if (a > b) return 1;
    if (a < b) return 0;
    return ia < ib;
}

int oracle_route_row(const float* logits, int E, const float* bias, int top_k, int n_group,
                     int topk_group, int norm_topk_prob, float routed_scaling_factor,
                     int32_t* inds, float* scores) {
    float* orig = (float*)malloc(sizeof(float) * (size_t)E);
    float* biased = (float*)malloc(sizeof(float) * (size_t)E);
    char* taken = (char*)calloc((size_t)E, 1);
    if (!orig || !biased || !taken) {
        free(orig); free(biased); free(taken);
        return -1;
    }
    /* scores = sigmoid(f32(gates)); orig = scores */
    for (int e = 0; e < E; ++e) {
        float s = 1.0f / (1.0f + expf(-logits[e]));
        orig[e] = s;
        /* scores = scores + bias   (selection only) */
        biased[e] = s + bias[e];
    }
    /* if n_group > 1: group score = sum of the two largest biased scores of the group;
     * zero the experts of the k_drop = n_group - topk_group worst groups. */
    int k_drop = n_group - topk_group;
    if (n_group > 1 && k_drop > 0) {
        int eg = E / n_group;
        float* gs = (float*)malloc(sizeof(float) * (size_t)n_group);
        char* keep = (char*)calloc((size_t)n_group, 1);
        for (int g = 0; g < n_group; ++g) {
            /* two largest (with multiplicity) of the group */
            int i1 = -1, i2 = -1;
            for (int j = 0; j < eg; ++j) {
                int e = g * eg + j;
                if (i1 < 0 || route_better(biased[e], e, biased[i1], i1)) {
                    i2 = i1;
                    i1 = e;
                } else if (i2 < 0 || route_better(biased[e], e, biased[i2], i2)) {
                    i2 = e;
                }
            }
            gs[g] = biased[i1] + biased[i2];
        }
        /* keep the topk_group best groups (R2) */
        for (int r = 0; r < topk_group; ++r) {
            int best = -1;
            for (int g = 0; g < n_group; ++g)
                if (!keep[g] && (best < 0 || route_better(gs[g], g, gs[best], best))) best = g;
            keep[best] = 1;
        }
        for (int g = 0; g < n_group; ++g)
            if (!keep[g])
                for (int j = 0; j < eg; ++j) biased[g * eg + j] = 0.0f;
        free(gs);
        free(keep);
    }
    /* inds = topk(biased scores), in the order of R1 */
    for (int k = 0; k < top_k; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || route_better(biased[e], e, biased[best], best))) best = e;
        taken[best] = 1;
        inds[k] = best;
        /* scores = take_along(orig, inds): the pre-bias sigmoid */
        scores[k] = orig[best];
    }
    /* renormalise only when top_k > 1 and norm_topk_prob; no zero-sum guard */
    if (top_k > 1 && norm_topk_prob) {
        float sum = 0.0f;
        for (int k = 0; k < top_k; ++k) sum += scores[k];
        for (int k = 0; k < top_k; ++k) scores[k] = scores[k] / sum;
    }
    for (int k = 0; k < top_k; ++k) scores[k] = scores[k] * routed_scaling_factor;
    free(orig);
    free(biased);
    free(taken);
    return 0;
}

int oracle_route(const float* logits, int64_t rows, int E, const float* bias, int top_k,
                 int n_group, int topk_group, int norm_topk_prob, float routed_scaling_factor,
                 int32_t* inds, float* scores) {
    if (!logits || !bias || !inds || !scores) return -1;
    if (top_k < 1 || top_k > E || n_group < 1 || E % n_group != 0) return -1;
    if (topk_group < 1 || topk_group > n_group) return -1;
    if (n_group > 1 && E / n_group < 2) return -1;
    int rc = 0;
#pragma omp parallel for schedule(static) reduction(| : rc)
    for (int64_t r = 0; r < rows; ++r)
        rc |= oracle_route_row(logits + r * E, E, bias, top_k, n_group, topk_group,
                               norm_topk_prob, routed_scaling_factor, inds + r * top_k,
                               scores + r * top_k);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* softmax route ([gate] "Scope decisions" and review "What looks solid" 1: the softmax */
/* route of the generic MoE block always renormalises its top-k weights)                */
/* ------------------------------------------------------------------------------------ */

/* R19: softmax is strictly increasing in the logit, so the K most probable experts are the
 * K largest logits (ties to the lower index, R1); the renormalised weight of a selected
 * expert, p_k / sum_sel p_j, is exp(l_k - l_max) / sum_sel exp(l_j - l_max), which does not
 * depend on the full softmax denominator.  fp32 throughout, sum left to right over k. */
int oracle_route_softmax_row(const float* logits, int E, int top_k, int32_t* inds,
                             float* scores) {
    char* taken = (char*)calloc((size_t)E, 1);
    if (!taken) return -1;
    for (int k = 0; k < top_k; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || route_better(logits[e], e, logits[best], best))) best = e;
        taken[best] = 1;
        inds[k] = best;
    }
    float lmax = logits[inds[0]];
    float sum = 0.0f;
    for (int k = 0; k < top_k; ++k) {
        scores[k] = expf(logits[inds[k]] - lmax);
        sum += scores[k];
    }
    for (int k = 0; k < top_k; ++k) scores[k] = scores[k] / sum;
    free(taken);
    return 0;
}

int oracle_route_softmax(const float* logits, int64_t rows, int E, int top_k, int32_t* inds,
                         float* scores) {
    if (!logits || !inds || !scores || top_k < 1 || top_k > E) return -1;
    int rc = 0;
#pragma omp parallel for schedule(static) reduction(| : rc)
    for (int64_t r = 0; r < rows; ++r)
        rc |= oracle_route_softmax_row(logits + r * E, E, top_k, inds + r * top_k,
                                       scores + r * top_k);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* token -> expert dispatch (R6)                                                        */
/* ------------------------------------------------------------------------------------ */

int oracle_permute(const int32_t* inds, int64_t T, int K, int E, int32_t* counts,
                   int32_t* offsets, int32_t* perm, int32_t* inv_perm) {
    int64_t P = T * K;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) {
        if (inds[p] < 0 || inds[p] >= E) return -1;
        counts[inds[p]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* walk the pairs in increasing p: within an expert, slots fill in pair order */
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    if (!fill) return -1;
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t p = 0; p < P; ++p) {
        int32_t j = fill[inds[p]]++;
        perm[j] = (int32_t)p;
        inv_perm[p] = j;
    }
    free(fill);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* router linear                                                                        */
/* ------------------------------------------------------------------------------------ */

/* logits[t, e] = sum_i x[t, i] * w_router[e, i] (+ logit_offset[e]); bf16 operands,
 * double accumulation, fp32 result. */
void oracle_router_logits(const uint16_t* x, int64_t T, int d, const uint16_t* w_router,
                          int E, const float* logit_offset, float* logits) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += (double)oracle_bf16_to_f32(x[t * d + i]) *
                       (double)oracle_bf16_to_f32(w_router[(int64_t)e * d + i]);
            if (logit_offset) acc += (double)logit_offset[e];
            logits[t * E + e] = (float)acc;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* expert weights: bf16 rows or affine 4-bit rows (R5)                                  */
/* ------------------------------------------------------------------------------------ */

/* One weight matrix [rows, cols] of one expert.  bits == 16: w16 holds bf16 [rows, cols].
 * bits == 4 or 8: q holds uint32 [rows, cols*bits/32] (32/bits codes per word, element j in
 * bits bits*(j % (32/bits)) .. upward of word j / (32/bits): R5 and, for 8 bits, R25);
 * scale and bias hold fp16 [rows, cols/group]. */
typedef struct {
    int bits;
    int group;
    const uint16_t* w16;
    const uint32_t* q;
    const uint16_t* scale;
    const uint16_t* bias;
} oracle_mat_t;

/* w = scale * q + bias, in fp32, element (r, c) of a `bits`-bit affine matrix with `cols`
 * columns ([epic] first paragraph: quantised experts through gather_qmm). */
float oracle_q_element(int bits, const uint32_t* q, const uint16_t* scale,
                       const uint16_t* bias, int64_t r, int64_t c, int64_t cols, int group) {
    const int per = 32 / bits;
    uint32_t word = q[r * (cols / per) + c / per];
    uint32_t code = (word >> (bits * (c % per))) & ((1u << bits) - 1u);
    int64_t ng = cols / group;
    float s = oracle_f16_to_f32(scale[r * ng + c / group]);
    float b = oracle_f16_to_f32(bias[r * ng + c / group]);
    return s * (float)code + b;
}

float oracle_q4_element(const uint32_t* q, const uint16_t* scale, const uint16_t* bias,
                        int64_t r, int64_t c, int64_t cols, int group) {
    return oracle_q_element(4, q, scale, bias, r, c, cols, group);
}

void oracle_dequant(int bits, const uint32_t* q, const uint16_t* scale, const uint16_t* bias,
                    int64_t rows, int64_t cols, int group, float* out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = oracle_q_element(bits, q, scale, bias, r, c, cols, group);
}

void oracle_dequant_q4(const uint32_t* q, const uint16_t* scale, const uint16_t* bias,
                       int64_t rows, int64_t cols, int group, float* out) {
    oracle_dequant(4, q, scale, bias, rows, cols, group, out);
}

static double mat_elem(const oracle_mat_t* m, int64_t r, int64_t c, int64_t cols) {
    if (m->bits == 16) return (double)oracle_bf16_to_f32(m->w16[r * cols + c]);
    return (double)oracle_q_element(m->bits, m->q, m->scale, m->bias, r, c, cols, m->group);
}

/* Expert FFN on one bf16 vector v[d]:  out = W_down (silu(W_gate v) * (W_up v)).
 * W_gate, W_up are [I, d]; W_down is [d, I].  Accumulates into out (double). */
static void expert_ffn(const uint16_t* v, int d, int I, const oracle_mat_t* wg,
                       const oracle_mat_t* wu, const oracle_mat_t* wd, double weight,
                       double* out, double* h) {
    for (int n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
            double vi = (double)oracle_bf16_to_f32(v[i]);
            g += mat_elem(wg, n, i, d) * vi;
            u += mat_elem(wu, n, i, d) * vi;
        }
        double silu = g / (1.0 + exp(-g));
        h[n] = silu * u;
    }
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int n = 0; n < I; ++n) acc += mat_elem(wd, o, n, I) * h[n];
        out[o] += weight * acc;
    }
}

/* Offsets the pointers of a stacked [E, rows, cols] weight to expert e. */
static oracle_mat_t expert_slice(const oracle_mat_t* m, int64_t e, int64_t rows, int64_t cols) {
    oracle_mat_t s = *m;
    if (m->bits == 16) {
        s.w16 = m->w16 + e * rows * cols;
    } else {
        s.q = m->q + e * rows * (cols / (32 / m->bits));
        s.scale = m->scale + e * rows * (cols / m->group);
        s.bias = m->bias + e * rows * (cols / m->group);
    }
    return s;
}

/*
 * The layer as a dense per-token loop ([arch]):
 *   y[t] = sum_k scores[t, k] * FFN_{inds[t, k]}(x[t]) + FFN_shared(x[t]).
 * Experts are stacked: gate/up [E, I, d], down [E, d, I].  The shared expert (one FFN of
 * the same shape, always active, weight 1, no gate) is skipped when has_shared == 0; with
 * shared_gate (bf16 [d]) non-NULL its output is scaled by sigmoid(x . shared_gate) instead
 * (the gated shared expert of the combine's has_shared_expert_gate = true).
 * `rows` lists which tokens to evaluate (n_rows of them); y is [n_rows, d] fp32.
 */
int oracle_moe_layer_rows(const uint16_t* x, int64_t T, int d, int I, int E, int K,
                          const int32_t* inds, const float* scores, int bits, int group,
                          const void* gate_w, const void* gate_s, const void* gate_b,
                          const void* up_w, const void* up_s, const void* up_b,
                          const void* down_w, const void* down_s, const void* down_b,
                          int has_shared,
                          const void* sgate_w, const void* sgate_s, const void* sgate_b,
                          const void* sup_w, const void* sup_s, const void* sup_b,
                          const void* sdown_w, const void* sdown_s, const void* sdown_b,
                          const void* shared_gate,
                          const int64_t* rows, int64_t n_rows, float* y) {
    (void)T;
    if (bits != 16 && bits != 4 && bits != 8) return -1;
    if (bits != 16 && (group < 1 || d % group || I % group)) return -1;
    oracle_mat_t g = {bits, group, (const uint16_t*)gate_w, (const uint32_t*)gate_w,
                      (const uint16_t*)gate_s, (const uint16_t*)gate_b};
    oracle_mat_t u = {bits, group, (const uint16_t*)up_w, (const uint32_t*)up_w,
                      (const uint16_t*)up_s, (const uint16_t*)up_b};
    oracle_mat_t dn = {bits, group, (const uint16_t*)down_w, (const uint32_t*)down_w,
                       (const uint16_t*)down_s, (const uint16_t*)down_b};
    /* the shared expert is always bf16 (the quantised checkpoint keeps it in bf16) */
    oracle_mat_t sg = {16, group, (const uint16_t*)sgate_w, 0, 0, 0};
    oracle_mat_t su = {16, group, (const uint16_t*)sup_w, 0, 0, 0};
    oracle_mat_t sd = {16, group, (const uint16_t*)sdown_w, 0, 0, 0};
    (void)sgate_s; (void)sgate_b; (void)sup_s; (void)sup_b; (void)sdown_s; (void)sdown_b;
    int rc = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : rc)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t t = rows[ri];
        double* acc = (double*)calloc((size_t)d, sizeof(double));
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        if (!acc || !h) { rc |= 1; free(acc); free(h); continue; }
        const uint16_t* v = x + t * d;
        for (int k = 0; k < K; ++k) {
            int e = inds[t * K + k];
            if (e < 0 || e >= E) { rc |= 1; continue; }
            oracle_mat_t ge = expert_slice(&g, e, I, d);
            oracle_mat_t ue = expert_slice(&u, e, I, d);
            oracle_mat_t de = expert_slice(&dn, e, d, I);
            expert_ffn(v, d, I, &ge, &ue, &de, (double)scores[t * K + k], acc, h);
        }
        if (has_shared) {
            /* gated shared expert (the combine's has_shared_expert_gate): the shared output
             * is scaled by sigmoid(x . w_gate_vec); weight 1 without a gate */
            double gw = 1.0;
            if (shared_gate) {
                double z = 0.0;
                for (int i = 0; i < d; ++i)
                    z += (double)oracle_bf16_to_f32(v[i]) *
                         (double)oracle_bf16_to_f32(((const uint16_t*)shared_gate)[i]);
                gw = 1.0 / (1.0 + exp(-z));
            }
            expert_ffn(v, d, I, &sg, &su, &sd, gw, acc, h);
        }
        for (int o = 0; o < d; ++o) y[ri * d + o] = (float)acc[o];
        free(acc);
        free(h);
    }
    return rc ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* DSA indexer top-k selection                                                          */
/* ------------------------------------------------------------------------------------ */
/*
 * [dsa] SwiftLM issue #139 (stage 2 of the DeepSeek-V3.2 / GLM sparse-attention port),
 * "What needs building" item 1: the indexer's selection is argPartition(scores,
 * kth: -index_topk), i.e. the index_topk largest scores of each query row; item 3: decode
 * gathers the selected key positions, prefill turns them into a boolean mask ANDed with the
 * causal mask; and the inertness remark: while a row has no more than index_topk positions
 * the selection is every position (dense attention).
 *
 * Readings where the page is silent: a row r has n_r valid positions j < n_r (n_r from
 * `lengths`, the causal length, or n); the selection is the min(k, n_r) largest valid scores
 * in the order "larger score first, equal scores by lower position" (NaN lowest, -0 == +0),
 * returned as positions in ascending order and padded with -1 up to k; the optional mask
 * row is 1 exactly at the selected positions.
 */
typedef struct {
    float v;
    int32_t j;
} oracle_scored_t;

static int scored_cmp(const void* pa, const void* pb) {
    const oracle_scored_t* a = (const oracle_scored_t*)pa;
    const oracle_scored_t* b = (const oracle_scored_t*)pb;
    if (route_better(a->v, a->j, b->v, b->j)) return -1;
    if (route_better(b->v, b->j, a->v, a->j)) return 1;
    return 0;
}

static int int_cmp(const void* pa, const void* pb) {
    const int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

int oracle_indexer_topk(const float* scores, int64_t rows, int32_t n, int64_t ld,
                        const int32_t* lengths, int32_t k, int32_t* inds, uint8_t* mask,
                        int64_t mask_ld) {
    if (rows < 0 || n < 0 || k < 1 || ld < n || (rows > 0 && (!scores || !inds)) ||
        (mask && mask_ld < n))
        return -1;
    int rc = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : rc)
    for (int64_t r = 0; r < rows; ++r) {
        int32_t nr = lengths ? lengths[r] : n;
        if (nr < 0) nr = 0;
        if (nr > n) nr = n;
        oracle_scored_t* it = (oracle_scored_t*)malloc(sizeof(oracle_scored_t) * (size_t)(nr + 1));
        int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k + 1));
        if (!it || !sel) {
            free(it);
            free(sel);
            rc |= 1;
            continue;
        }
        for (int32_t j = 0; j < nr; ++j) {
            it[j].v = scores[r * ld + j];
            it[j].j = j;
        }
        qsort(it, (size_t)nr, sizeof(oracle_scored_t), scored_cmp);
        const int32_t m = nr < k ? nr : k;
        for (int32_t i = 0; i < m; ++i) sel[i] = it[i].j;
        qsort(sel, (size_t)m, sizeof(int32_t), int_cmp);
        for (int32_t i = 0; i < k; ++i) inds[r * k + i] = i < m ? sel[i] : -1;
        if (mask) {
            uint8_t* mr = mask + r * mask_ld;
            for (int32_t j = 0; j < n; ++j) mr[j] = 0;
            for (int32_t i = 0; i < m; ++i) mr[sel[i]] = 1;
        }
        free(it);
        free(sel);
    }
    return rc ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
