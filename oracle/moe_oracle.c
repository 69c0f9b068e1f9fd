/*
 * moe_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow, obviously correct CPU statement of the forward pass of one top-k routed
 * mixture-of-experts FFN layer, and of its backward pass, in double precision. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the CUDA library never links, calls or includes it,
 * and it shares no code, header or table with the CUDA library.
 *
 * Sources (web pages on mixture of experts), cited by page and section:
 *   [CURIO]   llm.curionode.com "Mixture of Experts." (Plate 4), opening text and "Workshop":
 *             the layer replaces the MLP with E MLPs plus a router, a linear layer and a softmax;
 *             the top K experts run and their outputs are added, weighted by the normalised scores.
 *   [LENSA-1] lensaml.com "Mixture of Experts", Step 1 of 6 "Bigger Model, Same Compute".
 *   [LENSA-2] same page, Step 2 of 6 "The Router": logits = h . W_r, then a softmax over experts.
 *   [LENSA-3] same page, Step 3 of 6 "Top-k Routing": the gates are a softmax over the chosen
 *             logits (Mixtral: y = sum softmax(TopK(h . W_g))_i E_i(h)); Switch top-1 scales the
 *             output by the raw router probability p_i instead; y = sum g . E(h).
 *   [LENSA-4] same page, Step 4 of 6 "Load Balancing": the auxiliary term N . sum_i f_i P_i,
 *             f_i the fraction of tokens sent to expert i, P_i its mean router probability;
 *             it equals 1 under uniform routing.
 *   [LENSA-5] same page, Step 5 of 6 "Capacity & Dropped Tokens" (dropless grouping, MegaBlocks).
 *   [LENSA-6] same page, Step 6 of 6 "MoE in Practice" (Mixtral expert = 3 x 4096 x 14336).
 *   [JAGGI]   arjunjaggi.com "Mixture of Experts in LLMs: How Sparse Models Scale", sections
 *             "The Router" (Switch k = 1) and "Switch Transformers" (router kept in float32); its
 *             training section names the router z-loss of ST-MoE (Zoph et al., arXiv:2202.08906)
 *             as a penalty on large router logits.
 *   [LENSA-4] also: DeepSeek-V3 replaces the auxiliary loss by a per-expert routing bias that is
 *             nudged up or down. The pages give neither formula; both are taken from the cited
 *             papers (ST-MoE, router z-loss; DeepSeek-V3 Technical Report, auxiliary-loss-free
 *             load balancing), as read below.
 *
 * Readings where the pages leave a step open (each is also listed with the design notes):
 *   - f_i = count_i / (T k), so that sum_i f_i = 1 and the auxiliary term is exactly 1 under
 *     uniform routing for any k; P_i is the mean of the FULL softmax (before top-k).
 *   - The auxiliary value returned is E . sum f P; the weight alpha is the caller's.
 *   - Top-k order: logits descending, equal logits broken toward the lower expert index.
 *   - Renormalised gates are the softmax over the chosen logits (equal to p_j / sum_S p).
 *   - Activation "GELU" is the tanh form 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))).
 *   - SwiGLU expert: W2 (SiLU(W1 x) * (W3 x)), no biases; SiLU(x) = x / (1 + e^-x).
 *   - Grouping order: a stable counting sort of the flattened slots s = t k + j by expert,
 *     i.e. (expert ascending, token ascending); nothing is dropped unless a capacity is given.
 *   - Capacity ([LENSA-5]): C = floor(factor T k / E); an expert keeps the first C of its slots
 *     in that order; a dropped slot contributes nothing and the kept gates are not renormalised;
 *     the auxiliary value uses the routed (pre-drop) counts.
 *   - Router z-loss (ST-MoE): (1/T) sum_t (log sum_e exp z[t,e])^2 over the router logits z
 *     (router bias included); its weight is the caller's.
 *   - Selection-only routing bias (DeepSeek-V3): the k experts are chosen by the keys
 *     p[t,e] + b[e] (p the full softmax of this router, the affinity its gates use), descending,
 *     ties to the lower index; the gates, p and the auxiliary value stay those of the unbiased
 *     router. After a step, b[e] moves by +gamma when expert e received fewer routing slots than
 *     the mean T k / E, by -gamma when more, and not at all when equal.
 *
 * Precision: inputs are read exactly as stored (f32, or bf16 widened bit-exactly) and every sum,
 * product and transcendental is taken in double, in index order, with no intermediate rounding.
 *
 * Every forward function below is pinned by tests/test_oracle_pins.py against the pages' printed
 * values, closed forms, brute force or an independent library computation; the backward by
 * tests/test_oracle_backward_pins.py against finite differences of these forward functions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_GELU_TANH 0
#define OR_SWIGLU 1
#define OR_RENORM 0
#define OR_RAW_PROB 1

/* Read element i of a tensor stored as f32 or as raw bf16 bits, widened exactly to double. */
static double widen(const void *p, int dtype, int64_t i)
{
    if (dtype == OR_F32) return (double)((const float *)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float v;
    memcpy(&v, &bits, sizeof v);
    return (double)v;
}

/* [LENSA-2], [CURIO], [JAGGI]: logits z[t,e] = sum_i h[t,i] W_r[i,e] (+ b_r[e]); p = softmax_e(z),
 * evaluated with the maximum subtracted (an identity of the softmax). W_r is [d, E] row-major. */
void oracle_router(int64_t T, int32_t d, int32_t E, const void *h, int32_t h_dtype,
                   const float *W_r, const float *b_r, double *z, double *p)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double zmax = -INFINITY;
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t i = 0; i < d; ++i)
                acc += widen(h, h_dtype, t * d + i) * (double)W_r[(int64_t)i * E + e];
            if (b_r) acc += (double)b_r[e];
            z[t * E + e] = acc;
            if (acc > zmax) zmax = acc;
        }
        double s = 0.0;
        for (int32_t e = 0; e < E; ++e) s += exp(z[t * E + e] - zmax);
        for (int32_t e = 0; e < E; ++e) p[t * E + e] = exp(z[t * E + e] - zmax) / s;
    }
}

/* [LENSA-3], [CURIO] "Top-K routing": the k experts with the largest logits, listed in descending
 * order, equal logits toward the lower index. Also records, per token, the gap between the k-th
 * and (k+1)-th logit (boundary; +inf when k == E) and the smallest gap between consecutive chosen
 * logits (inset; +inf when k == 1): where those are tiny, another precision may choose otherwise. */
void oracle_topk(int64_t T, int32_t E, int32_t k, const double *z, int32_t *idx,
                 double *boundary_margin, double *inset_margin)
{
#pragma omp parallel
    {
        unsigned char *chosen = (unsigned char *)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const double *zt = z + t * E;
            memset(chosen, 0, (size_t)E);
            double inset = INFINITY, prev = 0.0;
            for (int32_t j = 0; j < k; ++j) {
                int32_t best = -1;
                for (int32_t e = 0; e < E; ++e)
                    if (!chosen[e] && (best < 0 || zt[e] > zt[best])) best = e;
                chosen[best] = 1;
                idx[t * k + j] = best;
                if (j > 0 && prev - zt[best] < inset) inset = prev - zt[best];
                prev = zt[best];
            }
            double boundary = INFINITY;
            if (k < E) {
                int32_t nxt = -1;
                for (int32_t e = 0; e < E; ++e)
                    if (!chosen[e] && (nxt < 0 || zt[e] > zt[nxt])) nxt = e;
                boundary = prev - zt[nxt];
            }
            if (boundary_margin) boundary_margin[t] = boundary;
            if (inset_margin) inset_margin[t] = inset;
        }
        free(chosen);
    }
}

/* [LENSA-3]: gate weights of the chosen experts.
 *   mode RENORM   : g_j = softmax over the chosen logits = exp(z_j - z_1) / sum_{i in S} exp(z_i - z_1)
 *                   (the Mixtral form softmax(TopK(h . W_g)); it sums to 1 over the chosen set)
 *   mode RAW_PROB : g_j = p_j, the full-softmax probability (the Switch top-1 form) */
void oracle_gates(int64_t T, int32_t E, int32_t k, int32_t mode, const double *z, const double *p,
                  const int32_t *idx, double *g)
{
    for (int64_t t = 0; t < T; ++t) {
        const int32_t *it = idx + t * k;
        if (mode == OR_RAW_PROB) {
            for (int32_t j = 0; j < k; ++j) g[t * k + j] = p[t * E + it[j]];
        } else {
            double zmax = z[t * E + it[0]];
            double s = 0.0;
            for (int32_t j = 0; j < k; ++j) s += exp(z[t * E + it[j]] - zmax);
            for (int32_t j = 0; j < k; ++j) g[t * k + j] = exp(z[t * E + it[j]] - zmax) / s;
        }
    }
}

/* [LENSA-4] (DeepSeek-V3's routing bias, reading above): the selection keys p[t,e] + b[e]; the
 * top-k of these keys (oracle_topk) is the biased choice. */
void oracle_selection_keys(int64_t T, int32_t E, const double *p, const double *b, double *key)
{
    for (int64_t t = 0; t < T; ++t)
        for (int32_t e = 0; e < E; ++e) key[t * E + e] = p[t * E + e] + b[e];
}

/* [LENSA-4] (reading above): b_out[e] = b_in[e] + gamma * sign(T k / E - counts[e]). */
void oracle_update_sel_bias(int64_t T, int32_t E, int32_t k, const int32_t *counts, double gamma,
                            const double *b_in, double *b_out)
{
    const double mean = (double)T * (double)k / (double)E;
    for (int32_t e = 0; e < E; ++e) {
        const double c = (double)counts[e];
        b_out[e] = b_in[e] + (c < mean ? gamma : (c > mean ? -gamma : 0.0));
    }
}

/* [JAGGI] (ST-MoE's router z-loss, reading above): (1/T) sum_t (log sum_e exp z[t,e])^2, the
 * log-sum-exp taken as zmax + log sum_e exp(z - zmax). 0 for T = 0. */
double oracle_zloss(int64_t T, int32_t E, const double *z)
{
    double acc = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const double *zt = z + t * E;
        double zmax = zt[0];
        for (int32_t e = 1; e < E; ++e)
            if (zt[e] > zmax) zmax = zt[e];
        double s = 0.0;
        for (int32_t e = 0; e < E; ++e) s += exp(zt[e] - zmax);
        const double lse = zmax + log(s);
        acc += lse * lse;
    }
    return T > 0 ? acc / (double)T : 0.0;
}

/* [LENSA-4] histogram of routing slots per expert, [LENSA-5] dropless grouping: a stable counting
 * sort of the flattened slots s = t*k + j by expert idx[s].
 *   counts[e]        slots routed to e
 *   offsets[0..E]    exclusive prefix sum of counts (offsets[E] = T k)
 *   sorted_token[r]  token of the r-th slot in (expert, token) order
 *   slot_of[s]       sorted position of slot s (the inverse map) */
void oracle_dispatch(int64_t T, int32_t E, int32_t k, const int32_t *idx, int32_t *counts,
                     int32_t *offsets, int32_t *sorted_token, int32_t *slot_of)
{
    const int64_t P = T * k;
    int64_t *cursor = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t s = 0; s < P; ++s) counts[idx[s]] += 1;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int32_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t s = 0; s < P; ++s) {
        int64_t pos = cursor[idx[s]]++;
        sorted_token[pos] = (int32_t)(s / k);
        slot_of[s] = (int32_t)pos;
    }
    free(cursor);
}

/* [LENSA-5] capacity: every expert gets a buffer of C = factor x T x k / E slots; routing slots
 * beyond it are skipped by the expert. Reading: C is rounded down, and within an expert the first
 * C slots in stable token order are kept (the grouping order of oracle_dispatch).
 *   counts[e]   slots routed to e (the demand, before dropping)
 *   offsets     exclusive prefix sum of min(counts[e], C); offsets[E] = slots kept
 *   sorted_token / slot_of as in oracle_dispatch for kept slots; slot_of[s] = -1 when dropped.
 * C < 0 means no capacity limit (the dropless dispatch). */
int64_t oracle_capacity(double factor, int64_t T, int32_t k, int32_t E)
{
    return (int64_t)floor(factor * (double)T * (double)k / (double)E);
}

void oracle_dispatch_capacity(int64_t T, int32_t E, int32_t k, const int32_t *idx, int64_t C,
                              int32_t *counts, int32_t *offsets, int32_t *sorted_token,
                              int32_t *slot_of)
{
    const int64_t P = T * k;
    int64_t *rank = (int64_t *)calloc((size_t)(E > 0 ? E : 1), sizeof(int64_t));
    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t s = 0; s < P; ++s) counts[idx[s]] += 1;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) {
        const int64_t kept = (C >= 0 && counts[e] > C) ? C : counts[e];
        offsets[e + 1] = offsets[e] + (int32_t)kept;
    }
    for (int64_t s = 0; s < P; ++s) {
        const int32_t e = idx[s];
        const int64_t r = rank[e]++;
        if (C >= 0 && r >= C) {
            slot_of[s] = -1;
        } else {
            const int64_t pos = offsets[e] + r;
            sorted_token[pos] = (int32_t)(s / k);
            slot_of[s] = (int32_t)pos;
        }
    }
    free(rank);
}

/* GELU in its tanh form and SiLU, in double. */
static double gelu_tanh(double x)
{
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

double oracle_gelu_tanh(double x) { return gelu_tanh(x); }
double oracle_silu(double x) { return silu(x); }

/* [CURIO] "Workshop" (experts are MLPs of width f), [LENSA-1]/[LENSA-6] (a full expert is three
 * d x f matrices): expert e applied to one input row x of length d.
 *   GELU form   : y = W2_e GELU(W1_e x + b1_e) + b2_e
 *   SwiGLU form : y = W2_e (SiLU(W1_e x) * (W3_e x))
 * W1, W3 are [E, f, d] and W2 is [E, d, f], row-major (output index, then input index). */
static void expert_mlp(int32_t d, int32_t f, int32_t act, const double *x, int32_t e,
                       const void *W1, const void *W3, const void *W2, int32_t w_dtype,
                       const float *b1, const float *b2, double *hid, double *y)
{
    const int64_t base1 = (int64_t)e * f * d;
    const int64_t base2 = (int64_t)e * d * f;
    for (int32_t j = 0; j < f; ++j) {
        double a = 0.0;
        for (int32_t i = 0; i < d; ++i) a += widen(W1, w_dtype, base1 + (int64_t)j * d + i) * x[i];
        if (act == OR_SWIGLU) {
            double c = 0.0;
            for (int32_t i = 0; i < d; ++i)
                c += widen(W3, w_dtype, base1 + (int64_t)j * d + i) * x[i];
            hid[j] = silu(a) * c;
        } else {
            if (b1) a += (double)b1[(int64_t)e * f + j];
            hid[j] = gelu_tanh(a);
        }
    }
    for (int32_t o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int32_t j = 0; j < f; ++j) acc += widen(W2, w_dtype, base2 + (int64_t)o * f + j) * hid[j];
        if (act != OR_SWIGLU && b2) acc += (double)b2[(int64_t)e * d + o];
        y[o] = acc;
    }
}

/* Expert MLPs on n independent rows: y[r] = FFN_{expert[r]}(x[r]); x and y are [n, d] double. */
void oracle_expert_ffn(int64_t n, int32_t d, int32_t f, int32_t act, const double *x,
                       const int32_t *expert, const void *W1, const void *W3, const void *W2,
                       int32_t w_dtype, const float *b1, const float *b2, double *y)
{
#pragma omp parallel
    {
        double *hid = (double *)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r)
            expert_mlp(d, f, act, x + r * d, expert[r], W1, W3, W2, w_dtype, b1, b2, hid, y + r * d);
        free(hid);
    }
}

/* [LENSA-3] "y = sum g . E(h)", [CURIO]: the chosen experts' outputs added, weighted by the gates,
 * in slot order j = 0..k-1. yslot is [n, k, d] (expert output of slot j of token t), g is [n, k]. */
void oracle_combine(int64_t n, int32_t k, int32_t d, const double *g, const double *yslot,
                    double *y)
{
    for (int64_t t = 0; t < n; ++t)
        for (int32_t o = 0; o < d; ++o) {
            double acc = 0.0;
            for (int32_t j = 0; j < k; ++j) acc += g[t * k + j] * yslot[(t * k + j) * d + o];
            y[t * d + o] = acc;
        }
}

/* The layer output of the listed tokens: y[r] = sum_j g[t,j] FFN_{idx[t,j]}(h[t]) with t = tokens[r].
 * Each output row depends only on its own token, so any subset of tokens can be evaluated.
 * keep (may be NULL) marks the routing slots t*k+j that an expert processes; a slot that is not
 * kept (dropped by the capacity limit, [LENSA-5]) contributes nothing. */
void oracle_forward_rows_kept(int64_t n, const int64_t *tokens, int32_t d, int32_t f, int32_t k,
                              int32_t act, const void *h, int32_t h_dtype, const int32_t *idx,
                              const double *g, const void *W1, const void *W3, const void *W2,
                              int32_t w_dtype, const float *b1, const float *b2,
                              const unsigned char *keep, double *y)
{
    const int64_t nk = n * k;
    double *x = (double *)malloc(sizeof(double) * (size_t)(nk * d + 1));
    double *ys = (double *)malloc(sizeof(double) * (size_t)(nk * d + 1));
    double *gs = (double *)malloc(sizeof(double) * (size_t)(nk + 1));
    int32_t *ex = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nk + 1));
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens[r];
        for (int32_t j = 0; j < k; ++j) {
            for (int32_t i = 0; i < d; ++i) x[(r * k + j) * d + i] = widen(h, h_dtype, t * d + i);
            ex[r * k + j] = idx[t * k + j];
            gs[r * k + j] = (keep && !keep[t * k + j]) ? 0.0 : g[t * k + j];
        }
    }
    oracle_expert_ffn(nk, d, f, act, x, ex, W1, W3, W2, w_dtype, b1, b2, ys);
    oracle_combine(n, k, d, gs, ys, y);
    free(x); free(ys); free(gs); free(ex);
}

void oracle_forward_rows(int64_t n, const int64_t *tokens, int32_t d, int32_t f, int32_t k,
                         int32_t act, const void *h, int32_t h_dtype, const int32_t *idx,
                         const double *g, const void *W1, const void *W3, const void *W2,
                         int32_t w_dtype, const float *b1, const float *b2, double *y)
{
    oracle_forward_rows_kept(n, tokens, d, f, k, act, h, h_dtype, idx, g, W1, W3, W2, w_dtype, b1,
                             b2, NULL, y);
}

/* [LENSA-4]: E . sum_e f_e P_e with f_e = counts[e] / (T k) and P_e = (1/T) sum_t p[t,e]
 * (the full softmax). The weight alpha is not applied. */
double oracle_aux_loss(int64_t T, int32_t E, int32_t k, const int32_t *counts, const double *p)
{
    double acc = 0.0;
    for (int32_t e = 0; e < E; ++e) {
        double Pe = 0.0;
        for (int64_t t = 0; t < T; ++t) Pe += p[t * E + e];
        Pe /= (double)T;
        const double fe = (double)counts[e] / ((double)T * (double)k);
        acc += fe * Pe;
    }
    return (double)E * acc;
}

/* [CURIO] "Parameters you hold, parameters you use", [LENSA-1], [LENSA-6]: total and active
 * parameter counts of a model whose FFN blocks are replaced by E experts of mats x d x f weights
 * each, k of them active per token. Everything else (attention, norms, embeddings) is shared:
 * shared_per_layer is counted once per layer, shared_global once per model. The router (d x E per
 * layer) is counted as shared when with_router is set. */
void oracle_param_count(int32_t n_layers, int64_t d, int64_t f, int32_t E, int32_t k,
                        int32_t mats, int64_t shared_per_layer, int64_t shared_global,
                        int32_t with_router, int64_t *total, int64_t *active)
{
    const int64_t expert = (int64_t)mats * d * f;
    const int64_t router = with_router ? d * E : 0;
    *total = (int64_t)n_layers * (shared_per_layer + router + (int64_t)E * expert) + shared_global;
    *active = (int64_t)n_layers * (shared_per_layer + router + (int64_t)k * expert) + shared_global;
}

/* ---------------------------------------------------------------------------------------------
 * Backward pass. [CURIO] opening text and [LENSA-3]: selecting the top-k experts is not
 * differentiable, so the gradient reaches the router only through the weights of the chosen
 * experts (for Switch top-1, through p_i); [LENSA-4]: of the auxiliary term only P_i is
 * differentiable; [JAGGI] "How Routing Works": the router trains by ordinary backpropagation.
 * Reading: idx, the routed counts (hence f_i) and the capacity drops are constants of the step;
 * everything else is differentiated exactly by the chain rule, in double.
 *
 * The loss whose gradient is returned is
 *     L = sum_{t,o} dy[t,o] y[t,o] + aux_weight * (E sum_e f_e P_e) + zloss_weight * zloss,
 * so dy is the upstream gradient of y. */

/* d/dx of the tanh-form GELU: with u = c (x + 0.044715 x^3), c = sqrt(2/pi),
 * 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) c (1 + 3 * 0.044715 x^2). */
static double gelu_tanh_grad(double x)
{
    const double c = sqrt(2.0 / M_PI);
    const double th = tanh(c * (x + 0.044715 * x * x * x));
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * c * (1.0 + 3.0 * 0.044715 * x * x);
}

/* d/dx of SiLU: s (1 + x (1 - s)) with s = 1 / (1 + e^-x). */
static double silu_grad(double x)
{
    const double s = 1.0 / (1.0 + exp(-x));
    return s * (1.0 + x * (1.0 - s));
}

double oracle_gelu_tanh_grad(double x) { return gelu_tanh_grad(x); }
double oracle_silu_grad(double x) { return silu_grad(x); }

/* Gradient of L with respect to the router logits of one token, given dg[j] = dL/dg_j of its k
 * gates (0 for a dropped slot):
 *   RENORM  : g = softmax over the chosen logits, so dz[e_j] = g_j (dg_j - sum_l g_l dg_l) and
 *             dz = 0 off the chosen set;
 *   RAW_PROB: g_j = p[e_j], so dz[i] = sum_j dg_j p[e_j] (delta(i, e_j) - p[i]);
 *   plus the auxiliary term: dL/dp[t,e] = aux_weight E f_e / T =: c_e, through the softmax
 *   dz[i] += p[i] (c_i - sum_e c_e p[e]);
 *   plus the z-loss: d/dz[i] of zloss_weight (1/T) lse^2 is zloss_weight (2/T) lse p[i]. */
static void router_logit_grad(int64_t T, int32_t E, int32_t k, int32_t gate_mode,
                              const double *zt, const double *pt, const int32_t *it,
                              const double *gt, const double *dg, const double *fe,
                              double aux_weight, double zloss_weight, double *dz)
{
    for (int32_t e = 0; e < E; ++e) dz[e] = 0.0;
    if (gate_mode == OR_RAW_PROB) {
        double s = 0.0;
        for (int32_t j = 0; j < k; ++j) s += dg[j] * pt[it[j]];
        for (int32_t e = 0; e < E; ++e) dz[e] = -pt[e] * s;
        for (int32_t j = 0; j < k; ++j) dz[it[j]] += dg[j] * pt[it[j]];
    } else {
        double s = 0.0;
        for (int32_t j = 0; j < k; ++j) s += gt[j] * dg[j];
        for (int32_t j = 0; j < k; ++j) dz[it[j]] += gt[j] * (dg[j] - s);
    }
    if (aux_weight != 0.0) {
        double s = 0.0;
        for (int32_t e = 0; e < E; ++e) s += aux_weight * (double)E * fe[e] / (double)T * pt[e];
        for (int32_t e = 0; e < E; ++e)
            dz[e] += pt[e] * (aux_weight * (double)E * fe[e] / (double)T - s);
    }
    if (zloss_weight != 0.0) {
        double zmax = zt[0];
        for (int32_t e = 1; e < E; ++e)
            if (zt[e] > zmax) zmax = zt[e];
        double s = 0.0;
        for (int32_t e = 0; e < E; ++e) s += exp(zt[e] - zmax);
        const double lse = zmax + log(s);
        for (int32_t e = 0; e < E; ++e) dz[e] += zloss_weight * 2.0 / (double)T * lse * pt[e];
    }
}

/* The whole backward of the layer for the routing idx [T, k] (keep [T, k] may be NULL: every
 * slot is processed). Outputs, all overwritten (NULL where the layer has no such parameter):
 *   dh [T, d], dW_r [d, E], db_r [E], dW1 and dW3 [E, f, d], dW2 [E, d, f], db1 [E, f],
 *   db2 [E, d]; dg_out [T, k] (may be NULL): dL/dg of every slot.
 * Expert e's weight gradients are sums over its slots in token order; dh[t] adds the k slots'
 * input gradients in slot order and then the router's h-gradient. */
void oracle_backward(int64_t T, int32_t d, int32_t f, int32_t E, int32_t k, int32_t act,
                     int32_t gate_mode, const void *h, int32_t h_dtype, const float *W_r,
                     const float *b_r, const void *W1, const void *W3, const void *W2,
                     int32_t w_dtype, const float *b1, const float *b2, const int32_t *idx,
                     const unsigned char *keep, const void *dy, int32_t dy_dtype,
                     double aux_weight, double zloss_weight, double *dh, double *dW_r,
                     double *db_r, double *dW1, double *dW3, double *dW2, double *db1,
                     double *db2, double *dg_out)
{
    const int64_t P = T * k;
    double *z = (double *)malloc(sizeof(double) * (size_t)(T * E + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(T * E + 1));
    double *g = (double *)malloc(sizeof(double) * (size_t)(P + 1));
    double *dg = (double *)calloc((size_t)(P + 1), sizeof(double));
    double *dxs = (double *)calloc((size_t)(P * d + 1), sizeof(double));
    double *fe = (double *)calloc((size_t)(E > 0 ? E : 1), sizeof(double));
    oracle_router(T, d, E, h, h_dtype, W_r, b_r, z, p);
    oracle_gates(T, E, k, gate_mode, z, p, idx, g);
    for (int64_t s = 0; s < P; ++s) fe[idx[s]] += 1.0;
    for (int32_t e = 0; e < E; ++e) fe[e] /= (double)T * (double)k;

    const int64_t wsz = (int64_t)E * f * d;
    for (int64_t i = 0; i < wsz; ++i) {
        dW1[i] = 0.0;
        dW2[i] = 0.0;
        if (dW3) dW3[i] = 0.0;
    }
    if (db1) for (int64_t i = 0; i < (int64_t)E * f; ++i) db1[i] = 0.0;
    if (db2) for (int64_t i = 0; i < (int64_t)E * d; ++i) db2[i] = 0.0;

    /* experts: each one owns its weight gradients; slots of expert e in token order */
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)d);
        double *dyt = (double *)malloc(sizeof(double) * (size_t)d);
        double *a1 = (double *)malloc(sizeof(double) * (size_t)f);
        double *a3 = (double *)malloc(sizeof(double) * (size_t)f);
        double *hid = (double *)malloc(sizeof(double) * (size_t)f);
        double *dhid = (double *)malloc(sizeof(double) * (size_t)f);
        double *da1 = (double *)malloc(sizeof(double) * (size_t)f);
        double *da3 = (double *)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int32_t e = 0; e < E; ++e) {
            const int64_t base1 = (int64_t)e * f * d, base2 = (int64_t)e * d * f;
            for (int64_t s = 0; s < P; ++s) {
                if (idx[s] != e || (keep && !keep[s])) continue;
                const int64_t t = s / k;
                for (int32_t i = 0; i < d; ++i) {
                    x[i] = widen(h, h_dtype, t * d + i);
                    dyt[i] = widen(dy, dy_dtype, t * d + i);
                }
                /* forward of this slot: pre-activations, hidden row and output */
                for (int32_t n = 0; n < f; ++n) {
                    double u = 0.0, v = 0.0;
                    for (int32_t i = 0; i < d; ++i) {
                        u += widen(W1, w_dtype, base1 + (int64_t)n * d + i) * x[i];
                        if (act == OR_SWIGLU) v += widen(W3, w_dtype, base1 + (int64_t)n * d + i) * x[i];
                    }
                    if (act != OR_SWIGLU && b1) u += (double)b1[(int64_t)e * f + n];
                    a1[n] = u;
                    a3[n] = v;
                    hid[n] = act == OR_SWIGLU ? silu(u) * v : gelu_tanh(u);
                }
                /* dL/dg of this slot: dy[t] . (W2_e hid + b2_e) */
                double dgs = 0.0;
                for (int32_t o = 0; o < d; ++o) {
                    double yo = 0.0;
                    for (int32_t n = 0; n < f; ++n) yo += widen(W2, w_dtype, base2 + (int64_t)o * f + n) * hid[n];
                    if (act != OR_SWIGLU && b2) yo += (double)b2[(int64_t)e * d + o];
                    dgs += dyt[o] * yo;
                }
                dg[s] = dgs;
                /* the slot's output enters y scaled by its gate */
                const double gs = g[s];
                for (int32_t n = 0; n < f; ++n) dhid[n] = 0.0;
                for (int32_t o = 0; o < d; ++o) {
                    const double dyo = gs * dyt[o];
                    for (int32_t n = 0; n < f; ++n) {
                        dW2[base2 + (int64_t)o * f + n] += dyo * hid[n];
                        dhid[n] += widen(W2, w_dtype, base2 + (int64_t)o * f + n) * dyo;
                    }
                    if (act != OR_SWIGLU && db2) db2[(int64_t)e * d + o] += dyo;
                }
                for (int32_t n = 0; n < f; ++n) {
                    if (act == OR_SWIGLU) {
                        da1[n] = dhid[n] * a3[n] * silu_grad(a1[n]);
                        da3[n] = dhid[n] * silu(a1[n]);
                    } else {
                        da1[n] = dhid[n] * gelu_tanh_grad(a1[n]);
                        da3[n] = 0.0;
                    }
                }
                double *dx = dxs + s * d;
                for (int32_t n = 0; n < f; ++n) {
                    for (int32_t i = 0; i < d; ++i) {
                        dW1[base1 + (int64_t)n * d + i] += da1[n] * x[i];
                        dx[i] += widen(W1, w_dtype, base1 + (int64_t)n * d + i) * da1[n];
                        if (act == OR_SWIGLU) {
                            dW3[base1 + (int64_t)n * d + i] += da3[n] * x[i];
                            dx[i] += widen(W3, w_dtype, base1 + (int64_t)n * d + i) * da3[n];
                        }
                    }
                    if (act != OR_SWIGLU && db1) db1[(int64_t)e * f + n] += da1[n];
                }
            }
        }
        free(x); free(dyt); free(a1); free(a3); free(hid); free(dhid); free(da1); free(da3);
    }

    /* router: dz per token, then dh, dW_r and db_r */
    double *dz = (double *)malloc(sizeof(double) * (size_t)(T * E + 1));
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        router_logit_grad(T, E, k, gate_mode, z + t * E, p + t * E, idx + t * k, g + t * k,
                          dg + t * k, fe, aux_weight, zloss_weight, dz + t * E);
        for (int32_t i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int32_t j = 0; j < k; ++j) acc += dxs[(t * k + j) * d + i];
            for (int32_t e = 0; e < E; ++e) acc += (double)W_r[(int64_t)i * E + e] * dz[t * E + e];
            dh[t * d + i] = acc;
        }
    }
    for (int64_t i = 0; i < (int64_t)d * E; ++i) dW_r[i] = 0.0;
    if (db_r) for (int32_t e = 0; e < E; ++e) db_r[e] = 0.0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t e = 0; e < E; ++e) {
            for (int32_t i = 0; i < d; ++i) dW_r[(int64_t)i * E + e] += widen(h, h_dtype, t * d + i) * dz[t * E + e];
            if (db_r) db_r[e] += dz[t * E + e];
        }
    if (dg_out) for (int64_t s = 0; s < P; ++s) dg_out[s] = dg[s];
    free(z); free(p); free(g); free(dg); free(dxs); free(fe); free(dz);
}

/* Selected entries of the same backward, at any size: each depends on a bounded set of slots.
 *   dh rows of the listed tokens (their k slots' input gradients, then the router's term);
 *   for each listed (expert e, hidden unit n): row n of dW1_e and of dW3_e (SwiGLU) and column n
 *   of dW2_e, sums over e's kept slots in token order.
 * z and p come from the router over all T tokens (the gates of every slot of a listed expert are
 * needed); counts are the routed counts of idx. Outputs: dh_rows [n_tok, d], dW1_rows and
 * dW3_rows [n_cols, d] (dW3_rows may be NULL), dW2_cols [n_cols, d] (dW2_e[o, n] at [c, o]). */
void oracle_backward_sampled(int64_t T, int32_t d, int32_t f, int32_t E, int32_t k, int32_t act,
                             int32_t gate_mode, const void *h, int32_t h_dtype, const float *W_r,
                             const float *b_r, const void *W1, const void *W3, const void *W2,
                             int32_t w_dtype, const float *b1, const float *b2,
                             const int32_t *idx, const unsigned char *keep, const void *dy,
                             int32_t dy_dtype, double aux_weight, double zloss_weight,
                             int64_t n_tok, const int64_t *tokens, double *dh_rows,
                             int64_t n_cols, const int32_t *col_e, const int32_t *col_n,
                             double *dW1_rows, double *dW3_rows, double *dW2_cols)
{
    const int64_t P = T * k;
    double *z = (double *)malloc(sizeof(double) * (size_t)(T * E + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(T * E + 1));
    double *g = (double *)malloc(sizeof(double) * (size_t)(P + 1));
    double *fe = (double *)calloc((size_t)(E > 0 ? E : 1), sizeof(double));
    oracle_router(T, d, E, h, h_dtype, W_r, b_r, z, p);
    oracle_gates(T, E, k, gate_mode, z, p, idx, g);
    for (int64_t s = 0; s < P; ++s) fe[idx[s]] += 1.0;
    for (int32_t e = 0; e < E; ++e) fe[e] /= (double)T * (double)k;

    /* dh rows: each token's slots, forward and backward in full, then the router term */
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)d);
        double *dyt = (double *)malloc(sizeof(double) * (size_t)d);
        double *a1 = (double *)malloc(sizeof(double) * (size_t)f);
        double *a3 = (double *)malloc(sizeof(double) * (size_t)f);
        double *hid = (double *)malloc(sizeof(double) * (size_t)f);
        double *dhid = (double *)malloc(sizeof(double) * (size_t)f);
        double *dg = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
        double *dz = (double *)malloc(sizeof(double) * (size_t)E);
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < n_tok; ++q) {
            const int64_t t = tokens[q];
            double *out = dh_rows + q * d;
            for (int32_t i = 0; i < d; ++i) {
                x[i] = widen(h, h_dtype, t * d + i);
                dyt[i] = widen(dy, dy_dtype, t * d + i);
                out[i] = 0.0;
            }
            for (int32_t j = 0; j < k; ++j) {
                const int64_t s = t * k + j;
                dg[j] = 0.0;
                if (keep && !keep[s]) continue;
                const int32_t e = idx[s];
                const int64_t base1 = (int64_t)e * f * d, base2 = (int64_t)e * d * f;
                for (int32_t n = 0; n < f; ++n) {
                    double u = 0.0, v = 0.0;
                    for (int32_t i = 0; i < d; ++i) {
                        u += widen(W1, w_dtype, base1 + (int64_t)n * d + i) * x[i];
                        if (act == OR_SWIGLU) v += widen(W3, w_dtype, base1 + (int64_t)n * d + i) * x[i];
                    }
                    if (act != OR_SWIGLU && b1) u += (double)b1[(int64_t)e * f + n];
                    a1[n] = u;
                    a3[n] = v;
                    hid[n] = act == OR_SWIGLU ? silu(u) * v : gelu_tanh(u);
                    dhid[n] = 0.0;
                }
                double dgs = 0.0;
                for (int32_t o = 0; o < d; ++o) {
                    double yo = 0.0;
                    for (int32_t n = 0; n < f; ++n) {
                        const double w2 = widen(W2, w_dtype, base2 + (int64_t)o * f + n);
                        yo += w2 * hid[n];
                        dhid[n] += w2 * g[s] * dyt[o];
                    }
                    if (act != OR_SWIGLU && b2) yo += (double)b2[(int64_t)e * d + o];
                    dgs += dyt[o] * yo;
                }
                dg[j] = dgs;
                for (int32_t n = 0; n < f; ++n) {
                    double d1, d3 = 0.0;
                    if (act == OR_SWIGLU) {
                        d1 = dhid[n] * a3[n] * silu_grad(a1[n]);
                        d3 = dhid[n] * silu(a1[n]);
                    } else {
                        d1 = dhid[n] * gelu_tanh_grad(a1[n]);
                    }
                    for (int32_t i = 0; i < d; ++i) {
                        out[i] += widen(W1, w_dtype, base1 + (int64_t)n * d + i) * d1;
                        if (act == OR_SWIGLU) out[i] += widen(W3, w_dtype, base1 + (int64_t)n * d + i) * d3;
                    }
                }
            }
            router_logit_grad(T, E, k, gate_mode, z + t * E, p + t * E, idx + t * k, g + t * k,
                              dg, fe, aux_weight, zloss_weight, dz);
            for (int32_t i = 0; i < d; ++i)
                for (int32_t e = 0; e < E; ++e) out[i] += (double)W_r[(int64_t)i * E + e] * dz[e];
        }
        free(x); free(dyt); free(a1); free(a3); free(hid); free(dhid); free(dg); free(dz);
    }

    /* weight-gradient rows and columns of the listed (e, n) */
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t c = 0; c < n_cols; ++c) {
            const int32_t e = col_e[c], n = col_n[c];
            const int64_t base1 = (int64_t)e * f * d, base2 = (int64_t)e * d * f;
            double *r1 = dW1_rows + c * d, *r2 = dW2_cols + c * d;
            double *r3 = dW3_rows ? dW3_rows + c * d : NULL;
            for (int32_t i = 0; i < d; ++i) {
                r1[i] = 0.0;
                r2[i] = 0.0;
                if (r3) r3[i] = 0.0;
            }
            for (int64_t s = 0; s < P; ++s) {
                if (idx[s] != e || (keep && !keep[s])) continue;
                const int64_t t = s / k;
                double u = 0.0, v = 0.0, dh_n = 0.0;
                for (int32_t i = 0; i < d; ++i) {
                    x[i] = widen(h, h_dtype, t * d + i);
                    u += widen(W1, w_dtype, base1 + (int64_t)n * d + i) * x[i];
                    if (act == OR_SWIGLU) v += widen(W3, w_dtype, base1 + (int64_t)n * d + i) * x[i];
                }
                if (act != OR_SWIGLU && b1) u += (double)b1[(int64_t)e * f + n];
                const double hid = act == OR_SWIGLU ? silu(u) * v : gelu_tanh(u);
                for (int32_t o = 0; o < d; ++o) {
                    const double dyo = g[s] * widen(dy, dy_dtype, t * d + o);
                    r2[o] += dyo * hid;
                    dh_n += widen(W2, w_dtype, base2 + (int64_t)o * f + n) * dyo;
                }
                double d1, d3 = 0.0;
                if (act == OR_SWIGLU) {
                    d1 = dh_n * v * silu_grad(u);
                    d3 = dh_n * silu(u);
                } else {
                    d1 = dh_n * gelu_tanh_grad(u);
                }
                for (int32_t i = 0; i < d; ++i) {
                    r1[i] += d1 * x[i];
                    if (r3) r3[i] += d3 * x[i];
                }
            }
        }
        free(x);
    }
    free(z); free(p); free(g); free(fe);
}
