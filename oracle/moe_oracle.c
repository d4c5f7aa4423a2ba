/*
 * moe_oracle.c -- plain, slow, CPU reference of the token-choice top-k
 * Mixture-of-Experts FFN layer forward.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  The product
 * (the CUDA library and its Python binding) never calls it, and it shares no
 * code, header, table or constant with the CUDA path.
 *
 * Arithmetic is fp64 throughout, except where the pages fix fp32:
 *   - router logits are stored as fp32 ("Mixture of Experts (MoE) From
 *     Scratch to DeepSeek V3", stability tricks: the router is computed in
 *     float32), and expert selection compares fp32 keys;
 *   - the sigmoid selection key of DeepSeek-V3-style routing is an fp32
 *     value (see orc_exp32 / orc_sigmoid32 below);
 *   - the aux-loss-free bias b_i is an fp32 parameter updated in place.
 * For bf16 layers the activation output H is rounded to bf16, because that
 * is the storage precision of the layer's intermediate (a bf16 Linear ->
 * activation -> Linear chain keeps H in bf16).
 *
 * Functions and the passages they follow:
 *   orc_router_logits    "MoE Training: Mixture of Experts", Quick Start
 *                        MoELayer (gate = nn.Linear(hidden, E) with bias);
 *                        "...From Scratch to DeepSeek V3", routing formula
 *                        h(x) = x . W_g.
 *   orc_route            same pages: softmax -> top-k -> renormalise
 *                        (MoELayer.forward; moe_code.py MixtureOfExperts
 *                        steps 1-3); sigmoid scores with selection bias b_i
 *                        (DeepSeek V3 page: sigmoid routing, aux-loss-free
 *                        balancing, Score_i = x.e_i + b_i).
 *   orc_capacity         "MoE Training Guide", Core MoE Parameters:
 *                        capacity = tokens / num_experts x capacity_factor,
 *                        min_capacity 4, drop_tokens.
 *   orc_dispatch         same + DeepSeek V3 page "Token Dropping": slots
 *                        beyond an expert's capacity are left unprocessed.
 *   orc_forward_tokens   moe_code.py MixtureOfExperts.forward, the
 *                        per-position loop  output[i] += p_j * E_j(x_i);
 *                        experts: Quick Start Linear-GELU-Linear,
 *                        moe_code.py Expert ReLU FFN (dropout = identity in
 *                        a forward pass), SwiGLU (three-matrix expert of the
 *                        Mixtral parameter arithmetic in the MoE technical
 *                        survey page); shared expert and the "+ x" residual
 *                        of the routing formula from the DeepSeek V3 page.
 *   orc_dense_all        moe_code.py EfficientMoE.forward: every expert on
 *                        every token, then gather and weight (brute force).
 *   orc_stats            "MoE Training: Mixture of Experts", Load Balancing
 *                        (auxiliary loss N * sum f_i P_i; router z-loss
 *                        mean(logsumexp^2)); "MoE Training Guide",
 *                        Monitoring (imbalance, utilisation, drop rate).
 *   orc_bias_update      DeepSeek V3 page, aux-loss-free balancing: lower
 *                        b_i for an overloaded expert, raise it for an idle
 *                        one.
 *   orc_param_counts     moe_code.py compare_moe_vs_dense; the Mixtral
 *                        parameter arithmetic of the MoE technical survey.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* configuration and tensors (the oracle's own layout description)     */
/* ------------------------------------------------------------------ */
typedef struct {
    int64_t T;               /* tokens (batch * seq, flattened)          */
    int32_t d, E, k, F;      /* d_model, routed experts, top_k, d_ff      */
    int32_t score_fn;        /* 0 softmax, 1 sigmoid                     */
    int32_t activation;      /* 0 GELU (erf), 1 ReLU, 2 SwiGLU           */
    int32_t renormalize;     /* 1: gates renormalised over the top-k     */
    int32_t drop_tokens;     /* 1: capacity limit applies                */
    int32_t min_capacity;
    int32_t num_shared;      /* always-on experts, weight 1              */
    int32_t residual;        /* 1: output adds x                          */
    int32_t dtype;           /* storage of x and all weights: 0 f32, 1 bf16 */
    double capacity_factor;
} orc_cfg;

typedef struct {
    const void *x;           /* [T, d]                                    */
    const void *w_router;    /* [E, d]                                    */
    const float *b_router;   /* [E] fp32, or NULL                         */
    const float *sel_bias;   /* [E] fp32 (sigmoid routing), or NULL       */
    const void *w1, *b1;     /* [E, F, d], [E, F] (b1 may be NULL)        */
    const void *w3;          /* [E, F, d] (SwiGLU only)                   */
    const void *w2, *b2;     /* [E, d, F], [E, d] (b2 may be NULL)        */
    const void *sw1, *sw3, *sw2; /* shared experts: [S,F,d],[S,F,d],[S,d,F] */
} orc_tensors;

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* storage decode: fp32 as is, bf16 = upper 16 bits of an fp32 (exact) */
static double elem(const void *p, int dtype, int64_t i) {
    if (dtype == 0) return (double)((const float *)p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static void decode_row(const void *p, int dtype, int64_t off, int64_t n, double *dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = elem(p, dtype, off + i);
}

static double dot_row(const void *p, int dtype, int64_t off, const double *v, int64_t n) {
    double acc = 0.0;
    if (dtype == 0) {
        const float *q = (const float *)p + off;
        for (int64_t i = 0; i < n; ++i) acc += (double)q[i] * v[i];
    } else {
        const uint16_t *q = (const uint16_t *)p + off;
        for (int64_t i = 0; i < n; ++i) {
            uint32_t u = (uint32_t)q[i] << 16;
            float f;
            memcpy(&f, &u, 4);
            acc += (double)f * v[i];
        }
    }
    return acc;
}

/* round an fp64 value to the nearest bf16 value (8 significant bits, ties to
 * even), returned as fp64.  Used only to mirror bf16 storage of H. */
double orc_round_bf16(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    int ex;
    double m = frexp(v, &ex);          /* v = m * 2^ex, 0.5 <= |m| < 1 */
    double q = nearbyint(m * 256.0);   /* 8 significant bits, ties-to-even */
    return ldexp(q / 256.0, ex);
}

/* ------------------------------------------------------------------ */
/* fp32 sigmoid key                                                      */
/* ------------------------------------------------------------------ */
/*
 * The selection key of sigmoid routing is an fp32 number, and an integer
 * decision (which experts) is taken on it, so both sides of a parity check
 * must produce the same bits.  The key is therefore fixed by a written
 * recipe built only from IEEE-754 correctly rounded fp32 operations:
 *
 *   exp32(a):  Cody-Waite argument reduction with ln 2 split in two
 *              (hi part = ln 2 truncated to 16 bits, lo part = the fp32
 *              remainder):  n = rint(a * log2e),  r = fma(-n, ln2_hi, a),
 *              r = fma(-n, ln2_lo, r);  e^r by the degree-7 Taylor
 *              polynomial sum r^i / i! in Horner form with fma;  result =
 *              p * 2^n (one multiply by an exact power of two).
 *              a > 88 gives +inf, a < -87 gives 0, NaN propagates.
 *   sigmoid32(x) = 1 / (1 + exp32(-x))      (fp32 add and divide)
 *   key         = sigmoid32(logit) + b_i     (fp32 add)
 *
 * Constants are the fp32 values nearest to log2(e), 1/i!, and the exact
 * 16-bit head of ln 2 with its fp32 tail.
 */
static const float K_LOG2E = 0x1.715476p+0f;
static const float K_LN2_HI = 0x1.62e4p-1f;
static const float K_LN2_LO = 0x1.7f7d1cp-20f;
static const float K_INV_FACT[8] = {1.0f, 1.0f, 0x1p-1f, 0x1.555556p-3f, 0x1.555556p-5f,
                                    0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f};

float orc_exp32(float a) {
    if (a != a) return a;
    if (a > 88.0f) return INFINITY;
    if (a < -87.0f) return 0.0f;
    float t = a * K_LOG2E;
    float n = rintf(t);
    float r = fmaf(-n, K_LN2_HI, a);
    r = fmaf(-n, K_LN2_LO, r);
    float p = K_INV_FACT[7];
    for (int i = 6; i >= 0; --i) p = fmaf(p, r, K_INV_FACT[i]);
    int ni = (int)n;                       /* -126 <= ni <= 127 here */
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float scale;
    memcpy(&scale, &bits, 4);
    return p * scale;
}

float orc_sigmoid32(float x) {
    float e = orc_exp32(-x);
    float den = 1.0f + e;
    return 1.0f / den;
}

/* selection keys of sigmoid routing for a [T, E] block of logits */
void orc_sigmoid_keys(const float *logits, const float *sel_bias, int64_t T, int64_t E, float *keys) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t e = 0; e < E; ++e) {
            float s = orc_sigmoid32(logits[t * E + e]);
            float b = sel_bias ? sel_bias[e] : 0.0f;
            keys[t * E + e] = s + b;
        }
}

/* ------------------------------------------------------------------ */
/* step 1: router logits                                                */
/* ------------------------------------------------------------------ */
/* logits[t,e] = sum_i x[t,i] * W_r[e,i] (+ b_r[e]), summed in fp64 and
 * stored as fp32. */
void orc_router_logits(const orc_cfg *c, const orc_tensors *w, float *logits) {
    const int64_t T = c->T, d = c->d, E = c->E;
    double *wr = (double *)malloc(sizeof(double) * (size_t)(E * d));
    decode_row(w->w_router, c->dtype, 0, E * d, wr);
#pragma omp parallel
    {
        double *xv = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            decode_row(w->x, c->dtype, t * d, d, xv);
            for (int64_t e = 0; e < E; ++e) {
                double acc = 0.0;
                const double *we = wr + e * d;
                for (int64_t i = 0; i < d; ++i) acc += xv[i] * we[i];
                if (w->b_router) acc += (double)w->b_router[e];
                logits[t * E + e] = (float)acc;
            }
        }
        free(xv);
    }
    free(wr);
}

/* ------------------------------------------------------------------ */
/* step 2: scores, top-k, gates, per-token logsumexp                   */
/* ------------------------------------------------------------------ */
/*
 * Keys: softmax routing ranks experts by their fp32 logit (softmax is
 * strictly increasing, so the top-k set of the probabilities is the top-k
 * set of the logits); sigmoid routing ranks by sigmoid32(logit) + b_i.
 * The k largest keys are taken largest first; equal keys go to the lower
 * expert index.
 *
 * Gates (fp64): softmax p_j = exp(l_j - lse); sigmoid s_j = 1/(1+exp(-l_j))
 * (b_i is not part of the gate).  With renormalize the selected values are
 * divided by their sum.
 *
 * Outputs: idx[t*k+j], gate[t*k+j], lse[t] (fp64) and, if prob_sum is not
 * NULL, prob_sum[e] = sum_t softmax(logits_t)_e summed in token order.
 */
void orc_route(const orc_cfg *c, const float *logits, const float *sel_bias,
               int32_t *idx, double *gate, double *lse, double *prob_sum) {
    const int64_t T = c->T, E = c->E, k = c->k;
#pragma omp parallel
    {
        float *key = (float *)malloc(sizeof(float) * (size_t)E);
        unsigned char *taken = (unsigned char *)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const float *l = logits + t * E;
            for (int64_t e = 0; e < E; ++e) {
                if (c->score_fn == 0) {
                    key[e] = l[e];
                } else {
                    float s = orc_sigmoid32(l[e]);
                    float b = sel_bias ? sel_bias[e] : 0.0f;
                    key[e] = s + b;
                }
                taken[e] = 0;
            }
            /* selection: k passes, each takes the largest remaining key */
            for (int64_t j = 0; j < k; ++j) {
                int64_t best = -1;
                for (int64_t e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    if (best < 0 || key[e] > key[best]) best = e;
                }
                taken[best] = 1;
                idx[t * k + j] = (int32_t)best;
            }
            /* log-sum-exp of the logits in fp64 */
            double m = -INFINITY;
            for (int64_t e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
            double s = 0.0;
            for (int64_t e = 0; e < E; ++e) s += exp((double)l[e] - m);
            lse[t] = m + log(s);
            /* gates */
            double tot = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                double le = (double)l[idx[t * k + j]];
                double v = (c->score_fn == 0) ? exp(le - lse[t]) : 1.0 / (1.0 + exp(-le));
                gate[t * k + j] = v;
                tot += v;
            }
            if (c->renormalize)
                for (int64_t j = 0; j < k; ++j) gate[t * k + j] /= tot;
        }
        free(key);
        free(taken);
    }
    if (prob_sum) {
        for (int64_t e = 0; e < E; ++e) prob_sum[e] = 0.0;
        for (int64_t t = 0; t < T; ++t)
            for (int64_t e = 0; e < E; ++e)
                prob_sum[e] += exp((double)logits[t * E + e] - lse[t]);
    }
}

/*
 * Hash routing (MoE technical survey page, "Hash layers for large sparse
 * models"; "hash-based route": a fixed token -> expert mapping fixed before
 * training, no gating network).  The page names no hash function; the one
 * used is MurmurHash3's 32-bit finalizer (fmix32) of token_id + j * 0x9E3779B9
 * (a golden-ratio stride per choice j), taken modulo E; a choice already
 * taken by an earlier j of the same token moves to the next expert,
 * cyclically.  Every chosen expert gets gate 1/k.
 */
uint32_t orc_fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

void orc_route_hash(int64_t T, int32_t E, int32_t k, const int32_t *token_ids, int32_t *idx, double *gate) {
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            uint32_t key = (uint32_t)token_ids[t] + (uint32_t)j * 0x9E3779B9u;
            int32_t e = (int32_t)(orc_fmix32(key) % (uint32_t)E);
            for (;;) {   /* next free expert if an earlier choice took e */
                int taken = 0;
                for (int32_t i = 0; i < j; ++i)
                    if (idx[t * k + i] == e) taken = 1;
                if (!taken) break;
                e = (e + 1) % E;
            }
            idx[t * k + j] = e;
            gate[t * k + j] = 1.0 / (double)k;
        }
    }
}

/*
 * Expert-choice routing ("MoE Training: Mixture of Experts", Routing
 * Mechanisms, Expert Choice: expert_scores = router(x) transposed, each
 * expert takes topk over tokens with k = capacity per expert).
 *   C = min(T, max(min_capacity, ceil(T / E * capacity_factor)))
 *   expert e takes the C tokens with the largest fp32 logit[t, e] (equal
 *   logits: lower token index first); its rows e*C .. e*C+C-1 hold those
 *   tokens in token order;
 *   gate(t, e) = softmax(logits_t)_e (fp64) for a chosen pair.
 * Outputs: row_token [E*C]; tok_row [T*E] (row of (t, e), -1 if e did not
 * choose t); tok_gate [T*E] (0 where not chosen).
 */
int64_t orc_ec_capacity(int64_t T, int32_t E, double cf, int32_t min_capacity) {
    int64_t c = (int64_t)ceil((double)T / (double)E * cf);
    if (c < min_capacity) c = min_capacity;
    return c < T ? c : T;
}

void orc_route_expert_choice(int64_t T, int32_t E, int64_t C, const float *logits, int32_t *row_token,
                             int32_t *tok_row, double *tok_gate) {
    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    unsigned char *chosen = (unsigned char *)malloc((size_t)(T > 0 ? T : 1));
    for (int64_t i = 0; i < T * E; ++i) {
        tok_row[i] = -1;
        tok_gate[i] = 0.0;
    }
    for (int32_t e = 0; e < E; ++e) {
        /* C selection passes: each takes the best remaining token */
        for (int64_t t = 0; t < T; ++t) chosen[t] = 0;
        for (int64_t r = 0; r < C; ++r) {
            int64_t best = -1;
            for (int64_t t = 0; t < T; ++t) {
                if (chosen[t]) continue;
                if (best < 0 || logits[t * E + e] > logits[best * E + e]) best = t;
            }
            if (best < 0) break;   /* C <= T: never */
            chosen[best] = 1;
        }
        int64_t n = 0;
        for (int64_t t = 0; t < T; ++t)
            if (chosen[t]) order[n++] = t;   /* token order */
        for (int64_t r = 0; r < n; ++r) {
            const int64_t t = order[r];
            row_token[e * C + r] = (int32_t)t;
            tok_row[t * E + e] = (int32_t)(e * C + r);
        }
    }
    for (int64_t t = 0; t < T; ++t) {
        double m = -INFINITY, s = 0.0;
        for (int32_t e = 0; e < E; ++e) m = fmax(m, (double)logits[t * E + e]);
        for (int32_t e = 0; e < E; ++e) s += exp((double)logits[t * E + e] - m);
        for (int32_t e = 0; e < E; ++e)
            if (tok_row[t * E + e] >= 0) tok_gate[t * E + e] = exp((double)logits[t * E + e] - m) / s;
    }
    free(order);
    free(chosen);
}

/* ------------------------------------------------------------------ */
/* step 3: capacity, drop, permutation                                  */
/* ------------------------------------------------------------------ */
/* capacity = max(min_capacity, ceil(T / E * capacity_factor)); without
 * token dropping every slot is kept (returns T * k, an upper bound). */
int64_t orc_capacity(const orc_cfg *c) {
    if (!c->drop_tokens) return c->T * (int64_t)c->k;
    double v = ceil((double)c->T / (double)c->E * c->capacity_factor);
    int64_t cap = (int64_t)v;
    return cap > c->min_capacity ? cap : c->min_capacity;
}

/*
 * Slots s = t*k + j are visited in priority order: all j = 0 slots in token
 * order, then all j = 1 slots, and so on (the Quick Start loop runs over
 * the top-k rank outside and the tokens inside).  Each slot takes the next
 * rank of its expert; a rank >= capacity is dropped.  Kept slots of expert
 * e fill rows offsets[e] .. offsets[e+1]-1 in that priority order.
 *
 * counts[e]: slots routed to e before dropping; kept[e] = min(counts, cap);
 * offsets[E+1]: exclusive prefix sum of kept; perm[row] = slot (rows past
 * offsets[E] are -1); inv[slot] = row or -1 for a dropped slot.
 */
void orc_dispatch(const orc_cfg *c, const int32_t *idx, int32_t *counts, int32_t *kept,
                  int32_t *offsets, int32_t *perm, int32_t *inv) {
    const int64_t T = c->T, E = c->E, k = c->k, S = T * k;
    const int64_t cap = orc_capacity(c);
    int32_t *rank = (int32_t *)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t j = 0; j < k; ++j)
        for (int64_t t = 0; t < T; ++t) {
            int64_t s = t * k + j;
            rank[s] = counts[idx[s]]++;
        }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) {
        kept[e] = counts[e] < cap ? counts[e] : (int32_t)cap;
        offsets[e + 1] = offsets[e] + kept[e];
    }
    for (int64_t r = 0; r < S; ++r) perm[r] = -1;
    for (int64_t s = 0; s < S; ++s) {
        if (rank[s] < cap) {
            int32_t row = offsets[idx[s]] + rank[s];
            inv[s] = row;
            perm[row] = (int32_t)s;
        } else {
            inv[s] = -1;
        }
    }
    free(rank);
}

/* ------------------------------------------------------------------ */
/* step 4: experts                                                       */
/* ------------------------------------------------------------------ */
static double act_gelu(double a) { return 0.5 * a * (1.0 + erf(a / sqrt(2.0))); }
static double act_relu(double a) { return a > 0.0 ? a : 0.0; }
static double act_silu(double a) { return a / (1.0 + exp(-a)); }

double orc_gelu(double a) { return act_gelu(a); }
double orc_silu(double a) { return act_silu(a); }

/*
 * One expert on one token row (fp64):
 *   GELU / ReLU:  y = W2 act(W1 x + b1) + b2
 *   SwiGLU:       y = W2 (silu(W1 x) * (W3 x))        (no biases)
 * W1, W3: [F, d] and W2: [d, F] slices of expert e; h holds F scratch values.
 */
static void expert_row(const orc_cfg *c, const void *W1, const void *B1, const void *W3,
                       const void *W2, const void *B2, int64_t e, const double *xv,
                       double *h, double *y) {
    const int64_t d = c->d, F = c->F;
    const int dt = c->dtype;
    for (int64_t f = 0; f < F; ++f) {
        double a = dot_row(W1, dt, e * F * d + f * d, xv, d);
        double v;
        if (c->activation == 2) {
            double u = dot_row(W3, dt, e * F * d + f * d, xv, d);
            v = act_silu(a) * u;
        } else {
            if (B1) a += elem(B1, dt, e * F + f);
            v = (c->activation == 0) ? act_gelu(a) : act_relu(a);
        }
        h[f] = (dt == 1) ? orc_round_bf16(v) : v;
    }
    for (int64_t n = 0; n < d; ++n) {
        double acc = dot_row(W2, dt, e * d * F + n * F, h, F);
        if (c->activation != 2 && B2) acc += elem(B2, dt, e * d + n);
        y[n] = acc;
    }
}

/* Exposed for tests: one routed expert on one row (y has d entries). */
void orc_expert_row(const orc_cfg *c, const orc_tensors *w, int64_t e, const double *xv, double *y) {
    double *h = (double *)malloc(sizeof(double) * (size_t)c->F);
    expert_row(c, w->w1, w->b1, w->w3, w->w2, w->b2, e, xv, h, y);
    free(h);
}

/* Several (expert, row) evaluations in parallel: y[i] = E_{experts[i]}(x[i]);
 * experts[i] < 0 selects shared expert -experts[i]-1.  x is fp64 [n, d]. */
void orc_expert_rows(const orc_cfg *c, const orc_tensors *w, int64_t n, const int32_t *experts,
                     const double *x, double *y) {
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)c->F);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n; ++i) {
            const int32_t e = experts[i];
            if (e >= 0)
                expert_row(c, w->w1, w->b1, w->w3, w->w2, w->b2, e, x + i * c->d, h, y + i * c->d);
            else
                expert_row(c, w->sw1, NULL, w->sw3, w->sw2, NULL, -e - 1, x + i * c->d, h, y + i * c->d);
        }
        free(h);
    }
}

/*
 * Layer output for the listed tokens (fp64, out[n_tok, d]):
 *   out_t = sum_j [slot kept] gate[t,j] * E_{idx[t,j]}(x_t)
 *         + sum_s Shared_s(x_t) + (residual ? x_t : 0)
 * summed in that order, j ascending.
 */
void orc_forward_tokens(const orc_cfg *c, const orc_tensors *w, const int32_t *idx,
                        const double *gate, const int32_t *inv, const int64_t *tokens,
                        int64_t n_tok, double *out) {
    const int64_t d = c->d, k = c->k;
#pragma omp parallel
    {
        double *xv = (double *)malloc(sizeof(double) * (size_t)d);
        double *y = (double *)malloc(sizeof(double) * (size_t)d);
        double *h = (double *)malloc(sizeof(double) * (size_t)c->F);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_tok; ++i) {
            const int64_t t = tokens[i];
            double *o = out + i * d;
            decode_row(w->x, c->dtype, t * d, d, xv);
            for (int64_t n = 0; n < d; ++n) o[n] = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                const int64_t s = t * k + j;
                if (inv && inv[s] < 0) continue;   /* dropped: contributes 0 */
                expert_row(c, w->w1, w->b1, w->w3, w->w2, w->b2, idx[s], xv, h, y);
                for (int64_t n = 0; n < d; ++n) o[n] += gate[s] * y[n];
            }
            for (int64_t sh = 0; sh < c->num_shared; ++sh) {
                expert_row(c, w->sw1, NULL, w->sw3, w->sw2, NULL, sh, xv, h, y);
                for (int64_t n = 0; n < d; ++n) o[n] += y[n];
            }
            if (c->residual)
                for (int64_t n = 0; n < d; ++n) o[n] += xv[n];
        }
        free(xv);
        free(y);
        free(h);
    }
}

/*
 * Brute force (EfficientMoE): all[t, e, :] = E_e(x_t) for every token and
 * every routed expert, then out_t = sum_j gate[t,j] * all[t, idx[t,j], :]
 * (+ shared + residual as above).  Dropped slots (inv < 0) are skipped.
 * Only for tiny layers: T * E expert evaluations.
 */
void orc_dense_all(const orc_cfg *c, const orc_tensors *w, const int32_t *idx,
                   const double *gate, const int32_t *inv, double *all, double *out) {
    const int64_t T = c->T, d = c->d, E = c->E, k = c->k;
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)c->F);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int64_t t = 0; t < T; ++t) {
        decode_row(w->x, c->dtype, t * d, d, xv);
        for (int64_t e = 0; e < E; ++e)
            expert_row(c, w->w1, w->b1, w->w3, w->w2, w->b2, e, xv, h, all + (t * E + e) * d);
    }
    for (int64_t t = 0; t < T; ++t) {
        double *o = out + t * d;
        decode_row(w->x, c->dtype, t * d, d, xv);
        for (int64_t n = 0; n < d; ++n) o[n] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            const int64_t s = t * k + j;
            if (inv && inv[s] < 0) continue;
            const double *sel = all + (t * E + idx[s]) * d;
            for (int64_t n = 0; n < d; ++n) o[n] += gate[s] * sel[n];
        }
        for (int64_t sh = 0; sh < c->num_shared; ++sh) {
            expert_row(c, w->sw1, NULL, w->sw3, w->sw2, NULL, sh, xv, h, y);
            for (int64_t n = 0; n < d; ++n) o[n] += y[n];
        }
        if (c->residual)
            for (int64_t n = 0; n < d; ++n) o[n] += xv[n];
    }
    free(xv);
    free(h);
    free(y);
}

/* ------------------------------------------------------------------ */
/* step 5: balance statistics and monitoring                            */
/* ------------------------------------------------------------------ */
/*
 * f_e = counts_e / (T k)            (fraction of routed slots, pre-drop)
 * P_e = prob_sum_e / T              (mean softmax probability)
 * aux = E * sum_e f_e P_e
 * z   = mean_t lse_t^2
 * scal[0..5] = aux, z, dropped, imbalance (max kept / min kept, +inf when
 * an expert is empty), utilisation (#experts with kept > 0 / E),
 * drop rate (dropped / (T k)).
 */
void orc_stats(const orc_cfg *c, const int32_t *counts, const int32_t *kept,
               const double *prob_sum, const double *lse, double *f, double *P, double *scal) {
    const int64_t T = c->T, E = c->E, S = c->T * (int64_t)c->k;
    double aux = 0.0, z = 0.0;
    int64_t dropped = 0, used = 0, kmax = 0, kmin = -1;
    for (int64_t e = 0; e < E; ++e) {
        f[e] = S > 0 ? (double)counts[e] / (double)S : 0.0;
        P[e] = T > 0 ? prob_sum[e] / (double)T : 0.0;
        aux += f[e] * P[e];
        dropped += counts[e] - kept[e];
        if (kept[e] > 0) ++used;
        if (kept[e] > kmax) kmax = kept[e];
        if (kmin < 0 || kept[e] < kmin) kmin = kept[e];
    }
    for (int64_t t = 0; t < T; ++t) z += lse[t] * lse[t];
    scal[0] = (double)E * aux;
    scal[1] = T > 0 ? z / (double)T : 0.0;
    scal[2] = (double)dropped;
    scal[3] = kmin > 0 ? (double)kmax / (double)kmin : INFINITY;
    scal[4] = (double)used / (double)E;
    scal[5] = S > 0 ? (double)dropped / (double)S : 0.0;
}

/* b_e <- b_e + gamma * sign(mean_load - counts_e), mean_load = T k / E,
 * sign(0) = 0, stored as fp32. */
void orc_bias_update(const orc_cfg *c, const int32_t *counts, float *bias, float gamma) {
    const int64_t E = c->E, S = c->T * (int64_t)c->k;
    for (int64_t e = 0; e < E; ++e) {
        int64_t diff = S - E * (int64_t)counts[e];   /* sign of S/E - counts_e */
        double sgn = diff > 0 ? 1.0 : (diff < 0 ? -1.0 : 0.0);
        bias[e] = (float)((double)bias[e] + (double)gamma * sgn);
    }
}

/* Parameter counts, biases ignored as on the pages:
 * out[0] = one expert (2 d F, or 3 d F for a gated expert), out[1] = router
 * d E, out[2] = total E * expert + router, out[3] = active k * expert +
 * router. */
void orc_param_counts(int64_t d, int64_t F, int64_t E, int64_t k, int gated, int64_t *out) {
    int64_t expert = (gated ? 3 : 2) * d * F;
    int64_t router = d * E;
    out[0] = expert;
    out[1] = router;
    out[2] = E * expert + router;
    out[3] = k * expert + router;
}

/* ------------------------------------------------------------------ */
/* backward                                                              */
/* ------------------------------------------------------------------ */
/*
 * Gradients of the training objective of one layer,
 *   L = sum_t <dout_t, out_t> + aux_coef * L_aux + z_coef * L_z,
 * with out, L_aux = E sum_e f_e P_e and L_z = mean_t lse_t^2 as in the
 * forward above.  No page prints a backward: the "MoE Training: Mixture of
 * Experts" page adds the auxiliary loss (and the router z-loss) to the main
 * loss of a training step, and the chain rule through the forward's
 * definitions gives every term below.
 *
 * Experts (slot j of token t kept in row inv[t,j], expert e, gate g):
 *   dy      = g * dout_t
 *   dW2_e  += dy h^T,  db2_e += dy,  dh = W2_e^T dy
 *   SwiGLU  h = silu(a1) * a3:  da1 = dh * a3 * silu'(a1),  da3 = dh * silu(a1)
 *   GELU / ReLU  h = act(a):    da = dh * act'(a)  (ReLU'(0) = 0)
 *   dW1_e  += da1 x^T,  dW3_e += da3 x^T,  db1_e += da,
 *   dx_t   += W1_e^T da1 (+ W3_e^T da3)
 *   dgate[t,j] = <dout_t, y>   (y the expert output; 0 for a dropped slot)
 * Shared experts: the same with g = 1 for every token.  Residual: dx += dout.
 * Router (fp64 from the fp32 logits l_t, p = softmax(l_t)):
 *   softmax, renormalised: w_j = p_j / sum_S p  ->  dl_j = w_j (dg_j - sum_i w_i dg_i)
 *   softmax, raw:          w_j = p_j             ->  dl_c = p_c (dg_c - sum_j p_j dg_j)
 *   sigmoid s = sigma(l), renormalised: w_j = s_j / sum_S s
 *                          ->  dl_j = s_j (1 - s_j) (dg_j - sum_i w_i dg_i) / sum_S s
 *   sigmoid, raw:          dl_j = s_j (1 - s_j) dg_j
 *   L_aux (f_e = counts_e / (T k) held constant, as a count has no gradient):
 *                          dl_c += aux_coef (E / T) p_c (f_c - sum_e f_e p_e)
 *   L_z:                   dl_c += z_coef (2 / T) lse_t p_c
 *   dW_r += dl x^T,  db_r += dl,  dx_t += W_r^T dl.
 *   The selection bias b_i enters only the choice, so it gets no gradient.
 * For bf16 layers the values the backward reads from bf16 storage are
 * rounded to bf16 at the points where they are stored: H (as in the
 * forward), the pre-activations a1 / a3 / a the forward keeps for the
 * backward (used by the activation derivative; H itself is formed from the
 * unrounded ones, as in the forward), dy and da1 / da3 / da; everything
 * else is fp64.
 *
 * Outputs (fp64, overwritten): dx [T,d], dw_router [E,d], db_router [E],
 * dw1 [E,F,d], db1 [E,F], dw3 [E,F,d], dw2 [E,d,F], db2 [E,d], dsw1 / dsw3
 * [S,F,d], dsw2 [S,d,F], dgate [T,k], dlogits [T,E]; NULL skips one.
 */
typedef struct {
    double *dx, *dw_router, *db_router, *dw1, *db1, *dw3, *dw2, *db2, *dsw1, *dsw3, *dsw2, *dgate, *dlogits;
} orc_grads;

static double rnd(const orc_cfg *c, double v) { return c->dtype == 1 ? orc_round_bf16(v) : v; }

static double act_grad(int activation, double a) {
    if (activation == 0) return 0.5 * (1.0 + erf(a / sqrt(2.0))) + a * exp(-0.5 * a * a) / sqrt(2.0 * acos(-1.0));
    return a > 0.0 ? 1.0 : 0.0;
}

/* Row f of one expert at input x: pre-activations (a1, a3 or a) and h_f. */
static void expert_unit(const orc_cfg *c, const void *W1, const void *B1, const void *W3, int64_t e, int64_t f,
                        const double *xv, double *a1, double *a3, double *h) {
    const int64_t d = c->d, F = c->F;
    *a1 = dot_row(W1, c->dtype, e * F * d + f * d, xv, d);
    if (c->activation == 2) {
        *a3 = dot_row(W3, c->dtype, e * F * d + f * d, xv, d);
        *h = rnd(c, act_silu(*a1) * *a3);
    } else {
        if (B1) *a1 += elem(B1, c->dtype, e * F + f);
        *a3 = 0.0;
        *h = rnd(c, c->activation == 0 ? act_gelu(*a1) : act_relu(*a1));
    }
}

/* d(pre-activations) of row f from dh_f (rounded like the stored operand). */
static void expert_unit_grad(const orc_cfg *c, double a1, double a3, double dh, double *da1, double *da3) {
    if (c->activation == 2) {
        const double sg = 1.0 / (1.0 + exp(-a1));
        const double dsilu = sg * (1.0 + a1 * (1.0 - sg));
        *da1 = rnd(c, dh * a3 * dsilu);
        *da3 = rnd(c, dh * act_silu(a1));
    } else {
        *da1 = rnd(c, dh * act_grad(c->activation, a1));
        *da3 = 0.0;
    }
}

/* Data path of one (expert, token): y (expert output) and dx += W^T da. */
static void expert_backward_row(const orc_cfg *c, const void *W1, const void *B1, const void *W3, const void *W2,
                                const void *B2, int64_t e, const double *xv, const double *dy, double *a1,
                                double *a3, double *h, double *y, double *dx) {
    const int64_t d = c->d, F = c->F;
    const int dt = c->dtype;
    for (int64_t f = 0; f < F; ++f) expert_unit(c, W1, B1, W3, e, f, xv, &a1[f], &a3[f], &h[f]);
    for (int64_t n = 0; n < d; ++n) {
        double acc = dot_row(W2, dt, e * d * F + n * F, h, F);
        if (c->activation != 2 && B2) acc += elem(B2, dt, e * d + n);
        y[n] = acc;
    }
    for (int64_t f = 0; f < F; ++f) {
        double dh = 0.0;
        for (int64_t n = 0; n < d; ++n) dh += elem(W2, dt, e * d * F + n * F + f) * dy[n];
        double da1, da3;
        expert_unit_grad(c, rnd(c, a1[f]), rnd(c, a3[f]), dh, &da1, &da3);
        for (int64_t i = 0; i < d; ++i) {
            dx[i] += elem(W1, dt, e * F * d + f * d + i) * da1;
            if (c->activation == 2) dx[i] += elem(W3, dt, e * F * d + f * d + i) * da3;
        }
    }
}

/* Weight gradients of one unit: row f of routed expert ee (ee < E) or of
 * shared expert ee - E, summed over the tokens the expert processed, in
 * token order.  Writes (when not NULL) dW1 row f [d], dW3 row f [d],
 * column f of dW2 [d], db1[f]; db2 [d] (the whole expert's, accumulated). */
static void wgrad_unit(const orc_cfg *c, const orc_tensors *w, const int32_t *idx, const double *gate,
                       const int32_t *inv, const double *dout, int64_t ee, int64_t f, double *dw1_row,
                       double *dw3_row, double *dw2_col, double *db1, double *db2) {
    const int64_t T = c->T, d = c->d, E = c->E, k = c->k, F = c->F;
    const int dt = c->dtype;
    const int shared = ee >= E;
    const int64_t e = shared ? ee - E : ee;
    const void *W1 = shared ? w->sw1 : w->w1, *W3 = shared ? w->sw3 : w->w3;
    const void *W2 = shared ? w->sw2 : w->w2, *B1 = shared ? NULL : w->b1;
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *dy = (double *)malloc(sizeof(double) * (size_t)d);
    if (dw1_row) memset(dw1_row, 0, sizeof(double) * (size_t)d);
    if (dw3_row) memset(dw3_row, 0, sizeof(double) * (size_t)d);
    if (dw2_col) memset(dw2_col, 0, sizeof(double) * (size_t)d);
    *db1 = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        double gt = 1.0;
        if (!shared) {
            int64_t jj = -1;
            for (int64_t j = 0; j < k; ++j)
                if (idx[t * k + j] == e && !(inv && inv[t * k + j] < 0)) jj = j;
            if (jj < 0) continue;
            gt = gate[t * k + jj];
        }
        decode_row(w->x, dt, t * d, d, xv);
        for (int64_t n = 0; n < d; ++n) dy[n] = rnd(c, gt * dout[t * d + n]);
        double a1, a3, h;
        expert_unit(c, W1, B1, W3, e, f, xv, &a1, &a3, &h);
        double dh = 0.0;
        for (int64_t n = 0; n < d; ++n) dh += elem(W2, dt, e * d * F + n * F + f) * dy[n];
        double da1, da3;
        expert_unit_grad(c, rnd(c, a1), rnd(c, a3), dh, &da1, &da3);
        if (dw1_row)
            for (int64_t i = 0; i < d; ++i) dw1_row[i] += da1 * xv[i];
        if (dw3_row && c->activation == 2)
            for (int64_t i = 0; i < d; ++i) dw3_row[i] += da3 * xv[i];
        if (dw2_col)
            for (int64_t n = 0; n < d; ++n) dw2_col[n] += dy[n] * h;
        *db1 += da1;
        if (db2)
            for (int64_t n = 0; n < d; ++n) db2[n] += dy[n];
    }
    free(xv);
    free(dy);
}

/* Weight gradients of the listed units only (u = ee * F + f, ee >= E for a
 * shared expert), each row [d]: dw1 / dw3 rows, dw2 columns, db1 values.
 * Same sums as orc_backward; for layers too large for full fp64 arrays. */
void orc_backward_units(const orc_cfg *c, const orc_tensors *w, const int32_t *idx, const double *gate,
                        const int32_t *inv, const double *dout, const int64_t *units, int64_t n, double *dw1,
                        double *dw3, double *dw2, double *db1) {
    const int64_t d = c->d, F = c->F;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i)
        wgrad_unit(c, w, idx, gate, inv, dout, units[i] / F, units[i] % F, dw1 + i * d, dw3 ? dw3 + i * d : NULL,
                   dw2 + i * d, db1 + i, NULL);
}

void orc_backward(const orc_cfg *c, const orc_tensors *w, const float *logits, const int32_t *idx,
                  const double *gate, const int32_t *inv, const int32_t *counts, const double *dout,
                  double aux_coef, double z_coef, orc_grads *g) {
    const int64_t T = c->T, d = c->d, E = c->E, k = c->k, F = c->F, S = c->num_shared;
    const int dt = c->dtype;
    double *dx = (double *)calloc((size_t)(T * d + 1), sizeof(double));
    double *dgate = (double *)calloc((size_t)(T * k + 1), sizeof(double));
    double *dl = (double *)calloc((size_t)(T * E + 1), sizeof(double));

    /* A: per token, experts' data path, dgate, residual */
#pragma omp parallel
    {
        double *xv = (double *)malloc(sizeof(double) * (size_t)d);
        double *dy = (double *)malloc(sizeof(double) * (size_t)d);
        double *y = (double *)malloc(sizeof(double) * (size_t)d);
        double *a1 = (double *)malloc(sizeof(double) * (size_t)F);
        double *a3 = (double *)malloc(sizeof(double) * (size_t)F);
        double *h = (double *)malloc(sizeof(double) * (size_t)F);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            decode_row(w->x, dt, t * d, d, xv);
            const double *go = dout + t * d;
            double *dxt = dx + t * d;
            for (int64_t j = 0; j < k; ++j) {
                const int64_t s = t * k + j;
                if (inv && inv[s] < 0) continue;
                for (int64_t n = 0; n < d; ++n) dy[n] = rnd(c, gate[s] * go[n]);
                expert_backward_row(c, w->w1, w->b1, w->w3, w->w2, w->b2, idx[s], xv, dy, a1, a3, h, y, dxt);
                double acc = 0.0;
                for (int64_t n = 0; n < d; ++n) acc += go[n] * y[n];
                dgate[s] = acc;
            }
            for (int64_t sh = 0; sh < S; ++sh) {
                for (int64_t n = 0; n < d; ++n) dy[n] = rnd(c, go[n]);
                expert_backward_row(c, w->sw1, NULL, w->sw3, w->sw2, NULL, sh, xv, dy, a1, a3, h, y, dxt);
            }
            if (c->residual)
                for (int64_t n = 0; n < d; ++n) dxt[n] += go[n];
        }
        free(xv);
        free(dy);
        free(y);
        free(a1);
        free(a3);
        free(h);
    }

    /* B: router, per token */
    double *fe = (double *)malloc(sizeof(double) * (size_t)(E + 1));
    for (int64_t e = 0; e < E; ++e) fe[e] = T * k > 0 ? (double)counts[e] / (double)(T * k) : 0.0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        double *wr = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const float *l = logits + t * E;
            double *dlt = dl + t * E;
            double m = -INFINITY;
            for (int64_t e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
            double ssum = 0.0;
            for (int64_t e = 0; e < E; ++e) ssum += exp((double)l[e] - m);
            const double lse = m + log(ssum);
            for (int64_t e = 0; e < E; ++e) p[e] = exp((double)l[e] - lse);
            const int32_t *it = idx + t * k;
            const double *dg = dgate + t * k;
            if (c->score_fn == 0) {
                if (c->renormalize) {
                    double tot = 0.0, wdg = 0.0;
                    for (int64_t j = 0; j < k; ++j) tot += p[it[j]];
                    for (int64_t j = 0; j < k; ++j) wdg += p[it[j]] / tot * dg[j];
                    for (int64_t j = 0; j < k; ++j) dlt[it[j]] += p[it[j]] / tot * (dg[j] - wdg);
                } else {
                    double pdg = 0.0;
                    for (int64_t j = 0; j < k; ++j) pdg += p[it[j]] * dg[j];
                    for (int64_t e = 0; e < E; ++e) dlt[e] -= p[e] * pdg;
                    for (int64_t j = 0; j < k; ++j) dlt[it[j]] += p[it[j]] * dg[j];
                }
            } else {
                double tot = 0.0, wdg = 0.0;
                for (int64_t j = 0; j < k; ++j) tot += 1.0 / (1.0 + exp(-(double)l[it[j]]));
                for (int64_t j = 0; j < k; ++j) {
                    const double sj = 1.0 / (1.0 + exp(-(double)l[it[j]]));
                    wdg += sj / tot * dg[j];
                }
                for (int64_t j = 0; j < k; ++j) {
                    const double sj = 1.0 / (1.0 + exp(-(double)l[it[j]]));
                    const double ds = c->renormalize ? (dg[j] - wdg) / tot : dg[j];
                    dlt[it[j]] += sj * (1.0 - sj) * ds;
                }
            }
            double fp = 0.0;
            for (int64_t e = 0; e < E; ++e) fp += fe[e] * p[e];
            for (int64_t e = 0; e < E; ++e) {
                dlt[e] += aux_coef * ((double)E / (double)T) * p[e] * (fe[e] - fp);
                dlt[e] += z_coef * (2.0 / (double)T) * lse * p[e];
            }
            double *dxt = dx + t * d;
            for (int64_t e = 0; e < E; ++e) {
                decode_row(w->w_router, dt, e * d, d, wr);
                for (int64_t i = 0; i < d; ++i) dxt[i] += dlt[e] * wr[i];
            }
        }
        free(p);
        free(wr);
    }

    /* C: weight gradients, per (expert, row f); the expert's tokens in
     * token order */
    const int64_t n_units = (E + S) * F;
    if (g->dw1 || g->dw2 || g->dw3 || g->db1 || g->db2 || g->dsw1 || g->dsw2 || g->dsw3) {
        if (g->dw1) memset(g->dw1, 0, sizeof(double) * (size_t)(E * F * d));
        if (g->dw3) memset(g->dw3, 0, sizeof(double) * (size_t)(E * F * d));
        if (g->dw2) memset(g->dw2, 0, sizeof(double) * (size_t)(E * d * F));
        if (g->db1) memset(g->db1, 0, sizeof(double) * (size_t)(E * F));
        if (g->db2) memset(g->db2, 0, sizeof(double) * (size_t)(E * d));
        if (g->dsw1) memset(g->dsw1, 0, sizeof(double) * (size_t)(S * F * d));
        if (g->dsw3) memset(g->dsw3, 0, sizeof(double) * (size_t)(S * F * d));
        if (g->dsw2) memset(g->dsw2, 0, sizeof(double) * (size_t)(S * d * F));
#pragma omp parallel
        {
            double *col = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
            for (int64_t u = 0; u < n_units; ++u) {
                const int64_t ee = u / F, f = u % F;
                const int shared = ee >= E;
                const int64_t e = shared ? ee - E : ee;
                double *dW1 = shared ? g->dsw1 : g->dw1, *dW3 = shared ? g->dsw3 : g->dw3;
                double *dW2 = shared ? g->dsw2 : g->dw2;
                double db1 = 0.0;
                wgrad_unit(c, w, idx, gate, inv, dout, ee, f, dW1 ? dW1 + e * F * d + f * d : NULL,
                           dW3 ? dW3 + e * F * d + f * d : NULL, col, &db1,
                           (!shared && g->db2 && f == 0) ? g->db2 + e * d : NULL);
                if (dW2)
                    for (int64_t n = 0; n < d; ++n) dW2[e * d * F + n * F + f] = col[n];
                if (!shared && g->db1) g->db1[e * F + f] = db1;
            }
            free(col);
        }
    }
    if (g->dw_router || g->db_router) {
        if (g->dw_router) memset(g->dw_router, 0, sizeof(double) * (size_t)(E * d));
        if (g->db_router) memset(g->db_router, 0, sizeof(double) * (size_t)E);
#pragma omp parallel for schedule(static)
        for (int64_t e = 0; e < E; ++e) {
            for (int64_t t = 0; t < T; ++t) {
                const double v = dl[t * E + e];
                if (g->db_router) g->db_router[e] += v;
                if (g->dw_router)
                    for (int64_t i = 0; i < d; ++i) g->dw_router[e * d + i] += v * elem(w->x, dt, t * d + i);
            }
        }
    }
    if (g->dx) memcpy(g->dx, dx, sizeof(double) * (size_t)(T * d));
    if (g->dgate) memcpy(g->dgate, dgate, sizeof(double) * (size_t)(T * k));
    if (g->dlogits) memcpy(g->dlogits, dl, sizeof(double) * (size_t)(T * E));
    free(dx);
    free(dgate);
    free(dl);
    free(fe);
}
