/*
 * oracle.c -- plain, slow CPU reference for the forward pass of a sparse
 * Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path
 * (the CUDA library under sparse_mixture_experts_69_b300/) shares no code
 * with it and never calls it.
 *
 * Everything is computed in double with per-token loops, in the order the
 * method is described:
 *   router      "MoE notes" (chiang97912.github.io), section Expert
 *               selection: G(x) = softmax(x . Wg); section KeepTopK:
 *               H(x)_i = (x.Wg)_i + StandardNormal() * Softplus((x.Wnoise)_i),
 *               KeepTopK(v,k), G(x) = Softmax(KeepTopK(H(x),k)).
 *   softmax     heavensheep.xyz "MoE" notes, section Training, the
 *               10-logit example: subtract the max, exponentiate in high
 *               precision.
 *   sel. bias   ld246.com "MoE" Q3 (loss-free bias balance): a per-expert
 *               bias is added to the softmax scores before Top-K only.
 *   capacity    "MoE notes", section Expert capacity: capacity =
 *               tokens per batch / number of experts * capacity factor;
 *               mkbk-pku.cn MoE notes, load balance section: overflowing
 *               tokens are dropped (output zero / residual path).
 *   experts     mkbk-pku.cn MoE notes, section on experts: each expert is
 *               an FFN, two linear maps around an activation.
 *   combine     "MoE notes": y = sum_i G(x)_i E_i(x).
 *   aux stats   heavensheep.xyz notes (Switch aux loss from f_i, P_i);
 *               "MoE notes", section Auxiliary loss: Importance(X) =
 *               sum_x G(x), CV = sigma/mu, L = w * CV^2.
 *   bias update heavensheep.xyz notes / ld246.com Q3: an over-used expert's
 *               bias goes down, an idle expert's goes up.
 *   overflow    "MoE notes", section Expert capacity: once an expert is
 *   policies    full, later tokens go to their next candidate expert, and a
 *               token whose candidates are all full skips the layer;
 *               mkbk-pku.cn MoE notes, capacity section: drop, second-choice
 *               re-routing, or padding every expert to its capacity.
 *   expert      heavensheep.xyz notes, Routing Function ("expert choose
 *   choice      token" balances the load); xutianle.me CS336-04, section 3
 *               (routing can be reversed: experts select tokens).
 *   sequence    heavensheep.xyz notes, Training: the same balance
 *   statistics  statistics taken inside each sequence instead of the batch.
 *   noise       the router's StandardNormal() draws, when drawn rather than
 *               passed in: Philox4x32-10 and the Box-Muller transform (the
 *               generator is not the pages'; see oracle_philox4x32_10).
 *
 * Inputs arrive as float (bf16 values are widened exactly by the caller).
 * Rounding of intermediates to the storage dtype is optional (round_dtype:
 * -1 none, 0 fp32, 1 bf16) so that the pure-double definition can be
 * pinned and the GPU's storage policy can be mirrored.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_RELU 0
#define ORACLE_GELU 1
#define ORACLE_SWIGLU 2

/* ---------------------------------------------------------------- rounding */

/* Round a double to the nearest bfloat16 (ties to even), returned as double. */
static double round_bf16(double v) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int e;
    double m = frexp(fabs(v), &e); /* |v| = m * 2^e, m in [0.5, 1) */
    /* bf16 keeps 8 significant bits: scale so the kept bits are the integer part */
    double scaled = ldexp(m, 8);
    double r = nearbyint(scaled); /* default rounding mode: to nearest, ties to even */
    double out = ldexp(r, e - 8);
    /* below the smallest normal bf16 (2^-126) the grid is 2^-133 */
    if (fabs(v) < ldexp(1.0, -126)) out = ldexp(nearbyint(ldexp(fabs(v), 133)), -133);
    if (out > 3.3895313892515355e38) out = INFINITY; /* beyond the largest finite bf16 */
    return v < 0 ? -out : out;
}

static double round_to(double v, int round_dtype) {
    if (round_dtype == 0) return (double)(float)v;
    if (round_dtype == 1) return round_bf16(v);
    return v;
}

double oracle_round(double v, int round_dtype) { return round_to(v, round_dtype); }

/* ----------------------------------------------------------------- scalars */

double oracle_softplus(double u) { return fmax(u, 0.0) + log1p(exp(-fabs(u))); }

/* ------------------------------------------------------------ router noise */

/* The StandardNormal() draws of the noisy router ("MoE notes", KeepTopK), when
 * they are drawn rather than passed in. The pages name no generator; this is
 * the counter-based Philox4x32-10 of Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3" (SC 2011): ten rounds, each two 32x32
 * -> 64-bit products with the multipliers 0xD2511F53 and 0xCD9E8D57, the high
 * halves xored with the other counter words and the key, the key bumped by
 * 0x9E3779B9 and 0xBB67AE85 between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n1 = lo1;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        const uint32_t n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
        if (round < 9) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* eps[t,e] for the stream (seed, counter): the Philox block with counter words
 * (e, t, counter low, counter high) and key (seed low, seed high) gives r0, r1;
 * their top 24 bits make u1 = (r0 >> 8) + 1 over 2^24 in (0, 1] and u2 =
 * (r1 >> 8) over 2^24 in [0, 1); Box and Muller (1958) turn them into the
 * standard normal sqrt(-2 ln u1) cos(2 pi u2). */
static const double kPi = 3.14159265358979323846;

void oracle_draw_noise(int T, int E, uint64_t seed, uint64_t counter, double* eps) {
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            const uint32_t ctr[4] = {(uint32_t)e, (uint32_t)t, (uint32_t)counter,
                                     (uint32_t)(counter >> 32)};
            uint32_t r[4];
            oracle_philox4x32_10(ctr, key, r);
            const double u1 = (double)((r[0] >> 8) + 1u) / 16777216.0;
            const double u2 = (double)(r[1] >> 8) / 16777216.0;
            eps[(size_t)t * E + e] = sqrt(-2.0 * log(u1)) * cos(2.0 * kPi * u2);
        }
}

static double act_relu(double u) { return u > 0.0 ? u : 0.0; }
/* GELU, exact form u * Phi(u); Phi written with erfc to avoid cancellation for u << 0 */
static double act_gelu(double u) { return 0.5 * u * erfc(-u / sqrt(2.0)); }
static double act_silu(double u) { return u / (1.0 + exp(-u)); }

double oracle_activation(int act, double u) {
    if (act == ORACLE_RELU) return act_relu(u);
    if (act == ORACLE_GELU) return act_gelu(u);
    return act_silu(u);
}

/* Max-subtracted softmax of n values (double in, double out). */
void oracle_softmax(int n, const double* v, double* p) {
    double m = v[0];
    for (int i = 1; i < n; ++i)
        if (v[i] > m) m = v[i];
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
        p[i] = exp(v[i] - m);
        sum += p[i];
    }
    for (int i = 0; i < n; ++i) p[i] /= sum;
}

/* -------------------------------------------------------------- selection */

/* KeepTopK on one row: the k largest scores, largest first; among equal
 * scores the lower expert index comes first. */
static void topk_row(int E, int k, const double* s, int32_t* ids) {
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            int taken = 0;
            for (int q = 0; q < j; ++q)
                if (ids[q] == e) taken = 1;
            if (taken) continue;
            if (best < 0 || s[e] > s[best]) best = e;
        }
        ids[j] = best;
    }
}

/* Gate weights for the chosen experts: renorm=1 gives
 * Softmax(KeepTopK(.)) = p_j / sum of chosen p; renorm=0 gives p_j. */
static void gates_row(int k, const int32_t* ids, const double* p, int renorm, double* w) {
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += p[ids[j]];
    for (int j = 0; j < k; ++j) w[j] = renorm ? p[ids[j]] / sum : p[ids[j]];
}

/* Top-k and gates from given selection scores s[T,E] and probabilities
 * p[T,E] (both float, as stored by a caller). */
void oracle_select(int T, int E, int k, const float* s, const float* p, int renorm,
                   int32_t* ids, double* w) {
    double* srow = (double*)malloc(sizeof(double) * E);
    double* prow = (double*)malloc(sizeof(double) * E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            srow[e] = s[(size_t)t * E + e];
            prow[e] = p[(size_t)t * E + e];
        }
        topk_row(E, k, srow, ids + (size_t)t * k);
        gates_row(k, ids + (size_t)t * k, prow, renorm, w + (size_t)t * k);
    }
    free(srow);
    free(prow);
}

/* Top-n_cand candidates per token (n_cand >= k): the first k are the
 * KeepTopK choice, the rest are the next candidates in score order, tried
 * when a choice is full. Every candidate's gate uses the denominator of the
 * top-k choice: w_j = p_j / sum_{j'<k} p_j' (renorm=1) or p_j (renorm=0), so
 * the capacity stage never changes a gate value, only which candidates are
 * kept. ids and w are [T,n_cand]. */
void oracle_select_candidates(int T, int E, int k, int n_cand, const float* s, const float* p,
                              int renorm, int32_t* ids, double* w) {
    double* srow = (double*)malloc(sizeof(double) * E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) srow[e] = s[(size_t)t * E + e];
        int32_t* id = ids + (size_t)t * n_cand;
        topk_row(E, n_cand, srow, id);
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += (double)p[(size_t)t * E + id[j]];
        for (int j = 0; j < n_cand; ++j) {
            double pj = (double)p[(size_t)t * E + id[j]];
            w[(size_t)t * n_cand + j] = renorm ? pj / den : pj;
        }
    }
    free(srow);
}

/* ----------------------------------------------------------------- router */

/* Router for T tokens.
 *   z[t,e] = sum_i x[t,i] Wg[i,e] (+ offset[e])            logits
 *   H[t,e] = z[t,e] + noise[t,e] * softplus(zn[t,e])       if Wnoise && noise
 *            zn[t,e] = sum_i x[t,i] Wnoise[i,e]
 *   p[t,:] = softmax(H[t,:])
 *   s[t,e] = H[t,e]             without a selection bias (softmax is monotone)
 *          = p[t,e] + bias[e]   with one
 *   ids    = KeepTopK(s, k), gates w from p.
 * x is [T,d], Wg and Wnoise are [d,E]; optional pointers may be NULL. */
void oracle_router(int T, int d, int E, int k, const float* x, const float* Wg,
                   const float* Wnoise, const float* noise, const float* offset,
                   const float* bias, int renorm, double* z, double* H, double* p, double* s,
                   int32_t* ids, double* w) {
#pragma omp parallel
    {
        double* zn = (double*)malloc(sizeof(double) * E);
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            const float* xt = x + (size_t)t * d;
            double* zt = z + (size_t)t * E;
            double* Ht = H + (size_t)t * E;
            double* pt = p + (size_t)t * E;
            double* st = s + (size_t)t * E;
            /* each z[t,e] (and zn[t,e]) is summed over i = 0..d-1 in order; the
             * loop over e sits inside only so that Wg is read row by row */
            for (int e = 0; e < E; ++e) {
                zt[e] = 0.0;
                zn[e] = 0.0;
            }
            for (int i = 0; i < d; ++i) {
                const double xi = (double)xt[i];
                const float* wrow = Wg + (size_t)i * E;
                for (int e = 0; e < E; ++e) zt[e] += xi * (double)wrow[e];
                if (Wnoise && noise) {
                    const float* nrow = Wnoise + (size_t)i * E;
                    for (int e = 0; e < E; ++e) zn[e] += xi * (double)nrow[e];
                }
            }
            for (int e = 0; e < E; ++e) {
                if (offset) zt[e] += (double)offset[e];
                double h = zt[e];
                if (Wnoise && noise) h += (double)noise[(size_t)t * E + e] * oracle_softplus(zn[e]);
                Ht[e] = h;
            }
            oracle_softmax(E, Ht, pt);
            for (int e = 0; e < E; ++e) st[e] = bias ? pt[e] + (double)bias[e] : Ht[e];
            topk_row(E, k, st, ids + (size_t)t * k);
            gates_row(k, ids + (size_t)t * k, pt, renorm, w + (size_t)t * k);
        }
        free(zn);
    }
}

/* --------------------------------------------------------------- capacity */

/* Expert capacity: (tokens per batch / number of experts) * capacity factor,
 * rounded up; a non-positive factor means no limit (capacity = T). */
int oracle_capacity_of(int T, int E, float capacity_factor) {
    if (capacity_factor <= 0.0f) return T;
    return (int)ceil((double)T * (double)capacity_factor / (double)E);
}

/* Token-order slot assignment. Assignments are visited token by token
 * (and within a token in rank order); each takes the next free slot of its
 * expert and is kept while that slot is below the capacity C. Outputs:
 *   counts[e]  assignments routed to e before the cap
 *   kept[e]    = min(counts[e], C)
 *   offsets    exclusive prefix sum of kept, E+1 entries
 *   slot[t,j]  row offsets[e] + slot of a kept assignment, -1 if dropped
 *   row_token  token of each kept row (length offsets[E]) */
void oracle_capacity(int T, int k, int E, int C, const int32_t* ids, int32_t* counts,
                     int32_t* kept, int32_t* offsets, int32_t* slot, int32_t* row_token) {
    int32_t* local = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            int sl = counts[e]++;
            local[(size_t)t * k + j] = sl < C ? sl : -1;
        }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        kept[e] = counts[e] < C ? counts[e] : C;
        offsets[e + 1] = offsets[e] + kept[e];
    }
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            size_t a = (size_t)t * k + j;
            if (local[a] < 0) {
                slot[a] = -1;
            } else {
                int row = offsets[ids[a]] + local[a];
                slot[a] = row;
                row_token[row] = t;
            }
        }
    free(local);
}

/* Capacity with an overflow policy. Each token needs k experts and holds
 * n_cand >= k candidates ids[t,0..n_cand-1] in rank order. Candidates are
 * visited one at a time in the priority order
 *   priority 0 (token order): token by token, each token's candidates in rank order
 *   priority 1 (rank order):  rank by rank, each rank's tokens in token order
 * and a visit does: if the token still needs an expert, it tries the candidate;
 * the try succeeds when the expert holds fewer than C rows, and the candidate
 * takes the expert's next row. A failed try moves the token on to its next
 * candidate (re-routing); a token that runs out of candidates keeps fewer than
 * k experts (with n_cand == k this is plain dropping).
 * Outputs:
 *   counts[e]  top-k choices (candidates 0..k-1) naming e, before capacity
 *   kept[e]    rows taken by expert e
 *   offsets    pad == 0: exclusive prefix sum of kept (E+1 entries);
 *              pad == 1: offsets[e] = e C (every expert's block is C rows)
 *   slot[t,j]  row of a kept candidate, -1 otherwise ([T,n_cand])
 *   row_token  token of each kept row */
void oracle_capacity_policy(int T, int k, int n_cand, int E, int C, const int32_t* ids,
                            int priority, int pad, int32_t* counts, int32_t* kept,
                            int32_t* offsets, int32_t* slot, int32_t* row_token) {
    const size_t n = (size_t)T * n_cand;
    int32_t* local = (int32_t*)malloc(sizeof(int32_t) * (n ? n : 1));
    int32_t* need = (int32_t*)malloc(sizeof(int32_t) * (T ? T : 1));
    for (int e = 0; e < E; ++e) {
        counts[e] = 0;
        kept[e] = 0;
    }
    for (int t = 0; t < T; ++t) {
        need[t] = k;
        for (int j = 0; j < k; ++j) counts[ids[(size_t)t * n_cand + j]] += 1;
    }
    for (size_t a = 0; a < n; ++a) local[a] = -1;
    for (size_t v = 0; v < n; ++v) {
        int t, j;
        if (priority == 0) {
            t = (int)(v / n_cand);
            j = (int)(v % n_cand);
        } else {
            j = (int)(v / T);
            t = (int)(v % T);
        }
        if (need[t] == 0) continue;
        size_t a = (size_t)t * n_cand + j;
        int e = ids[a];
        if (kept[e] < C) {
            local[a] = kept[e];
            kept[e] += 1;
            need[t] -= 1;
        }
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = pad ? (e + 1) * C : offsets[e] + kept[e];
    for (size_t a = 0; a < n; ++a) {
        if (local[a] < 0) {
            slot[a] = -1;
        } else {
            int row = offsets[ids[a]] + local[a];
            slot[a] = row;
            row_token[row] = (int32_t)(a / n_cand);
        }
    }
    free(local);
    free(need);
}

/* Expert-choice routing: expert e takes the C tokens with the largest
 * probability p[t,e] (ties: the lower token index first). Expert e's rows are
 * e C .. e C + C - 1, holding its chosen tokens in increasing token order; the
 * gate of a row is p[token,e]. C must not exceed T.
 *   row_token [E*C], row_w [E*C], tok_row [T,E] (row of (t,e) or -1). */
typedef struct {
    double p;
    int t;
} oracle_pt;
static int cmp_pt_desc(const void* a, const void* b) {
    const oracle_pt* x = (const oracle_pt*)a;
    const oracle_pt* y = (const oracle_pt*)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    return x->t < y->t ? -1 : (x->t > y->t);
}
static int cmp_int(const void* a, const void* b) {
    int x = *(const int*)a, y = *(const int*)b;
    return x < y ? -1 : (x > y);
}
void oracle_expert_choice(int T, int E, int C, const float* p, int32_t* row_token, double* row_w,
                          int32_t* tok_row) {
    oracle_pt* col = (oracle_pt*)malloc(sizeof(oracle_pt) * (T ? T : 1));
    int* chosen = (int*)malloc(sizeof(int) * (C ? C : 1));
    for (size_t i = 0; i < (size_t)T * E; ++i) tok_row[i] = -1;
    for (int e = 0; e < E; ++e) {
        for (int t = 0; t < T; ++t) {
            col[t].p = (double)p[(size_t)t * E + e];
            col[t].t = t;
        }
        qsort(col, T, sizeof(oracle_pt), cmp_pt_desc);
        for (int i = 0; i < C; ++i) chosen[i] = col[i].t;
        qsort(chosen, C, sizeof(int), cmp_int);
        for (int i = 0; i < C; ++i) {
            int r = e * C + i, t = chosen[i];
            row_token[r] = t;
            row_w[r] = (double)p[(size_t)t * E + e];
            tok_row[(size_t)t * E + e] = r;
        }
    }
    free(col);
    free(chosen);
}

/* Dispatch: xp[slot[t,j]] = x[t] for every kept assignment. */
void oracle_dispatch(int T, int d, int k, const float* x, const int32_t* slot, float* xp) {
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int row = slot[(size_t)t * k + j];
            if (row < 0) continue;
            memcpy(xp + (size_t)row * d, x + (size_t)t * d, sizeof(float) * d);
        }
}

/* ------------------------------------------------------------------ FFN */

/* One expert FFN on n rows X[n,d]:
 *   ReLU/GELU : h = act(W1 x),  W1 [F,d]
 *   SwiGLU    : h = silu(W1[0:F] x) * (W1[F:2F] x),  W1 [2F,d]
 *   out       : o = W2 h,  W2 [d,F]
 * h and o are rounded to round_dtype (the storage dtype) when >= 0. */
void oracle_expert_ffn(int n, int d, int F, int act, const float* W1, const float* W2,
                       const float* X, int round_dtype, double* O) {
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * F);
#pragma omp for schedule(static)
        for (int r = 0; r < n; ++r) {
            const float* xr = X + (size_t)r * d;
            for (int f = 0; f < F; ++f) {
                double u = 0.0;
                const float* w = W1 + (size_t)f * d;
                for (int i = 0; i < d; ++i) u += (double)w[i] * (double)xr[i];
                double hv;
                if (act == ORACLE_SWIGLU) {
                    double up = 0.0;
                    const float* wu = W1 + (size_t)(F + f) * d;
                    for (int i = 0; i < d; ++i) up += (double)wu[i] * (double)xr[i];
                    hv = act_silu(u) * up;
                } else {
                    hv = oracle_activation(act, u);
                }
                h[f] = round_to(hv, round_dtype);
            }
            for (int j = 0; j < d; ++j) {
                double o = 0.0;
                const float* w2 = W2 + (size_t)j * F;
                for (int f = 0; f < F; ++f) o += (double)w2[f] * h[f];
                O[(size_t)r * d + j] = round_to(o, round_dtype);
            }
        }
        free(h);
    }
}

/* ---------------------------------------------------------------- combine */

/* y[t] = sum over kept j of w[t,j] * O[t,j,:]  +  sum_s Os[s,t,:].
 * O is [n,k,d] (expert outputs per assignment), Os is [S,n,d] or NULL.
 * A dropped assignment (slot < 0) contributes nothing; the gates are not
 * renormalised after a drop. */
void oracle_combine(int n, int d, int k, int S, const double* w, const int32_t* slot,
                    const double* O, const double* Os, int round_dtype, double* y) {
    for (int t = 0; t < n; ++t)
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                size_t a = (size_t)t * k + j;
                if (slot[a] < 0) continue;
                acc += w[a] * O[a * d + i];
            }
            for (int s = 0; s < S; ++s) acc += Os[((size_t)s * n + t) * d + i];
            y[(size_t)t * d + i] = round_to(acc, round_dtype);
        }
}

/* Expert-choice combine: y[t] = sum over experts e (ascending) that chose t
 * of p[t,e] * O[tok_row[t,e],:]  +  sum_s Os[s,t,:]. O is [E*C,d]. */
void oracle_combine_expert_choice(int T, int d, int E, int S, const int32_t* tok_row,
                                  const float* p, const double* O, const double* Os,
                                  int round_dtype, double* y) {
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int e = 0; e < E; ++e) {
                int r = tok_row[(size_t)t * E + e];
                if (r < 0) continue;
                acc += (double)p[(size_t)t * E + e] * O[(size_t)r * d + i];
            }
            for (int s2 = 0; s2 < S; ++s2) acc += Os[((size_t)s2 * T + t) * d + i];
            y[(size_t)t * d + i] = round_to(acc, round_dtype);
        }
}

/* -------------------------------------------------------------- statistics */

/* Load-balance statistics over the batch.
 *   f[e] = (assignments routed to e, before capacity) / (T k)
 *   P[e] = mean over tokens of p[t,e]
 *   aux  = E * sum_e f[e] P[e]                        (Switch aux loss)
 *   I[e] = sum over tokens of the sparse gate G(x)_e  (Importance)
 *   cv2  = (population std of I / mean of I)^2,  L_imp = w_imp * cv2
 * out3 = {aux, cv2, L_imp}. p is [T,E] float, w is [T,k] float. */
void oracle_aux_stats(int T, int E, int k, const float* p, const int32_t* ids, const float* w,
                      double w_imp, double* f, double* P, double* I, double* out3) {
    for (int e = 0; e < E; ++e) {
        f[e] = 0.0;
        P[e] = 0.0;
        I[e] = 0.0;
    }
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            f[e] += 1.0;
            I[e] += (double)w[(size_t)t * k + j];
        }
        for (int e = 0; e < E; ++e) P[e] += (double)p[(size_t)t * E + e];
    }
    double aux = 0.0, mean = 0.0;
    for (int e = 0; e < E; ++e) {
        f[e] /= (double)T * (double)k;
        P[e] /= (double)T;
        aux += f[e] * P[e];
        mean += I[e];
    }
    aux *= (double)E;
    mean /= (double)E;
    double var = 0.0;
    for (int e = 0; e < E; ++e) var += (I[e] - mean) * (I[e] - mean);
    var /= (double)E;
    double cv2 = var / (mean * mean);
    out3[0] = aux;
    out3[1] = cv2;
    out3[2] = w_imp * cv2;
}

/* Sequence-level balance statistics: the Switch aux loss of the batch,
 * taken inside each sequence. Sequence q holds tokens seq_offsets[q] ..
 * seq_offsets[q+1]-1 (T_q of them):
 *   f[q,e]  = (top-k choices of its tokens naming e) / (T_q k)
 *   P[q,e]  = mean over its tokens of p[t,e]
 *   aux[q]  = E * sum_e f[q,e] P[q,e]
 *   mean    = mean of aux[q] over the non-empty sequences (0 if none)
 * An empty sequence has f = P = aux = 0. ids has `stride` columns per token;
 * its first k are the top-k choice. */
void oracle_seq_aux_stats(int E, int k, int stride, const float* p, const int32_t* ids,
                          int n_seq, const int32_t* seq_offsets, double* f, double* P,
                          double* aux, double* mean) {
    double total = 0.0;
    int nonempty = 0;
    for (int q = 0; q < n_seq; ++q) {
        int t0 = seq_offsets[q], t1 = seq_offsets[q + 1];
        double* fq = f + (size_t)q * E;
        double* Pq = P + (size_t)q * E;
        for (int e = 0; e < E; ++e) {
            fq[e] = 0.0;
            Pq[e] = 0.0;
        }
        aux[q] = 0.0;
        if (t1 <= t0) continue;
        for (int t = t0; t < t1; ++t) {
            for (int j = 0; j < k; ++j) fq[ids[(size_t)t * stride + j]] += 1.0;
            for (int e = 0; e < E; ++e) Pq[e] += (double)p[(size_t)t * E + e];
        }
        double a = 0.0;
        for (int e = 0; e < E; ++e) {
            fq[e] /= (double)(t1 - t0) * (double)k;
            Pq[e] /= (double)(t1 - t0);
            a += fq[e] * Pq[e];
        }
        aux[q] = (double)E * a;
        total += aux[q];
        nonempty += 1;
    }
    *mean = nonempty ? total / nonempty : 0.0;
}

/* Loss-free balance: bias[e] -= rate when expert e took more than the mean
 * load T k / E, += rate when it took less, unchanged at the mean. fp32. */
void oracle_bias_update(int E, int T, int k, const int32_t* counts, float rate, float* bias) {
    for (int e = 0; e < E; ++e) {
        long long diff = (long long)counts[e] * E - (long long)T * k;
        float b = bias[e];
        if (diff > 0) b = b - rate;
        if (diff < 0) b = b + rate;
        bias[e] = b;
    }
}
