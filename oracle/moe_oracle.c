/*
 * moe_oracle.c -- plain fp64 CPU oracle of the MegaMoE expert path.
 *
 * TEST INFRASTRUCTURE ONLY. The only code allowed to load or run this library
 * is tests/, __graft_entry__.smoke() and the cpu_baseline / reference legs of
 * bench.py. The product library (libmoe) never links, loads or calls it, and
 * the two share no source: no headers, helpers, tables or constants.
 *
 * What it computes. The MegaMoE guide (opening section "MegaMoE") describes
 * the expert path as a fused router (score function, group-limited top-k and
 * an aux load-balance score) followed by dispatch -> L1 grouped GEMM ->
 * SwiGLU -> L2 grouped GEMM -> top-k-weighted combine. Its section "Design:
 * two stages + weight modules" fixes the weight shapes: w1 [g, 2I, H] holding
 * the gate rows then the up rows, and w2 [g, H, I]. The SwiGLU is
 * silu(gate) * up, the form named in the "GDN <-> FLA Parity in Primus" page,
 * section B (Megatron-LM behavioural patches, the fla_swiglu row).
 *
 * With one device, dispatch and combine are a gather and a weighted sum, so
 * the exact result has a plain per-token definition:
 *
 *     y_t = sum_{e in K_t} w_{t,e} * W2_e ( silu(W1g_e x_t) (.) (W1u_e x_t) )
 *
 * This file evaluates exactly that, token by token, in double, from the exact
 * values of the bf16 / fp32 inputs. It uses no permutation, no tiling, no
 * blocking and no reordering of the arithmetic beyond the definition.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - the gate is rows [0, I) of w1[e] and the up projection rows [I, 2I);
 *   - top-k ties go to the lower expert index, group ties to the lower group;
 *   - the selection bias (sel_bias) enters only the selection and the group
 *     scores, never the weights;
 *   - aux = E * sum_e f_e * P_e with f_e = c_e / (T k) and
 *     P_e = (1/T) sum_t s_{t,e} over the full score vector.
 *
 * Parity status: every exported function is pinned by tests that do not call
 * its own formula again: closed forms of hand-built examples, the even
 * round-robin routing of the guide's force-load-balancing table, a dense
 * SwiGLU MLP in an independent library, brute force and invariants for the
 * forward; torch fp64 autograd through an independently written forward for
 * the backward. The aux value for sigmoid scoring has no pin beyond its
 * definition: parity unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact value of a bf16 bit pattern: the top 16 bits of an IEEE float. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Index of the largest v[i] among i in [0, n) with ok[i] != 0; on equal values
 * the lower index wins (scan in ascending order with a strict comparison).
 * Returns -1 when no index is eligible.
 */
static int64_t argmax_eligible(const double *v, const unsigned char *ok, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (!ok[i]) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best;
}

/*
 * Scores of one token: l_e = sum_h x_h Wr[e,h] (+ logit_offset[e]), then
 * s = softmax(l) over all E experts (score_fn 0) or sigmoid(l) (score_fn 1).
 */
static void token_scores(int64_t H, int64_t E, const uint16_t *x_t, const float *w_r,
                         const float *logit_offset, int32_t score_fn, double *s) {
    for (int64_t e = 0; e < E; ++e) {
        double l = 0.0;
        for (int64_t h = 0; h < H; ++h) l += bf16_value(x_t[h]) * (double)w_r[e * H + h];
        if (logit_offset) l += (double)logit_offset[e];
        s[e] = l;
    }
    if (score_fn == 0) {
        double m = s[0];
        for (int64_t e = 1; e < E; ++e) if (s[e] > m) m = s[e];
        double z = 0.0;
        for (int64_t e = 0; e < E; ++e) { s[e] = exp(s[e] - m); z += s[e]; }
        for (int64_t e = 0; e < E; ++e) s[e] /= z;
    } else {
        for (int64_t e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-s[e]));
    }
}

/*
 * Router for one token (MegaMoE opening section: "score function +
 * group-limited top-k + aux score").
 *
 *   l_e   = sum_h x_h * Wr[e,h]  (+ logit_offset[e] when given)
 *   s     = softmax(l) (score_fn 0) or sigmoid(l) elementwise (score_fn 1)
 *   sel_e = s_e + sel_bias[e]    (bias only steers the selection)
 *   with n_group > 1: group g holds experts [g*E/n_group, (g+1)*E/n_group);
 *     its score is the sum of its group_topn largest sel values; the
 *     topk_group best groups stay eligible, the rest are masked out
 *   K     = the k eligible experts with the largest sel, best first
 *   w_j   = s_{K_j}, divided by sum_j s_{K_j} when normalize, times scale
 *
 * sel_gap is sel of the k-th choice minus sel of the best unchosen eligible
 * expert (+inf when none is left); group_gap is the same for groups.
 */
static void route_one_token(int64_t H, int64_t E, int32_t k,
                            const uint16_t *x_t, const float *w_r,
                            const float *logit_offset, const float *sel_bias,
                            int32_t score_fn, int32_t normalize, double scale,
                            int32_t n_group, int32_t topk_group, int32_t group_topn,
                            double *s, double *sel, double *gscore,
                            unsigned char *ok, unsigned char *gok,
                            int32_t *idx_out, double *w_out,
                            double *sel_gap_out, double *group_gap_out) {
    token_scores(H, E, x_t, w_r, logit_offset, score_fn, s);
    for (int64_t e = 0; e < E; ++e) sel[e] = s[e] + (sel_bias ? (double)sel_bias[e] : 0.0);

    /* group limit */
    for (int64_t e = 0; e < E; ++e) ok[e] = 1;
    double group_gap = INFINITY;
    if (n_group > 1) {
        int64_t gs = E / n_group;
        for (int32_t g = 0; g < n_group; ++g) {
            /* sum of the group_topn largest sel values of group g */
            unsigned char *left = ok + g * gs; /* reused as scratch, reset below */
            double sum = 0.0;
            for (int32_t n = 0; n < group_topn && n < gs; ++n) {
                int64_t b = argmax_eligible(sel + g * gs, left, gs);
                sum += sel[g * gs + b];
                left[b] = 0;
            }
            for (int64_t i = 0; i < gs; ++i) left[i] = 1;
            gscore[g] = sum;
        }
        for (int32_t g = 0; g < n_group; ++g) gok[g] = 1;
        unsigned char kept[1024];
        for (int32_t g = 0; g < n_group; ++g) kept[g] = 0;
        for (int32_t n = 0; n < topk_group; ++n) {
            int64_t b = argmax_eligible(gscore, gok, n_group);
            kept[b] = 1;
            gok[b] = 0;
        }
        int64_t nb = argmax_eligible(gscore, gok, n_group);
        if (nb >= 0) {
            double worst_kept = INFINITY;
            for (int32_t g = 0; g < n_group; ++g)
                if (kept[g] && gscore[g] < worst_kept) worst_kept = gscore[g];
            group_gap = worst_kept - gscore[nb];
        }
        for (int64_t e = 0; e < E; ++e) ok[e] = kept[e / gs];
    }

    /* top-k of sel among the eligible experts */
    double chosen_sum = 0.0;
    for (int32_t j = 0; j < k; ++j) {
        int64_t b = argmax_eligible(sel, ok, E);
        idx_out[j] = (int32_t)b;
        ok[b] = 0;
        w_out[j] = s[b];
        chosen_sum += s[b];
    }
    int64_t next = argmax_eligible(sel, ok, E);
    double sel_gap = INFINITY;
    if (next >= 0) sel_gap = sel[idx_out[k - 1]] - sel[next];
    for (int32_t j = 0; j < k; ++j) {
        if (normalize) w_out[j] /= chosen_sum;
        w_out[j] *= scale;
    }
    if (sel_gap_out) *sel_gap_out = sel_gap;
    if (group_gap_out) *group_gap_out = group_gap;
}

/*
 * Router over T tokens, plus the aux load-balance value (MegaMoE opening
 * section: the aux loss is computed internally and returned; section
 * "Configuration": only the standard aux loss is supported).
 *
 *   aux = E * sum_e (c_e / (T k)) * ((1/T) sum_t s_{t,e})
 *
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_router(int64_t T, int64_t H, int64_t E, int32_t k,
                  const uint16_t *x, const float *w_r,
                  const float *logit_offset, const float *sel_bias,
                  int32_t score_fn, int32_t normalize, double scale,
                  int32_t n_group, int32_t topk_group, int32_t group_topn,
                  int32_t *topk_idx, double *topk_w,
                  double *scores, double *sel_gap, double *group_gap,
                  double *aux) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || !x || !w_r || !topk_idx || !topk_w)
        return -1;
    if (n_group > 1 && (E % n_group != 0 || topk_group <= 0 || topk_group > n_group ||
                        n_group > 1024 || group_topn <= 0))
        return -1;
    if (n_group > 1 && (int64_t)topk_group * (E / n_group) < k) return -1;

    double *all_s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * (size_t)E);
    if (!all_s) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *sel = (double *)malloc(sizeof(double) * (size_t)E);
        double *gscore = (double *)malloc(sizeof(double) * 1024);
        unsigned char *ok = (unsigned char *)malloc((size_t)E);
        unsigned char *gok = (unsigned char *)malloc(1024);
        if (!sel || !gscore || !ok || !gok) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < T; ++t) {
                route_one_token(H, E, k, x + t * H, w_r, logit_offset, sel_bias,
                                score_fn, normalize, scale, n_group, topk_group, group_topn,
                                all_s + t * E, sel, gscore, ok, gok,
                                topk_idx + t * k, topk_w + t * k,
                                sel_gap ? sel_gap + t : NULL, group_gap ? group_gap + t : NULL);
            }
        }
        free(sel); free(gscore); free(ok); free(gok);
    }
    if (bad) { free(all_s); return -1; }

    if (scores) memcpy(scores, all_s, sizeof(double) * (size_t)T * (size_t)E);
    if (aux) {
        double a = 0.0;
        for (int64_t e = 0; e < E; ++e) {
            int64_t c = 0;
            for (int64_t i = 0; i < T * k; ++i) if (topk_idx[i] == e) ++c;
            double p = 0.0;
            for (int64_t t = 0; t < T; ++t) p += all_s[t * E + e];
            double f = (T > 0) ? (double)c / ((double)T * (double)k) : 0.0;
            double P = (T > 0) ? p / (double)T : 0.0;
            a += f * P;
        }
        *aux = (double)E * a;
    }
    free(all_s);
    return 0;
}

/*
 * Routing metadata for one device (expert parallelism 1): the local stand-in
 * for the dispatch all-to-all (MegaMoE opening section, dispatch_grouped_gemm).
 *
 *   counts[e]     number of slots (t, j) with topk_idx[t*k + j] == e
 *   offsets[e]    exclusive prefix sum of counts; offsets[E] = routed rows
 *   perm_slot[r]  flat slot index t*k + j of routed row r; rows of expert e
 *                 are offsets[e] .. offsets[e+1]-1 in increasing slot order
 *   row_of[s]     routed row of slot s, or -1 if its index is outside [0, E)
 *
 * Written as a direct scan per expert so that stability is evident.
 * Returns the number of slots dropped for an out-of-range index.
 */
int64_t oracle_routing_metadata(int64_t T, int32_t k, int64_t E, const int32_t *topk_idx,
                                int32_t *counts, int32_t *offsets,
                                int32_t *perm_slot, int32_t *row_of) {
    int64_t R = T * k;
    int64_t dropped = 0;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t s = 0; s < R; ++s) {
        int32_t e = topk_idx[s];
        if (e >= 0 && e < E) counts[e] += 1; else ++dropped;
        row_of[s] = -1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int64_t e = 0; e < E; ++e) {
        int32_t r = offsets[e];
        for (int64_t s = 0; s < R; ++s) {
            if (topk_idx[s] != e) continue;
            perm_slot[r] = (int32_t)s;
            row_of[s] = r;
            ++r;
        }
    }
    return dropped;
}

/*
 * One slot of expert e, given the token's values xt [H]:
 *   g_i = sum_h W1[i, h] x_h        (gate rows [0, I))
 *   u_i = sum_h W1[I + i, h] x_h    (up rows [I, 2I))
 *   a_i = silu(g_i) * u_i
 */
static void slot_hidden(int64_t H, int64_t I, const uint16_t *W1, const double *xt,
                        double *g, double *u, double *a) {
    for (int64_t i = 0; i < I; ++i) {
        double gi = 0.0, ui = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            gi += bf16_value(W1[i * H + h]) * xt[h];
            ui += bf16_value(W1[(I + i) * H + h]) * xt[h];
        }
        g[i] = gi;
        u[i] = ui;
        a[i] = silu(gi) * ui;
    }
}

/* o_h = sum_i W2[h, i] a_i for one slot. */
static void slot_output(int64_t H, int64_t I, const uint16_t *W2, const double *a, double *o) {
    for (int64_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i) acc += bf16_value(W2[h * I + i]) * a[i];
        o[h] = acc;
    }
}

/*
 * Expert path forward, token by token (MegaMoE opening section:
 * dispatch_grouped_gemm -> SwiGLU -> grouped_gemm_combine).
 *
 *   for each token t and choice j with e = topk_idx[t,j] in [0, E):
 *     g_i = sum_h w1[e, i, h]     x[t, h]        i in [0, I)   (gate rows)
 *     u_i = sum_h w1[e, I + i, h] x[t, h]                      (up rows)
 *     a_i = silu(g_i) * u_i
 *     o_h = sum_i w2[e, h, i] a_i
 *     y[t, h] += topk_w[t, j] * o_h
 *
 * Slots with an index outside [0, E) contribute nothing. a_slot, when given,
 * receives a for every slot in flat slot order [T*k, I] (zero for dropped
 * slots); o_slot likewise receives the unweighted o rows [T*k, H].
 */
int oracle_expert_forward(int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                          const uint16_t *x, const int32_t *topk_idx, const double *topk_w,
                          const uint16_t *w1, const uint16_t *w2,
                          double *y, double *a_slot, double *o_slot) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || !x || !topk_idx || !topk_w ||
        !w1 || !w2 || !y)
        return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *a = (double *)malloc(sizeof(double) * (size_t)I);
        double *o = (double *)malloc(sizeof(double) * (size_t)H);
        if (!xt || !g || !u || !a || !o) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < T; ++t) {
                double *yt = y + t * H;
                for (int64_t h = 0; h < H; ++h) { yt[h] = 0.0; xt[h] = bf16_value(x[t * H + h]); }
                for (int32_t j = 0; j < k; ++j) {
                    int64_t slot = t * k + j;
                    int32_t e = topk_idx[slot];
                    if (e < 0 || e >= E) {
                        if (a_slot) for (int64_t i = 0; i < I; ++i) a_slot[slot * I + i] = 0.0;
                        if (o_slot) for (int64_t h = 0; h < H; ++h) o_slot[slot * H + h] = 0.0;
                        continue;
                    }
                    const uint16_t *W1 = w1 + (int64_t)e * 2 * I * H;
                    const uint16_t *W2 = w2 + (int64_t)e * H * I;
                    slot_hidden(H, I, W1, xt, g, u, a);
                    slot_output(H, I, W2, a, o);
                    if (a_slot) for (int64_t i = 0; i < I; ++i) a_slot[slot * I + i] = a[i];
                    if (o_slot) for (int64_t h = 0; h < H; ++h) o_slot[slot * H + h] = o[h];
                    double w = topk_w[slot];
                    for (int64_t h = 0; h < H; ++h) yt[h] += w * o[h];
                }
            }
        }
        free(xt); free(g); free(u); free(a); free(o);
    }
    return bad ? -1 : 0;
}

/*
 * Expert path backward, from its plain chain rule (MegaMoE guide, section
 * "Design: two stages": stage 2's backward yields dW2, stage 1's dW1). With
 * dY the gradient of y, for each token t and choice j with e = topk_idx[t,j]:
 *
 *   forward values  g, u, a = silu(g) * u, o = W2_e a      (as in the forward)
 *   dw[t,j]   = <dY_t, o>                  gradient of the routing weight
 *   dO        = w[t,j] dY_t
 *   dA_i      = sum_h W2_e[h,i] dO_h
 *   dU_i      = dA_i silu(g_i)
 *   dG_i      = dA_i u_i silu'(g_i),   silu'(z) = s(z) (1 + z (1 - s(z))), s = sigmoid
 *   dX_t     += sum_i W1_e[i,:] dG_i + W1_e[I+i,:] dU_i
 *   dW1_e[i,:]   += dG_i x_t ;  dW1_e[I+i,:] += dU_i x_t
 *   dW2_e[:,i]   += dO a_i
 *
 * dw1 [E,2I,H], dw2 [E,H,I], dx [T,H] and dtopk_w [T,k] are outputs (any may
 * be NULL except dx). The weight gradients are accumulated per expert over its
 * slots in flat slot order. Slots with an index outside [0, E) contribute
 * nothing (their dtopk_w is 0).
 */
/*
 * The data-gradient path of one slot of expert e, given the slot's g, u and
 * a = silu(g) u (bf16 weights W1 = w1[e], W2 = w2[e]; the chain rule of the
 * forward above):
 *   o = W2 a,  dw = <dY_t, o>,  dO = w dY_t,  dA_i = sum_h W2[h,i] dO_h,
 *   dU_i = dA_i silu(g_i),  dG_i = dA_i u_i silu'(g_i),
 *   dX_t += sum_i W1[i,:] dG_i + W1[I+i,:] dU_i
 * dh receives [dG | dU] (2I values); o, dO, dA are scratch ([H], [H], [I]).
 * Returns dw.
 */
static double slot_data_gradient(int64_t H, int64_t I, const uint16_t *W1, const uint16_t *W2, double w,
                                 const double *dyt, const double *g, const double *u, const double *a,
                                 double *o, double *dO, double *dA, double *dxt, double *dh) {
    slot_output(H, I, W2, a, o);
    double dwt = 0.0;
    for (int64_t h = 0; h < H; ++h) {
        dwt += dyt[h] * o[h];
        dO[h] = w * dyt[h];
    }
    for (int64_t i = 0; i < I; ++i) {
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h) acc += bf16_value(W2[h * I + i]) * dO[h];
        dA[i] = acc;
    }
    for (int64_t i = 0; i < I; ++i) {
        const double sg = 1.0 / (1.0 + exp(-g[i]));
        const double dsilu = sg * (1.0 + g[i] * (1.0 - sg));
        const double dU = dA[i] * silu(g[i]);
        const double dG = dA[i] * u[i] * dsilu;
        for (int64_t h = 0; h < H; ++h)
            dxt[h] += bf16_value(W1[i * H + h]) * dG + bf16_value(W1[(I + i) * H + h]) * dU;
        dh[i] = dG;
        dh[I + i] = dU;
    }
    return dwt;
}

int oracle_expert_backward(int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                           const uint16_t *x, const int32_t *topk_idx, const double *topk_w,
                           const uint16_t *w1, const uint16_t *w2, const uint16_t *dy,
                           double *dx, double *dw1, double *dw2, double *dtopk_w) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || !x || !topk_idx || !topk_w || !w1 ||
        !w2 || !dy || !dx)
        return -1;
    const int64_t R = T * k;
    /* per-slot values kept for the weight gradients: dG|dU [R, 2I], dO [R, H], a [R, I] */
    double *dh_s = (dw1 || dw2) ? (double *)calloc((size_t)R * 2 * I, sizeof(double)) : NULL;
    double *do_s = dw2 ? (double *)calloc((size_t)R * H, sizeof(double)) : NULL;
    double *a_s = dw2 ? (double *)calloc((size_t)R * I, sizeof(double)) : NULL;
    if (((dw1 || dw2) && !dh_s) || (dw2 && (!do_s || !a_s))) {
        free(dh_s); free(do_s); free(a_s);
        return -1;
    }
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *dyt = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *a = (double *)malloc(sizeof(double) * (size_t)I);
        double *o = (double *)malloc(sizeof(double) * (size_t)H);
        double *dO = (double *)malloc(sizeof(double) * (size_t)H);
        double *dA = (double *)malloc(sizeof(double) * (size_t)I);
        double *dh = (double *)malloc(sizeof(double) * 2 * (size_t)I);
        if (!xt || !dyt || !g || !u || !a || !o || !dO || !dA || !dh) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < T; ++t) {
                double *dxt = dx + t * H;
                for (int64_t h = 0; h < H; ++h) {
                    dxt[h] = 0.0;
                    xt[h] = bf16_value(x[t * H + h]);
                    dyt[h] = bf16_value(dy[t * H + h]);
                }
                for (int32_t j = 0; j < k; ++j) {
                    const int64_t slot = t * k + j;
                    const int32_t e = topk_idx[slot];
                    if (e < 0 || e >= E) {
                        if (dtopk_w) dtopk_w[slot] = 0.0;
                        continue;
                    }
                    const uint16_t *W1 = w1 + (int64_t)e * 2 * I * H;
                    const uint16_t *W2 = w2 + (int64_t)e * H * I;
                    slot_hidden(H, I, W1, xt, g, u, a);
                    const double w = topk_w[slot];
                    const double dwt = slot_data_gradient(H, I, W1, W2, w, dyt, g, u, a, o, dO, dA, dxt, dh);
                    if (dtopk_w) dtopk_w[slot] = dwt;
                    if (dh_s) memcpy(dh_s + slot * 2 * I, dh, sizeof(double) * 2 * (size_t)I);
                    if (do_s) {
                        for (int64_t h = 0; h < H; ++h) do_s[slot * H + h] = dO[h];
                        for (int64_t i = 0; i < I; ++i) a_s[slot * I + i] = a[i];
                    }
                }
            }
        }
        free(xt); free(dyt); free(g); free(u); free(a); free(o); free(dO); free(dA); free(dh);
    }
    if (!bad && (dw1 || dw2)) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t e = 0; e < E; ++e) {
            double *DW1 = dw1 ? dw1 + e * 2 * I * H : NULL;
            double *DW2 = dw2 ? dw2 + e * H * I : NULL;
            if (DW1) for (int64_t q = 0; q < 2 * I * H; ++q) DW1[q] = 0.0;
            if (DW2) for (int64_t q = 0; q < H * I; ++q) DW2[q] = 0.0;
            for (int64_t slot = 0; slot < R; ++slot) {
                if (topk_idx[slot] != e) continue;
                const int64_t t = slot / k;
                if (DW1) {
                    for (int64_t jj = 0; jj < 2 * I; ++jj) {
                        const double d = dh_s[slot * 2 * I + jj];
                        for (int64_t h = 0; h < H; ++h) DW1[jj * H + h] += d * bf16_value(x[t * H + h]);
                    }
                }
                if (DW2) {
                    for (int64_t h = 0; h < H; ++h) {
                        const double d = do_s[slot * H + h];
                        for (int64_t i = 0; i < I; ++i) DW2[h * I + i] += d * a_s[slot * I + i];
                    }
                }
            }
        }
    }
    free(dh_s); free(do_s); free(a_s);
    return bad ? -1 : 0;
}

/*
 * Router backward: the gradient of the logits from the gradient of the
 * routing weights, then dX and dW_r through l = x W_r^T (+ offset). The
 * selection (top-k, groups, bias) is piecewise constant and passes no
 * gradient; the aux value is reported, not differentiated. With K the chosen
 * experts of a token and p = the score function:
 *
 *   softmax, normalised:   w_j = scale e^{l_j} / sum_K e^l
 *                          dl_i = w_i dw_i - (w_i / scale) sum_K w_j dw_j   (i in K)
 *   softmax, plain:        w_j = scale s_j,  s = softmax over all E
 *                          dl_i = scale s_i ([i in K] dw_i - sum_K s_j dw_j)
 *   sigmoid, normalised:   w_j = scale s_j / S,  S = sum_K s
 *                          dl_i = (s_i (1 - s_i) / S) (scale dw_i - sum_K w_j dw_j)   (i in K)
 *   sigmoid, plain:        dl_i = scale s_i (1 - s_i) dw_i   (i in K)
 *
 *   dX_t += sum_e dl_{t,e} W_r[e,:]      dW_r[e,:] = sum_t dl_{t,e} x_t
 *
 * dlogits [T,E] (zero outside K for the normalised cases), dx_add [T,H] (added
 * to, not overwritten) and dw_r [E,H] are outputs; any may be NULL.
 */
int oracle_router_backward(int64_t T, int64_t H, int64_t E, int32_t k,
                           const uint16_t *x, const float *w_r, const float *logit_offset,
                           int32_t score_fn, int32_t normalize, double scale,
                           const int32_t *topk_idx, const double *topk_w, const double *dtopk_w,
                           double *dlogits, double *dx_add, double *dw_r) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || !x || !w_r || !topk_idx || !topk_w || !dtopk_w)
        return -1;
    double *dl = (double *)calloc((size_t)(T > 0 ? T : 1) * (size_t)E, sizeof(double));
    if (!dl) return -1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        double *dlt = dl + t * E;
        const int32_t *K = topk_idx + t * k;
        const double *w = topk_w + t * k;
        const double *dw = dtopk_w + t * k;
        /* scores of the token (needed by the plain softmax and the sigmoid cases) */
        double *s = (double *)malloc(sizeof(double) * (size_t)E);
        if (!s) continue;
        token_scores(H, E, x + t * H, w_r, logit_offset, score_fn, s);
        double sum_wdw = 0.0, sum_sdw = 0.0, S = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            if (K[j] < 0 || K[j] >= E) continue;
            sum_wdw += w[j] * dw[j];
            sum_sdw += s[K[j]] * dw[j];
            S += s[K[j]];
        }
        if (score_fn == 0 && normalize) {
            for (int32_t j = 0; j < k; ++j)
                if (K[j] >= 0 && K[j] < E) dlt[K[j]] += w[j] * dw[j] - (w[j] / scale) * sum_wdw;
        } else if (score_fn == 0) {
            for (int64_t e = 0; e < E; ++e) dlt[e] = -scale * s[e] * sum_sdw;
            for (int32_t j = 0; j < k; ++j)
                if (K[j] >= 0 && K[j] < E) dlt[K[j]] += scale * s[K[j]] * dw[j];
        } else if (normalize) {
            for (int32_t j = 0; j < k; ++j) {
                if (K[j] < 0 || K[j] >= E) continue;
                const double si = s[K[j]];
                dlt[K[j]] += si * (1.0 - si) / S * (scale * dw[j] - sum_wdw);
            }
        } else {
            for (int32_t j = 0; j < k; ++j) {
                if (K[j] < 0 || K[j] >= E) continue;
                const double si = s[K[j]];
                dlt[K[j]] += scale * si * (1.0 - si) * dw[j];
            }
        }
        if (dx_add)
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t e = 0; e < E; ++e) acc += dlt[e] * (double)w_r[e * H + h];
                dx_add[t * H + h] += acc;
            }
        free(s);
    }
    if (dw_r) {
#pragma omp parallel for schedule(static)
        for (int64_t e = 0; e < E; ++e)
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t) acc += dl[t * E + e] * bf16_value(x[t * H + h]);
                dw_r[e * H + h] = acc;
            }
    }
    if (dlogits) memcpy(dlogits, dl, sizeof(double) * (size_t)T * (size_t)E);
    free(dl);
    return 0;
}

/*
 * ------------------------------------------------------------------ MXFP8
 *
 * The guide's second expert precision (section "Expert precision": mxfp8 runs
 * the two expert stages in MXFP8). MXFP8 is the Open Compute Project
 * Microscaling format (OCP MX v1.0): blocks of 32 consecutive elements along
 * the reduction dimension share one power-of-two scale X stored as E8M0
 * (biased exponent, bias 127); the elements are FP8 E4M3 (bias 7, no infinity,
 * largest finite 448 = 1.75 * 2^8). Per the spec the shared exponent is
 * floor(log2(max |v|)) - emax with emax = 8 for E4M3, and each element is
 * v / X converted to E4M3, here with round-to-nearest-even and saturation to
 * +-448, keeping the sign of zero as IEEE-754 conversions do. A block of zeros
 * gets the smallest scale, 2^-127 (code 0).
 */

/* Value of an E4M3 code (finite codes only; 0x7F / 0xFF are NaN). */
static double e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    const double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E4M3 code of q, rounded to nearest (ties to even) and saturated. */
static uint8_t e4m3_encode(double q) {
    const uint8_t sign = signbit(q) ? 0x80 : 0x00;      /* -0 keeps its sign, as in IEEE conversions */
    double a = fabs(q);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                 /* subnormals: m * 2^-9 */
        const double m = rint(a * 512.0);     /* 8 -> the smallest normal, code 0x08 */
        return sign | (uint8_t)m;
    }
    int p;
    frexp(a, &p);                             /* a = f 2^p, f in [0.5, 1) */
    p -= 1;                                   /* a in [2^p, 2^(p+1)) */
    const double m = rint((ldexp(a, -p) - 1.0) * 8.0);   /* 0..8 */
    int code = ((p + 7) << 3) + (int)m;       /* m = 8 carries into the exponent */
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* E8M0 scale code of a block whose largest magnitude is amax. */
static uint8_t mx_scale_code(double amax) {
    if (amax == 0.0) return 0;
    int p;
    frexp(amax, &p);
    int e = (p - 1) - 8;                      /* floor(log2 amax) - emax(E4M3) */
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

static double e8m0_value(uint8_t s) { return ldexp(1.0, (int)s - 127); }

/*
 * Quantize a [rows, cols] matrix (cols a multiple of 32) to MXFP8 along its
 * rows: codes [rows, cols], scales [rows, cols / 32]. Input as bf16 bit
 * patterns (in_bf16) or doubles (in_f64); exactly one of them is non-NULL.
 */
/* One block of 32 values: its E8M0 scale code, and each value's E4M3 code. */
static uint8_t mx_quantize_block(const double *v, uint8_t *codes) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i)
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    const uint8_t s = mx_scale_code(amax);
    for (int i = 0; i < 32; ++i) codes[i] = e4m3_encode(v[i] / e8m0_value(s));
    return s;
}

static void mx_quantize_rows(int64_t rows, int64_t cols, const uint16_t *in_bf16, const double *in_f64,
                             uint8_t *codes, uint8_t *scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < cols / 32; ++b) {
            double v[32];
            for (int i = 0; i < 32; ++i) {
                const int64_t j = r * cols + b * 32 + i;
                v[i] = in_bf16 ? bf16_value(in_bf16[j]) : in_f64[j];
            }
            scales[r * (cols / 32) + b] = mx_quantize_block(v, codes + r * cols + b * 32);
        }
    }
}

int oracle_mx_quantize_bf16(int64_t rows, int64_t cols, const uint16_t *in, uint8_t *codes, uint8_t *scales) {
    if (rows < 0 || cols <= 0 || cols % 32 != 0 || !in || !codes || !scales) return -1;
    mx_quantize_rows(rows, cols, in, NULL, codes, scales);
    return 0;
}

int oracle_mx_quantize_f64(int64_t rows, int64_t cols, const double *in, uint8_t *codes, uint8_t *scales) {
    if (rows < 0 || cols <= 0 || cols % 32 != 0 || !in || !codes || !scales) return -1;
    mx_quantize_rows(rows, cols, NULL, in, codes, scales);
    return 0;
}

/* v = code value * scale value, for a quantized [rows, cols] matrix. */
static double mx_value(const uint8_t *codes, const uint8_t *scales, int64_t cols, int64_t r, int64_t c) {
    return e4m3_value(codes[r * cols + c]) * e8m0_value(scales[r * (cols / 32) + c / 32]);
}

/*
 * Expert path forward in MXFP8 (the guide's mxfp8 expert precision): x, w1 and
 * w2 are given quantized along their reduction dimension (x, w1 along H; w2
 * along I). For each token t and choice j with e = topk_idx[t,j] in [0, E):
 *
 *   g_i, u_i = sum_h X(x)[t,h] X(w1)[e, i or I+i, h]       (exact, in double)
 *   a_i      = silu(g_i) u_i
 *   a_q      = MXFP8 quantization of a along I (blocks of 32)
 *   o_h      = sum_i X(a_q)_i X(w2)[e,h,i]
 *   y[t,:]  += topk_w[t,j] o
 *
 * X() is the dequantized value (code value times block scale). a_pre, when
 * given, receives a before quantization per slot [T*k, I]; a_codes / a_scales
 * its quantization [T*k, I] / [T*k, I/32] (zero for dropped slots).
 */
int oracle_expert_forward_mx(int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                             const uint8_t *x_codes, const uint8_t *x_scales,
                             const int32_t *topk_idx, const double *topk_w,
                             const uint8_t *w1_codes, const uint8_t *w1_scales,
                             const uint8_t *w2_codes, const uint8_t *w2_scales,
                             double *y, double *a_pre, uint8_t *a_codes, uint8_t *a_scales) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || H % 32 || I % 32 || !x_codes || !x_scales ||
        !topk_idx || !topk_w || !w1_codes || !w1_scales || !w2_codes || !w2_scales || !y)
        return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *a = (double *)malloc(sizeof(double) * (size_t)I);
        double *aq = (double *)malloc(sizeof(double) * (size_t)I);
        uint8_t *ac = (uint8_t *)malloc((size_t)I);
        uint8_t *as = (uint8_t *)malloc((size_t)(I / 32));
        if (!xt || !a || !aq || !ac || !as) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < T; ++t) {
                double *yt = y + t * H;
                for (int64_t h = 0; h < H; ++h) { yt[h] = 0.0; xt[h] = mx_value(x_codes, x_scales, H, t, h); }
                for (int32_t j = 0; j < k; ++j) {
                    const int64_t slot = t * k + j;
                    const int32_t e = topk_idx[slot];
                    if (e < 0 || e >= E) {
                        if (a_pre) for (int64_t i = 0; i < I; ++i) a_pre[slot * I + i] = 0.0;
                        if (a_codes) memset(a_codes + slot * I, 0, (size_t)I);
                        if (a_scales) memset(a_scales + slot * (I / 32), 0, (size_t)(I / 32));
                        continue;
                    }
                    const int64_t r1 = (int64_t)e * 2 * I;      /* first w1 row of expert e */
                    for (int64_t i = 0; i < I; ++i) {
                        double g = 0.0, u = 0.0;
                        for (int64_t h = 0; h < H; ++h) {
                            g += mx_value(w1_codes, w1_scales, H, r1 + i, h) * xt[h];
                            u += mx_value(w1_codes, w1_scales, H, r1 + I + i, h) * xt[h];
                        }
                        a[i] = silu(g) * u;
                    }
                    mx_quantize_rows(1, I, NULL, a, ac, as);
                    for (int64_t i = 0; i < I; ++i) aq[i] = e4m3_value(ac[i]) * e8m0_value(as[i / 32]);
                    if (a_pre) for (int64_t i = 0; i < I; ++i) a_pre[slot * I + i] = a[i];
                    if (a_codes) memcpy(a_codes + slot * I, ac, (size_t)I);
                    if (a_scales) memcpy(a_scales + slot * (I / 32), as, (size_t)(I / 32));
                    const int64_t r2 = (int64_t)e * H;           /* first w2 row of expert e */
                    const double w = topk_w[slot];
                    for (int64_t h = 0; h < H; ++h) {
                        double o = 0.0;
                        for (int64_t i = 0; i < I; ++i) o += mx_value(w2_codes, w2_scales, I, r2 + h, i) * aq[i];
                        yt[h] += w * o;
                    }
                }
            }
        }
        free(xt); free(a); free(aq); free(ac); free(as);
    }
    return bad ? -1 : 0;
}

/*
 * MXFP8 quantization of one block of 32 values along the block, returned as
 * their dequantized values (code value times block scale): the same rule as
 * mx_quantize_rows, for a block gathered from a column.
 */
static void mx_block_values(const double *v, double *q) {
    uint8_t c[32];
    const uint8_t s = mx_quantize_block(v, c);
    for (int i = 0; i < 32; ++i) q[i] = e4m3_value(c[i]) * e8m0_value(s);
}

/*
 * An MXFP8 weight gradient from given operands (the last step of the MXFP8
 * training backward below). A [R, M] and B [R, N] hold one row per routed row;
 * rows offsets[e] .. offsets[e+1]-1 belong to expert e. Per expert, its rows
 * are cut into blocks of 32 consecutive rows from its first row (a last,
 * partial block is completed with zeros), every column of A and of B is
 * quantized to MXFP8 per block, and
 *   dW[e][m][n] = sum over e's rows r of Q(A)[r,m] Q(B)[r,n]      dW [E, M, N]
 */
int oracle_mx_wgrad(int64_t E, const int32_t *offsets, int64_t M, int64_t N, const double *A, const double *B,
                    double *dW) {
    if (E <= 0 || M <= 0 || N <= 0 || !offsets || !A || !B || !dW) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *col = (double *)malloc(sizeof(double) * 32);
        double *cq = (double *)malloc(sizeof(double) * 32);
        double *qa = (double *)malloc(sizeof(double) * 32 * (size_t)M);   /* a block of Q(A): [32][M] */
        double *qb = (double *)malloc(sizeof(double) * 32 * (size_t)N);
        if (!col || !cq || !qa || !qb) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t e = 0; e < E; ++e) {
                double *D = dW + e * M * N;
                for (int64_t q = 0; q < M * N; ++q) D[q] = 0.0;
                const int64_t end = offsets[e + 1];
                for (int64_t b0 = offsets[e]; b0 < end; b0 += 32) {
                    const int64_t n = (end - b0 < 32) ? end - b0 : 32;
                    /* per column: the block's values (zeros past the expert's rows),
                       quantized, kept dequantized */
                    for (int64_t m = 0; m < M; ++m) {
                        for (int r = 0; r < 32; ++r) col[r] = (r < n) ? A[(b0 + r) * M + m] : 0.0;
                        mx_block_values(col, cq);
                        for (int r = 0; r < 32; ++r) qa[r * M + m] = cq[r];
                    }
                    for (int64_t c = 0; c < N; ++c) {
                        for (int r = 0; r < 32; ++r) col[r] = (r < n) ? B[(b0 + r) * N + c] : 0.0;
                        mx_block_values(col, cq);
                        for (int r = 0; r < 32; ++r) qb[r * N + c] = cq[r];
                    }
                    for (int r = 0; r < 32; ++r)
                        for (int64_t m = 0; m < M; ++m) {
                            const double d = qa[r * M + m];
                            if (d == 0.0) continue;
                            for (int64_t c = 0; c < N; ++c) D[m * N + c] += d * qb[r * N + c];
                        }
                }
            }
        }
        free(col); free(cq); free(qa); free(qb);
    }
    return bad ? -1 : 0;
}

/*
 * Training backward of the MXFP8 expert precision (MegaMoE guide, section
 * "Expert precision": mxfp8 runs fc1, the SwiGLU, fc2 and the dW1 / dW2
 * weight gradients in MXFP8). Reading, where the pages name no more:
 *
 *   - The forward is that of oracle_expert_forward_mx: g, u from X(x) and
 *     X(w1) (quantized along H), a = silu(g) u.
 *   - The data-gradient path is the bf16 backward's (the pages list no MXFP8
 *     data gradients), taken at that forward's g and u with the bf16 weights;
 *     quantization passes the gradient through unchanged:
 *       dw[t,j] = <dY_t, W2_e a>,  dO = w dY_t,  dA = W2_e^T dO,
 *       dU = dA silu(g),  dG = dA u silu'(g),  dX_t += W1_e^T [dG ; dU].
 *   - The two weight gradients take MXFP8 operands quantized along their
 *     reduction dimension, the expert's routed rows: the rows of expert e are
 *     its slots in increasing flat slot order (the routed order), cut into
 *     blocks of 32 consecutive rows from its first row (a last, partial block
 *     is completed with zeros); every column of an operand is quantized per
 *     block. The routing weight is carried by the activation side, as the
 *     forward multiplies it onto fc2's output:
 *       dW2_e[h,i] = sum_r Q(dY)[r,h] Q(w a)[r,i]
 *       dW1_e[j,h] = sum_r Q(dH)[r,j] Q(x)[r,h],   dH = [dG | dU]
 *     with dY[r] and x[r] the rows of the slot's token.
 *
 * x, dy, w1, w2 are bf16 [T,H], [T,H], [E,2I,H], [E,H,I]; x_codes / x_scales
 * and w1_codes / w1_scales the forward's quantization of x and w1 (along H).
 * Outputs as in oracle_expert_backward; dh_slot [T*k, 2I] and wa_slot
 * [T*k, I], when given, receive dH and w a per slot in flat slot order (zero
 * for dropped slots), before quantization.
 */
int oracle_expert_backward_mx(int64_t T, int64_t H, int64_t I, int64_t E, int32_t k,
                              const uint16_t *x, const uint8_t *x_codes, const uint8_t *x_scales,
                              const int32_t *topk_idx, const double *topk_w,
                              const uint16_t *w1, const uint8_t *w1_codes, const uint8_t *w1_scales,
                              const uint16_t *w2, const uint16_t *dy,
                              double *dx, double *dw1, double *dw2, double *dtopk_w,
                              double *dh_slot, double *wa_slot) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || H % 32 || I % 32 || !x || !x_codes ||
        !x_scales || !topk_idx || !topk_w || !w1 || !w1_codes || !w1_scales || !w2 || !dy || !dx)
        return -1;
    const int64_t R = T * k;
    double *dh_s = (double *)calloc((size_t)(R > 0 ? R : 1) * 2 * I, sizeof(double));
    double *wa_s = (double *)calloc((size_t)(R > 0 ? R : 1) * I, sizeof(double));
    if (!dh_s || !wa_s) {
        free(dh_s); free(wa_s);
        return -1;
    }
    int bad = 0;
#pragma omp parallel
    {
        double *xq = (double *)malloc(sizeof(double) * (size_t)H);
        double *dyt = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *a = (double *)malloc(sizeof(double) * (size_t)I);
        double *o = (double *)malloc(sizeof(double) * (size_t)H);
        double *dO = (double *)malloc(sizeof(double) * (size_t)H);
        double *dA = (double *)malloc(sizeof(double) * (size_t)I);
        if (!xq || !dyt || !g || !u || !a || !o || !dO || !dA) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < T; ++t) {
                double *dxt = dx + t * H;
                for (int64_t h = 0; h < H; ++h) {
                    dxt[h] = 0.0;
                    xq[h] = mx_value(x_codes, x_scales, H, t, h);
                    dyt[h] = bf16_value(dy[t * H + h]);
                }
                for (int32_t j = 0; j < k; ++j) {
                    const int64_t slot = t * k + j;
                    const int32_t e = topk_idx[slot];
                    if (e < 0 || e >= E) {
                        if (dtopk_w) dtopk_w[slot] = 0.0;
                        continue;
                    }
                    /* the MXFP8 forward's pre-activation: X(x) and X(w1) along H */
                    const int64_t w1_row = (int64_t)e * 2 * I;
                    for (int64_t i = 0; i < I; ++i) {
                        double gacc = 0.0, uacc = 0.0;
                        for (int64_t h = 0; h < H; ++h) {
                            gacc += mx_value(w1_codes, w1_scales, H, w1_row + i, h) * xq[h];
                            uacc += mx_value(w1_codes, w1_scales, H, w1_row + I + i, h) * xq[h];
                        }
                        g[i] = gacc;
                        u[i] = uacc;
                    }
                    for (int64_t i = 0; i < I; ++i) a[i] = silu(g[i]) * u[i];
                    /* the data-gradient path, bf16 weights */
                    const double w = topk_w[slot];
                    const double dwt = slot_data_gradient(H, I, w1 + (int64_t)e * 2 * I * H, w2 + (int64_t)e * H * I,
                                                          w, dyt, g, u, a, o, dO, dA, dxt, dh_s + slot * 2 * I);
                    if (dtopk_w) dtopk_w[slot] = dwt;
                    for (int64_t i = 0; i < I; ++i) wa_s[slot * I + i] = w * a[i];
                }
            }
        }
        free(xq); free(dyt); free(g); free(u); free(a); free(o); free(dO); free(dA);
    }
    if (!bad && (dw1 || dw2)) {
        /* the weight gradients' operands, one row per routed row (the routing
           metadata's stable order: expert-major, slots in increasing order) */
        int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
        int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
        int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
        int32_t *row_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
        double *ady = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * (size_t)H);
        double *awa = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * (size_t)I);
        double *adh = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * 2 * (size_t)I);
        double *ax = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1) * (size_t)H);
        if (!counts || !offsets || !perm || !row_of || !ady || !awa || !adh || !ax) {
            bad = 1;
        } else {
            oracle_routing_metadata(T, k, E, topk_idx, counts, offsets, perm, row_of);
            const int64_t routed = offsets[E];
            for (int64_t r = 0; r < routed; ++r) {
                const int64_t slot = perm[r];
                const int64_t tok = slot / k;
                for (int64_t h = 0; h < H; ++h) {
                    ady[r * H + h] = bf16_value(dy[tok * H + h]);
                    ax[r * H + h] = bf16_value(x[tok * H + h]);
                }
                memcpy(awa + r * I, wa_s + slot * I, sizeof(double) * (size_t)I);
                memcpy(adh + r * 2 * I, dh_s + slot * 2 * I, sizeof(double) * 2 * (size_t)I);
            }
            if (dw2 && oracle_mx_wgrad(E, offsets, H, I, ady, awa, dw2) != 0) bad = 1;
            if (dw1 && oracle_mx_wgrad(E, offsets, 2 * I, H, adh, ax, dw1) != 0) bad = 1;
        }
        free(counts); free(offsets); free(perm); free(row_of); free(ady); free(awa); free(adh); free(ax);
    }
    if (!bad && dh_slot) memcpy(dh_slot, dh_s, sizeof(double) * (size_t)R * 2 * I);
    if (!bad && wa_slot) memcpy(wa_slot, wa_s, sizeof(double) * (size_t)R * I);
    free(dh_s); free(wa_s);
    return bad ? -1 : 0;
}
