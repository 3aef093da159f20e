/*
 * moe_oracle.c -- plain, slow CPU oracle for one mixture-of-experts layer
 * forward pass: route -> dispatch -> expert compute -> combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this file.  It shares no
 * code, header, table or helper with the CUDA library in
 * expert_dispatch_top_b300/csrc, and the CUDA library never calls it.
 *
 * The four steps follow the Ultralytics glossary page "Expert Parallelism",
 * section "How Tokens Move Between GPUs" (steps 1-4: Route, Dispatch,
 * Compute, Combine), and the ai360xpert page "Expert Parallelism", section
 * "The All-to-All Bottleneck" (Routing, Scatter, Compute, Gather).  On one
 * device both all-to-all exchanges become an on-device permutation into an
 * expert-major buffer whose contiguous expert blocks are the virtual
 * expert-parallel ranks (mbrenndoerfer.com "Expert Parallelism > Summary":
 * uniform placement; Ultralytics snippet: experts 0-1 on GPU 0, 2-3 on GPU 1).
 *
 * Arithmetic: every sum is an fp64 sum taken in index order, with no FMA
 * contraction (built with -ffp-contract=off) and no reassociation.  Where a
 * floating-point value decides an integer (the top-k selection), the value is
 * first brought to fp32, the precision the device path decides in:
 *   logit  L = fp32( sum_i x_i * w_i )  [+ fp32 logit bias, one fp32 add]
 *   softmax routers select on L (softmax is monotone in L);
 *   sigmoid routers select on fp32( 1 / (1 + exp(-L)) ) [+ selection bias,
 *   one fp32 add].
 * Inputs on the dyadic grid (x multiples of 1/8, weights multiples of 1/512,
 * d <= 8192) make every partial sum exact, so L does not depend on the order.
 *
 * Readings taken where the pages are silent:
 *   - ties in the selection key go to the lower expert index;
 *   - capacity C = ceil(cf * T * k / E) (Ultralytics "Load Balancing and
 *     Capacity": a fixed number of tokens per expert, e.g. 1.25x the even
 *     share), or an explicit C; overflow is decided per (token, expert)
 *     assignment in token order; surviving gates of a partly dropped token
 *     are not renormalised;
 *   - a dropped assignment contributes nothing to the MoE output; with the
 *     residual added, a fully dropped token leaves the layer as it came in
 *     (ai360xpert "Load Balancing and Dropped Tokens", capacity limits;
 *     Ultralytics "Load Balancing and Capacity": skipped tokens ride the
 *     residual path);
 *   - source rank of token t is t / ceil(T/R); expert e lives on rank
 *     e / (E/R);
 *   - expert FFNs have no biases; GELU is the exact erf form; SwiGLU is
 *     silu(gate) * up followed by the down projection.
 *
 * Parallelism: OpenMP over independent tokens / rows only; nothing in the
 * arithmetic of one token depends on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_SOFTMAX = 0, OR_SIGMOID = 1 };
enum { OR_GELU = 0, OR_SWIGLU = 1, OR_IDENTITY = 2 };

/* Exact widening of one stored element to double. */
static double elem(const void* base, int dtype, int64_t i) {
    if (dtype == OR_BF16) {
        uint16_t h = ((const uint16_t*)base)[i];
        uint32_t bits = ((uint32_t)h) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[i];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Step 1: Route (Ultralytics, How Tokens Move Between GPUs, step 1): each   */
/* token gets a score per expert and the k best experts are kept.  The       */
/* selection-only bias is DeepSeek-V3's per-expert bias that changes which   */
/* experts win but not the weights (Ultralytics, Load Balancing and          */
/* Capacity, bias-based balancing); it is supported for sigmoid scores.      */
/* ------------------------------------------------------------------------ */

/* The fp32 logit of token t against expert e. */
static float logit32(const void* x, const void* w, int dtype, int64_t t, int e,
                     int d, const float* logit_bias) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
        acc += elem(x, dtype, t * (int64_t)d + i) * elem(w, dtype, (int64_t)e * d + i);
    float L = (float)acc;
    if (logit_bias) L = L + logit_bias[e];
    return L;
}

/* The fp32 sigmoid score used for selection and for sigmoid gates. */
float oracle_sigmoid32(float L) {
    return (float)(1.0 / (1.0 + exp(-(double)L)));
}

/*
 * x [T,d], w_router [E,d] (row-major, dtype), logit_bias [E] or NULL,
 * sel_bias [E] or NULL (sigmoid only).
 * Outputs: topk_idx [T,k] in selection order (descending key, ties to the
 * lower index), topk_gate [T,k], logits [T,E] (fp32, may be NULL).
 * Returns 0, or -1 for an unsupported combination.
 */
int oracle_route(int64_t T, int d, int E, int k, int dtype, int score, int renorm,
                 const void* x, const void* w_router, const float* logit_bias,
                 const float* sel_bias, int R, int max_ranks, int32_t* topk_idx,
                 float* topk_gate, float* logits_out) {
    if (k < 1 || k > E) return -1;
    if (score == OR_SOFTMAX && sel_bias) return -1;
    if (max_ranks > 0 && (R < 1 || E % R != 0 || max_ranks > R || max_ranks * (E / R) < k))
        return -1;
    const int per = (R > 0) ? E / R : E;
    int bad = 0;
#pragma omp parallel
    {
        float* L = (float*)malloc(sizeof(float) * E);
        float* key = (float*)malloc(sizeof(float) * E);
        float* s = (float*)malloc(sizeof(float) * E);
        char* taken = (char*)malloc(E);
        if (!L || !key || !s || !taken) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < T; ++t) {
                for (int e = 0; e < E; ++e) {
                    L[e] = logit32(x, w_router, dtype, t, e, d, logit_bias);
                    if (score == OR_SIGMOID) {
                        s[e] = oracle_sigmoid32(L[e]);
                        key[e] = sel_bias ? s[e] + sel_bias[e] : s[e];
                    } else {
                        key[e] = L[e];
                    }
                    taken[e] = 0;
                    if (logits_out) logits_out[t * E + e] = L[e];
                }
                /* Rank-limited routing (DeepSeek-V3 sends a token to experts on
                   at most max_ranks devices; Ultralytics, Load Balancing and
                   Capacity).  Reading: a rank's score is the best key among its
                   experts; max_ranks rounds pick the best rank not yet picked
                   (ties to the lower rank); experts of other ranks are taken
                   out of the selection below. */
                if (max_ranks > 0 && max_ranks < R) {
                    char* rank_taken = (char*)calloc((size_t)R, 1);
                    for (int m = 0; m < max_ranks; ++m) {
                        int best_r = -1;
                        float best_s = 0.f;
                        for (int r = 0; r < R; ++r) {
                            if (rank_taken[r]) continue;
                            float sr = key[r * per];
                            for (int e = r * per + 1; e < (r + 1) * per; ++e)
                                if (key[e] > sr) sr = key[e];
                            if (best_r < 0 || sr > best_s) {
                                best_r = r;
                                best_s = sr;
                            }
                        }
                        rank_taken[best_r] = 1;
                    }
                    for (int e = 0; e < E; ++e)
                        if (!rank_taken[e / per]) taken[e] = 1;  /* not selectable */
                    free(rank_taken);
                }
                /* k rounds: the largest key not yet taken; ascending scan and a
                   strict comparison give ties to the lower index. */
                int32_t* idx = topk_idx + t * k;
                for (int j = 0; j < k; ++j) {
                    int best = -1;
                    for (int e = 0; e < E; ++e) {
                        if (taken[e]) continue;
                        if (best < 0 || key[e] > key[best]) best = e;
                    }
                    taken[best] = 1;
                    idx[j] = best;
                }
                /* Gates: the router weights applied in step 4, Combine. */
                float* g = topk_gate + t * k;
                if (score == OR_SOFTMAX) {
                    double m = -INFINITY;
                    if (renorm) {
                        for (int j = 0; j < k; ++j) m = fmax(m, (double)L[idx[j]]);
                    } else {
                        for (int e = 0; e < E; ++e) m = fmax(m, (double)L[e]);
                    }
                    double z = 0.0;
                    if (renorm) {
                        for (int j = 0; j < k; ++j) z += exp((double)L[idx[j]] - m);
                    } else {
                        for (int e = 0; e < E; ++e) z += exp((double)L[e] - m);
                    }
                    for (int j = 0; j < k; ++j) g[j] = (float)(exp((double)L[idx[j]] - m) / z);
                } else {
                    if (renorm) {
                        double z = 0.0;
                        for (int j = 0; j < k; ++j) z += (double)s[idx[j]];
                        for (int j = 0; j < k; ++j) g[j] = (float)((double)s[idx[j]] / z);
                    } else {
                        for (int j = 0; j < k; ++j) g[j] = s[idx[j]];
                    }
                }
            }
        }
        free(L);
        free(key);
        free(s);
        free(taken);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: Dispatch, as counts, capacity and an on-device layout.           */
/* ------------------------------------------------------------------------ */

/* Capacity per expert: an explicit value, else ceil(cf*T*k/E) evaluated left
   to right in double, else -1 (no limit). */
int64_t oracle_capacity(int64_t T, int k, int E, double cf, int64_t explicit_cap) {
    if (explicit_cap > 0) return explicit_cap;
    if (!(cf > 0.0)) return -1;
    return (int64_t)ceil(cf * (double)T * (double)k / (double)E);
}

/*
 * topk_idx [T,k] -> per-expert load (pre-drop), expert-major row offsets of
 * the kept rows [E+1], kept rows per virtual rank [R], the would-be
 * all-to-all send counts [R,R] (source rank of the token, destination rank of
 * the expert), slot_row [T,k] (row in the expert-major buffer, -1 if dropped),
 * row_token [rows] (row -> token) and the number of dropped assignments.
 * Token order is kept inside every expert segment (mbrenndoerfer.com
 * Summary: the buffers must keep the tokens' order through dispatch, compute
 * and combine).  Returns the number of kept rows.
 */
int64_t oracle_dispatch(int64_t T, int E, int k, int R, int64_t C, const int32_t* topk_idx,
                        int32_t* expert_counts, int32_t* expert_offsets, int32_t* rank_counts,
                        int32_t* rank_splits, int32_t* slot_row, int32_t* row_token,
                        int64_t* n_dropped) {
    int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * k > 0 ? T * k : 1));
    if (!seen || !pos) {
        free(seen);
        free(pos);
        return -1;
    }
    /* Position of each assignment among the assignments of the same expert,
       counted in token order. */
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[t * k + j];
            pos[t * k + j] = seen[e]++;
        }
    for (int e = 0; e < E; ++e) expert_counts[e] = (int32_t)seen[e];
    /* Kept rows per expert and the exclusive prefix over experts. */
    expert_offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t kept = seen[e];
        if (C >= 0 && kept > C) kept = C;
        expert_offsets[e + 1] = expert_offsets[e] + (int32_t)kept;
    }
    int per_rank = E / R;
    int64_t tok_per_src = (T + R - 1) / R;
    for (int r = 0; r < R; ++r) rank_counts[r] = 0;
    for (int i = 0; i < R * R; ++i) rank_splits[i] = 0;
    int64_t dropped = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[t * k + j];
            int64_t p = pos[t * k + j];
            if (C >= 0 && p >= C) {
                slot_row[t * k + j] = -1;
                ++dropped;
                continue;
            }
            int32_t row = expert_offsets[e] + (int32_t)p;
            slot_row[t * k + j] = row;
            row_token[row] = (int32_t)t;
            int dst = e / per_rank;
            int src = (int)(t / tok_per_src);
            rank_counts[dst] += 1;
            rank_splits[src * R + dst] += 1;
        }
    *n_dropped = dropped;
    int64_t rows = expert_offsets[E];
    free(seen);
    free(pos);
    return rows;
}

/* The permutation itself: each token's hidden state is written to the row of
   every expert that kept it.  Elements are moved as raw bytes. */
void oracle_permute(int64_t T, int k, int64_t row_bytes, const void* x, const int32_t* slot_row,
                    void* xp) {
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int32_t row = slot_row[t * k + j];
            if (row < 0) continue;
            memcpy((char*)xp + (int64_t)row * row_bytes, (const char*)x + t * row_bytes,
                   (size_t)row_bytes);
        }
}

/* ------------------------------------------------------------------------ */
/* Step 3: Compute (step 3): every expert processes the rows dispatched to  */
/* it.  One expert FFN applied to n_rows rows.                               */
/* ------------------------------------------------------------------------ */

static double gelu_exact(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }
static double silu(double v) { return v / (1.0 + exp(-v)); }

/*
 * rows [n_rows,d] (dtype), w_up [f,d] (GELU) or [2f,d] with gate rows first
 * then up rows (SwiGLU), w_down [d,f]; out [n_rows,d] fp64, no intermediate
 * rounding.  Identity: out = rows.
 */
void oracle_expert_ffn(int64_t n_rows, int d, int f, int act, int dtype, const void* rows,
                       const void* w_up, const void* w_down, double* out) {
    if (act == OR_IDENTITY) {
        for (int64_t r = 0; r < n_rows; ++r)
            for (int c = 0; c < d; ++c) out[r * d + c] = elem(rows, dtype, r * d + c);
        return;
    }
#pragma omp parallel
    {
        double* xr = (double*)malloc(sizeof(double) * d);
        double* h = (double*)malloc(sizeof(double) * f);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int i = 0; i < d; ++i) xr[i] = elem(rows, dtype, r * d + i);
            for (int n = 0; n < f; ++n) {
                double a = 0.0;
                for (int i = 0; i < d; ++i) a += xr[i] * elem(w_up, dtype, (int64_t)n * d + i);
                if (act == OR_GELU) {
                    h[n] = gelu_exact(a);
                } else {
                    double u = 0.0;
                    for (int i = 0; i < d; ++i)
                        u += xr[i] * elem(w_up, dtype, (int64_t)(f + n) * d + i);
                    h[n] = silu(a) * u;
                }
            }
            for (int c = 0; c < d; ++c) {
                double a = 0.0;
                for (int n = 0; n < f; ++n) a += h[n] * elem(w_down, dtype, (int64_t)c * f + n);
                out[r * d + c] = a;
            }
        }
        free(xr);
        free(h);
    }
}

/* ------------------------------------------------------------------------ */
/* Step 4: Combine (step 4): expert outputs come back to token order and    */
/* are summed with the router gates as weights.                             */
/* ------------------------------------------------------------------------ */

/*
 * Tokens toks[0..n_tok) are produced into y [n_tok,d].  The expert-major
 * buffer is addressed through slot_row: the output of row r is
 * yp_rows[row_map[r] * d ...] (row_map lets a caller hold only the rows that
 * the listed tokens use).  shared [n_tok,d] fp64 or NULL (always-on shared
 * expert, gate 1); resid [T,d] (dtype) or NULL (the residual connection).
 */
void oracle_combine(int64_t n_tok, const int64_t* toks, int d, int k, const double* yp_rows,
                    const int32_t* row_map, const int32_t* slot_row, const float* topk_gate,
                    const double* shared, int dtype, const void* resid, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_tok; ++i) {
        int64_t t = toks[i];
        double* yt = y + i * d;
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t row = slot_row[t * k + j];
                if (row < 0) continue;
                acc += (double)topk_gate[t * k + j] * yp_rows[(int64_t)row_map[row] * d + c];
            }
            if (shared) acc += shared[i * d + c];
            if (resid) acc += elem(resid, dtype, t * d + c);
            yt[c] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Bias-based balancing (Ultralytics, Load Balancing and Capacity: DeepSeek-V3 */
/* lowers the selection bias of overloaded experts and raises it for idle     */
/* ones after each step).  The step size gamma is not on the pages.  Reading: */
/* an expert whose load is above the even share T*k/E is overloaded (bias -=  */
/* gamma), one below it is underloaded (bias += gamma), one exactly at it is   */
/* left alone; the comparison is exact (count*E against T*k in integers) and   */
/* the update is one fp32 addition.                                            */
/* ------------------------------------------------------------------------ */
void oracle_update_sel_bias(int64_t T, int k, int E, const int32_t* counts, float* bias,
                            float gamma) {
    const int64_t even = T * (int64_t)k;
    for (int e = 0; e < E; ++e) {
        const int64_t load = (int64_t)counts[e] * E;
        if (load > even) bias[e] = bias[e] - gamma;
        else if (load < even) bias[e] = bias[e] + gamma;
    }
}

/* ------------------------------------------------------------------------ */
/* Backward of the two exchanges (training is the pages' main setting:        */
/* topicspectrum "Training teaches both experts and router").                 */
/* Combine is y[t] = sum_j g[t,j] * yp[slot_row[t,j]] over kept slots, linear */
/* in yp and in g, so with dy = dL/dy:                                         */
/*   d_yp[slot_row[t,j]] = g[t,j] * dy[t]       (the reverse exchange),        */
/*   d_gate[t,j]         = sum_c dy[t,c] * yp[slot_row[t,j], c],               */
/* and 0 for dropped slots.  Dispatch is xp[slot_row[t,j]] = x[t], so          */
/*   dx[t] = sum over kept j of d_xp[slot_row[t,j]].                          */
/* ------------------------------------------------------------------------ */
void oracle_combine_backward(int64_t T, int d, int k, int dtype, const void* dy, const void* yp,
                             const int32_t* slot_row, const float* gate, double* d_yp,
                             double* d_gate) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int32_t row = slot_row[t * k + j];
            if (row < 0) {
                d_gate[t * k + j] = 0.0;
                continue;
            }
            double dot = 0.0;
            for (int c = 0; c < d; ++c) {
                const double g = elem(dy, dtype, t * d + c);
                dot += g * elem(yp, dtype, (int64_t)row * d + c);
                d_yp[(int64_t)row * d + c] = (double)gate[t * k + j] * g;
            }
            d_gate[t * k + j] = dot;
        }
}

void oracle_dispatch_backward(int64_t T, int d, int k, int dtype, const void* d_xp,
                              const int32_t* slot_row, double* dx) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                const int32_t row = slot_row[t * k + j];
                if (row >= 0) acc += elem(d_xp, dtype, (int64_t)row * d + c);
            }
            dx[t * d + c] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Backward through one expert FFN, for its n_rows rows: given the output    */
/* gradient d_out [n_rows,d], the input gradient d_in [n_rows,d] and, when   */
/* the pointers are not NULL, the weight gradients d_w_up [f or 2f, d] and    */
/* d_w_down [d, f] (accumulated over the rows).  fp64, no intermediate       */
/* rounding.  GELU: h = gelu(a), a = W1 x; gelu'(a) = Phi(a) + a phi(a).      */
/* SwiGLU: h = silu(g) u; silu'(g) = s (1 + g (1 - s)), s = sigmoid(g).       */
/* ------------------------------------------------------------------------ */
void oracle_expert_ffn_backward(int64_t n_rows, int d, int f, int act, int dtype, const void* rows,
                                const void* w_up, const void* w_down, const void* d_out,
                                double* d_in, double* d_w_up, double* d_w_down) {
    const int up_rows = act == OR_SWIGLU ? 2 * f : f;
    double* xr = (double*)malloc(sizeof(double) * d);
    double* pre = (double*)malloc(sizeof(double) * up_rows);
    double* h = (double*)malloc(sizeof(double) * f);
    double* dh = (double*)malloc(sizeof(double) * f);
    double* dpre = (double*)malloc(sizeof(double) * up_rows);
    double* dy = (double*)malloc(sizeof(double) * d);
    if (d_w_up) memset(d_w_up, 0, sizeof(double) * (size_t)up_rows * d);
    if (d_w_down) memset(d_w_down, 0, sizeof(double) * (size_t)d * f);
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int i = 0; i < d; ++i) {
            xr[i] = elem(rows, dtype, r * d + i);
            dy[i] = elem(d_out, dtype, r * d + i);
        }
        for (int n = 0; n < up_rows; ++n) {
            double a = 0.0;
            for (int i = 0; i < d; ++i) a += xr[i] * elem(w_up, dtype, (int64_t)n * d + i);
            pre[n] = a;
        }
        for (int n = 0; n < f; ++n) {
            if (act == OR_GELU) {
                h[n] = gelu_exact(pre[n]);
            } else {
                h[n] = silu(pre[n]) * pre[f + n];
            }
        }
        /* dh = W_down^T dy */
        for (int n = 0; n < f; ++n) {
            double a = 0.0;
            for (int c = 0; c < d; ++c) a += dy[c] * elem(w_down, dtype, (int64_t)c * f + n);
            dh[n] = a;
        }
        for (int n = 0; n < f; ++n) {
            if (act == OR_GELU) {
                const double a = pre[n];
                const double phi = exp(-0.5 * a * a) / sqrt(2.0 * 3.14159265358979323846);
                dpre[n] = dh[n] * (0.5 * (1.0 + erf(a / sqrt(2.0))) + a * phi);
            } else {
                const double g = pre[n], u = pre[f + n];
                const double s = 1.0 / (1.0 + exp(-g));
                dpre[n] = dh[n] * u * s * (1.0 + g * (1.0 - s));
                dpre[f + n] = dh[n] * g * s;
            }
        }
        /* d_in = W_up^T dpre */
        for (int i = 0; i < d; ++i) {
            double a = 0.0;
            for (int n = 0; n < up_rows; ++n) a += dpre[n] * elem(w_up, dtype, (int64_t)n * d + i);
            d_in[r * d + i] = a;
        }
        if (d_w_down)
            for (int c = 0; c < d; ++c)
                for (int n = 0; n < f; ++n) d_w_down[(int64_t)c * f + n] += dy[c] * h[n];
        if (d_w_up)
            for (int n = 0; n < up_rows; ++n)
                for (int i = 0; i < d; ++i) d_w_up[(int64_t)n * d + i] += dpre[n] * xr[i];
    }
    free(xr);
    free(pre);
    free(h);
    free(dh);
    free(dpre);
    free(dy);
}

/* ------------------------------------------------------------------------ */
/* Backward of Step 1, Route: the router is trained through its gates       */
/* (topicspectrum, Training teaches both experts and router).  Which        */
/* experts a token picks is piecewise constant in the logits, so no         */
/* gradient flows through the selection (nor into the selection-only bias); */
/* it flows through the gates, each a function of the logits L = x W^T + b: */
/*   softmax, renormalised: g_j = exp(L_j) / sum over chosen i of exp(L_i)  */
/*     dL_j = g_j (dg_j - sum_i g_i dg_i) for chosen j, 0 for the others;    */
/*   softmax, full: g_j = p_(e_j), p the softmax over all E experts          */
/*     dL_e = p_e (dg_e - sum_j p_(e_j) dg_j) for every e (dg_e = 0 unless   */
/*     e was chosen);                                                        */
/*   sigmoid, renormalised: g_j = s_j / sum over chosen i of s_i, s = sig(L) */
/*     ds_j = (dg_j - sum_i g_i dg_i) / sum_i s_i, dL_j = ds_j s_j (1 - s_j);*/
/*   sigmoid: g_j = s_j, dL_j = dg_j s_j (1 - s_j).                          */
/* Then d_logit_bias[e] = sum_t dL[t,e], dx[t] = sum_e dL[t,e] W[e] and      */
/* dW[e] = sum_t dL[t,e] x[t].  Everything in fp64 from the inputs (the      */
/* logits recomputed in fp64; exact on the dyadic test grid).               */
/* ------------------------------------------------------------------------ */
void oracle_route_backward(int64_t T, int d, int E, int k, int dtype, int score, int renorm,
                           const void* x, const void* w_router, const float* logit_bias,
                           const int32_t* topk_idx, const float* d_gate, double* d_logits,
                           double* dx, double* dw, double* d_logit_bias) {
#pragma omp parallel
    {
        double* L = (double*)malloc(sizeof(double) * E);
        double* g = (double*)malloc(sizeof(double) * k);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i)
                    acc += elem(x, dtype, t * (int64_t)d + i) * elem(w_router, dtype, (int64_t)e * d + i);
                L[e] = acc + (logit_bias ? (double)logit_bias[e] : 0.0);
            }
            const int32_t* idx = topk_idx + t * k;
            const float* dg = d_gate + t * k;
            double* dL = d_logits + t * E;
            for (int e = 0; e < E; ++e) dL[e] = 0.0;
            if (score == OR_SOFTMAX && renorm) {
                double m = -INFINITY, z = 0.0, dot = 0.0;
                for (int j = 0; j < k; ++j) m = fmax(m, L[idx[j]]);
                for (int j = 0; j < k; ++j) z += exp(L[idx[j]] - m);
                for (int j = 0; j < k; ++j) {
                    g[j] = exp(L[idx[j]] - m) / z;
                    dot += g[j] * (double)dg[j];
                }
                for (int j = 0; j < k; ++j) dL[idx[j]] = g[j] * ((double)dg[j] - dot);
            } else if (score == OR_SOFTMAX) {
                double m = -INFINITY, z = 0.0, dot = 0.0;
                for (int e = 0; e < E; ++e) m = fmax(m, L[e]);
                for (int e = 0; e < E; ++e) z += exp(L[e] - m);
                for (int j = 0; j < k; ++j) dot += exp(L[idx[j]] - m) / z * (double)dg[j];
                for (int e = 0; e < E; ++e) dL[e] = -exp(L[e] - m) / z * dot;
                for (int j = 0; j < k; ++j) dL[idx[j]] += exp(L[idx[j]] - m) / z * (double)dg[j];
            } else {
                double sum = 0.0, dot = 0.0;
                for (int j = 0; j < k; ++j) sum += 1.0 / (1.0 + exp(-L[idx[j]]));
                for (int j = 0; j < k; ++j) {
                    g[j] = (1.0 / (1.0 + exp(-L[idx[j]]))) / sum;
                    dot += g[j] * (double)dg[j];
                }
                for (int j = 0; j < k; ++j) {
                    const double s = 1.0 / (1.0 + exp(-L[idx[j]]));
                    const double ds = renorm ? ((double)dg[j] - dot) / sum : (double)dg[j];
                    dL[idx[j]] = ds * s * (1.0 - s);
                }
            }
            if (dx)
                for (int i = 0; i < d; ++i) {
                    double acc = 0.0;
                    for (int e = 0; e < E; ++e)
                        acc += dL[e] * elem(w_router, dtype, (int64_t)e * d + i);
                    dx[t * d + i] = acc;
                }
        }
        free(L);
        free(g);
    }
    if (dw)
#pragma omp parallel for schedule(static)
        for (int e = 0; e < E; ++e)
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t)
                    acc += d_logits[t * E + e] * elem(x, dtype, t * (int64_t)d + i);
                dw[(int64_t)e * d + i] = acc;
            }
    if (d_logit_bias)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) acc += d_logits[t * E + e];
            d_logit_bias[e] = acc;
        }
}
