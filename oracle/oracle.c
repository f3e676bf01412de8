/*
 * oracle.c -- plain, slow fp64 CPU reference for the KVpop hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; every function restates a
 * definition from the KVpop pages in the most direct form available.
 *
 * Sources (page title, section / equation):
 *   [KVpop notes] "KVpop -- Key-Value Cache Compression with Predictive Online
 *                  Pruning 精读笔记" (liuzhao09.github.io), sections 2.1-2.3:
 *                  budget B = s + w + k; eligible set E(q) = {t : s <= t <= q-w};
 *                  mask M_{q,t} = [t<s] v [q-t<w] v ([t in E(q)] ^ [rank(t) <= tau_q]);
 *                  future mass m_t = (1/N_t) sum_{d=t+w}^{S-1} A_{d,t};
 *                  Eq. (8): log m_t = log sum_{d>=t+w} exp(l(d,t) - LSE_d) - log N_t.
 *   [KVpop summary] "KVpop — 基于预测性在线剪枝的键值缓存压缩" (gist.science),
 *                  section 2.4: running threshold over static priorities kept
 *                  with a Fenwick tree.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of the repository):
 *   - causality t <= q is ANDed into M;
 *   - rank is 0-based, smaller = better; order = (priority desc, index asc);
 *     NaN priority counts as -inf; -0.0 == +0.0;
 *   - tau_q = INT32_MAX when |E(q)| <= k (all eligible kept), -1 when k == 0;
 *   - the future-attention target is the unnormalised sum over the query heads
 *     g of the group: no 1/N_t, no 1/G, no epsilon; an empty sum gives -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TAU_ALL INT32_MAX

/* ------------------------------------------------------------------------ */
/* static priority order                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    double v;
    int32_t idx;
} keyed_t;

static double prio_value(float p) { return isnan(p) ? -INFINITY : (double)p; }

/* better-first: larger priority first, then smaller index */
static int cmp_keyed(const void* a, const void* b) {
    const keyed_t* x = (const keyed_t*)a;
    const keyed_t* y = (const keyed_t*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/* rank[t] = position of token t in the (priority desc, index asc) order. */
int oracle_rank(const float* prio, int S, int32_t* rank) {
    keyed_t* a = (keyed_t*)malloc(sizeof(keyed_t) * (size_t)(S > 0 ? S : 1));
    if (!a) return -1;
    for (int t = 0; t < S; ++t) {
        a[t].v = prio_value(prio[t]);
        a[t].idx = t;
    }
    qsort(a, (size_t)S, sizeof(keyed_t), cmp_keyed);
    for (int r = 0; r < S; ++r) rank[a[r].idx] = r;
    free(a);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* running top-k threshold tau_q                                             */
/* ------------------------------------------------------------------------ */

/*
 * Fenwick (binary indexed) tree over rank values: for q = 0..S-1 the token
 * t_new = q - w enters E(q) (when t_new >= s); tau_q is the rank of the k-th
 * best eligible token, found with a k-th-order-statistic descent.
 */
int oracle_tau_fenwick(const int32_t* rank, int S, int s, int w, int k, int32_t* tau) {
    int32_t* bit = (int32_t*)calloc((size_t)S + 1, sizeof(int32_t));
    if (!bit) return -1;
    int top = 1;
    while (top * 2 <= S) top *= 2;
    int n = 0; /* |E(q)| */
    for (int q = 0; q < S; ++q) {
        int t_new = q - w;
        if (t_new >= s) {
            for (int i = rank[t_new] + 1; i <= S; i += i & (-i)) bit[i] += 1;
            n += 1;
        }
        if (k == 0) {
            tau[q] = -1;
        } else if (n <= k) {
            tau[q] = TAU_ALL;
        } else {
            /* smallest position p (1-based) whose prefix count reaches k */
            int pos = 0, rem = k;
            for (int step = top; step > 0; step >>= 1) {
                if (pos + step <= S && bit[pos + step] < rem) {
                    pos += step;
                    rem -= bit[pos];
                }
            }
            tau[q] = pos; /* 1-based position pos+1 holds rank value pos */
        }
    }
    free(bit);
    return 0;
}

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Brute force: sort the ranks of E(q) for every q and read the k-th. */
int oracle_tau_bruteforce(const int32_t* rank, int S, int s, int w, int k, int32_t* tau) {
    int32_t* buf = (int32_t*)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    if (!buf) return -1;
    for (int q = 0; q < S; ++q) {
        int n = 0;
        for (int t = s; t <= q - w; ++t) buf[n++] = rank[t];
        if (k == 0) {
            tau[q] = -1;
        } else if (n <= k) {
            tau[q] = TAU_ALL;
        } else {
            qsort(buf, (size_t)n, sizeof(int32_t), cmp_i32);
            tau[q] = buf[k - 1];
        }
    }
    free(buf);
    return 0;
}

/* M_{q,t} with causality: sinks, protected window, or kept eligible token. */
static int retained(const int32_t* rank, const int32_t* tau, int s, int w, int q, int t) {
    if (t > q) return 0;
    if (t < s) return 1;
    if (q - t < w) return 1;
    return rank[t] <= tau[q]; /* here s <= t <= q - w, i.e. t in E(q) */
}

int oracle_retained(const int32_t* rank, const int32_t* tau, int s, int w, int q, int t) {
    return retained(rank, tau, s, w, q, t);
}

/* Dense boolean mask [S,S] (row q, column t); small S only. */
void oracle_mask_dense(const int32_t* rank, const int32_t* tau, int S, int s, int w, uint8_t* M) {
    for (int q = 0; q < S; ++q)
        for (int t = 0; t < S; ++t) M[(size_t)q * S + t] = (uint8_t)retained(rank, tau, s, w, q, t);
}

/*
 * evict_at[t]: the first row q >= t + w at which t is no longer retained, or
 * S if t is retained until the end (sinks always get S).  Definition: scan.
 */
void oracle_evict_at_scan(const int32_t* rank, const int32_t* tau, int S, int s, int w, int32_t* ev) {
    for (int t = 0; t < S; ++t) {
        if (t < s) {
            ev[t] = S;
            continue;
        }
        int q = t + w;
        while (q < S && retained(rank, tau, s, w, q, t)) ++q;
        ev[t] = q < S ? q : S;
    }
}

/*
 * evict_at by online eviction: at row q the token u = q - w enters E(q); once
 * more than k tokens are eligible either u itself is rejected or the worst
 * member of the previous top-k set leaves.
 */
int oracle_evict_at_sweep(const int32_t* rank, const int32_t* tau, int S, int s, int w, int k,
                          int32_t* ev) {
    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    if (!perm) return -1;
    for (int t = 0; t < S; ++t) perm[rank[t]] = t;
    for (int t = 0; t < S; ++t) ev[t] = S;
    for (int q = 0; q < S; ++q) {
        int u = q - w;
        if (u < s) continue;
        int n = u - s + 1;
        if (k == 0) {
            ev[u] = q;
            continue;
        }
        if (n <= k) continue;
        if (rank[u] > tau[q]) {
            ev[u] = q;
        } else {
            int m;
            if (tau[q - 1] != TAU_ALL) {
                m = perm[tau[q - 1]];
            } else {
                m = s;
                for (int t = s; t < u; ++t)
                    if (rank[t] > rank[m]) m = t;
            }
            ev[m] = q;
        }
    }
    free(perm);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* attention rows                                                            */
/* ------------------------------------------------------------------------ */

static double dot_f(const float* a, const float* b, int D) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += (double)a[d] * (double)b[d];
    return acc;
}

/*
 * Softmax attention of one query vector over the retained keys of row qpos.
 *   qv   [nrows, D]          query vectors (row r uses qv + r*D)
 *   k, v [b, S, H, D]        keys / values
 *   rank, tau [b, H, S]      mask inputs; NULL => dense causal (t <= qpos)
 *   rows [nrows, 3]          (batch index, query head j, position qpos);
 *                            query head j reads KV head j / G
 *   O    [nrows, D] or NULL, lse [nrows]; an empty row gives O = 0, LSE = -inf.
 */
void oracle_attn_rows(const float* qv, const float* k, const float* v, int b, int S, int H, int G,
                      int D, double scale, const int32_t* rank, const int32_t* tau, int s, int w,
                      const int32_t* rows, int64_t nrows, double* O, double* lse) {
    (void)b;
#pragma omp parallel
    {
        double* l = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        uint8_t* keep = (uint8_t*)malloc((size_t)(S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            int bi = rows[3 * r + 0], j = rows[3 * r + 1], qp = rows[3 * r + 2];
            int h = j / G;
            const int32_t* rk = rank ? rank + ((size_t)bi * H + h) * S : NULL;
            const int32_t* tu = tau ? tau + ((size_t)bi * H + h) * S : NULL;
            const float* qrow = qv + (size_t)r * D;
            double m = -INFINITY;
            int any = 0;
            for (int t = 0; t <= qp; ++t) {
                keep[t] = (uint8_t)(rk ? retained(rk, tu, s, w, qp, t) : 1);
                if (!keep[t]) continue;
                const float* krow = k + (((size_t)bi * S + t) * H + h) * D;
                l[t] = scale * dot_f(qrow, krow, D);
                if (l[t] > m) m = l[t];
                any = 1;
            }
            if (!any) {
                lse[r] = -INFINITY;
                if (O) memset(O + (size_t)r * D, 0, sizeof(double) * (size_t)D);
                continue;
            }
            double sum = 0.0;
            for (int t = 0; t <= qp; ++t)
                if (keep[t]) sum += exp(l[t] - m);
            double L = m + log(sum);
            lse[r] = L;
            if (O) {
                double* o = O + (size_t)r * D;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (int t = 0; t <= qp; ++t) {
                    if (!keep[t]) continue;
                    double p = exp(l[t] - L);
                    const float* vrow = v + (((size_t)bi * S + t) * H + h) * D;
                    for (int d = 0; d < D; ++d) o[d] += p * (double)vrow[d];
                }
            }
        }
        free(l);
        free(keep);
    }
}

/* ------------------------------------------------------------------------ */
/* attention backward                                                        */
/* ------------------------------------------------------------------------ */

/*
 * [KVpop notes] 2.1 (Figure 1, training flow): the student runs attention over
 * the retained set M_{q,.} and is trained through it, so the sparse attention
 * needs its gradient.  For one row with logits l_t = scale * q.k_t over R_q,
 * softmax P_t = exp(l_t - LSE) and output O = sum_t P_t v_t, the gradient of a
 * loss L with upstream dO = dL/dO is the chain rule through the softmax:
 *   dv_t += P_t dO
 *   dP_t  = dO . v_t
 *   dS_t  = P_t (dP_t - sum_u P_u dP_u)          (the softmax Jacobian)
 *   dq    = scale * sum_t dS_t k_t
 *   dk_t += scale * dS_t q
 * This computes one row: idx[] receives the retained keys in position order,
 * P[] and dS[] their probabilities and logit gradients.  Returns |R_q|.
 */
static int row_grad(const float* qrow, const float* dorow, const float* k, const float* v, int bi,
                    int S, int H, int h, int D, double scale, const int32_t* rk, const int32_t* tu,
                    int s, int w, int qp, int32_t* idx, double* P, double* dS) {
    int n = 0;
    double m = -INFINITY;
    for (int t = 0; t <= qp; ++t) {
        if (rk && !retained(rk, tu, s, w, qp, t)) continue;
        idx[n] = t;
        P[n] = scale * dot_f(qrow, k + (((size_t)bi * S + t) * H + h) * D, D);
        if (P[n] > m) m = P[n];
        ++n;
    }
    if (n == 0) return 0;
    double sum = 0.0;
    for (int i = 0; i < n; ++i) sum += exp(P[i] - m);
    double L = m + log(sum);
    double dsum = 0.0;
    for (int i = 0; i < n; ++i) {
        P[i] = exp(P[i] - L);
        dS[i] = dot_f(dorow, v + (((size_t)bi * S + idx[i]) * H + h) * D, D);
        dsum += P[i] * dS[i];
    }
    for (int i = 0; i < n; ++i) dS[i] = P[i] * (dS[i] - dsum);
    return n;
}

/*
 * Gradients of every row: q, dO [b,S,Hq,D]; k, v [b,S,H,D]; rank/tau [b,H,S]
 * (NULL => dense causal).  dq [b,S,Hq,D], dk, dv [b,S,H,D] fp64, overwritten.
 * One (batch, KV head) per thread, so its dk/dv rows have a single writer.
 */
void oracle_attn_bwd(const float* q, const float* k, const float* v, const float* dO, int b, int S,
                     int H, int G, int D, double scale, const int32_t* rank, const int32_t* tau,
                     int s, int w, double* dq, double* dk, double* dv) {
    int Hq = H * G;
    memset(dq, 0, sizeof(double) * (size_t)b * S * Hq * D);
    memset(dk, 0, sizeof(double) * (size_t)b * S * H * D);
    memset(dv, 0, sizeof(double) * (size_t)b * S * H * D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < b * H; ++bh) {
        int bi = bh / H, h = bh % H;
        const int32_t* rk = rank ? rank + ((size_t)bi * H + h) * S : NULL;
        const int32_t* tu = tau ? tau + ((size_t)bi * H + h) * S : NULL;
        int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
        double* P = (double*)malloc(sizeof(double) * (size_t)S);
        double* dS = (double*)malloc(sizeof(double) * (size_t)S);
        for (int g = 0; g < G; ++g) {
            int j = h * G + g;
            for (int qp = 0; qp < S; ++qp) {
                size_t ro = (((size_t)bi * S + qp) * Hq + j) * D;
                int n = row_grad(q + ro, dO + ro, k, v, bi, S, H, h, D, scale, rk, tu, s, w, qp, idx, P, dS);
                for (int i = 0; i < n; ++i) {
                    size_t ko = (((size_t)bi * S + idx[i]) * H + h) * D;
                    for (int d = 0; d < D; ++d) {
                        dq[ro + d] += scale * dS[i] * (double)k[ko + d];
                        dk[ko + d] += scale * dS[i] * (double)q[ro + d];
                        dv[ko + d] += P[i] * (double)dO[ro + d];
                    }
                }
            }
        }
        free(idx);
        free(P);
        free(dS);
    }
}

/*
 * dq of explicit rows (batch, query head j, position): qv / dov [nrows, D] are
 * the rows' query and upstream-gradient vectors.  dq [nrows, D].
 */
void oracle_attn_bwd_rows(const float* qv, const float* dov, const float* k, const float* v, int b,
                          int S, int H, int G, int D, double scale, const int32_t* rank,
                          const int32_t* tau, int s, int w, const int32_t* rows, int64_t nrows,
                          double* dq) {
    (void)b;
#pragma omp parallel
    {
        int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
        double* P = (double*)malloc(sizeof(double) * (size_t)S);
        double* dS = (double*)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            int bi = rows[3 * r + 0], j = rows[3 * r + 1], qp = rows[3 * r + 2];
            int h = j / G;
            const int32_t* rk = rank ? rank + ((size_t)bi * H + h) * S : NULL;
            const int32_t* tu = tau ? tau + ((size_t)bi * H + h) * S : NULL;
            int n = row_grad(qv + (size_t)r * D, dov + (size_t)r * D, k, v, bi, S, H, h, D, scale, rk, tu,
                             s, w, qp, idx, P, dS);
            double* o = dq + (size_t)r * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int i = 0; i < n; ++i) {
                const float* krow = k + (((size_t)bi * S + idx[i]) * H + h) * D;
                for (int d = 0; d < D; ++d) o[d] += scale * dS[i] * (double)krow[d];
            }
        }
        free(idx);
        free(P);
        free(dS);
    }
}

/*
 * dk, dv of explicit keys (batch, KV head h, position t): every row q >= t of
 * the G query heads that retains t contributes; each such row is solved in
 * full.  q, dO [b,S,Hq,D].  dk, dv [nkeys, D].
 */
void oracle_attn_bwd_keys(const float* q, const float* k, const float* v, const float* dO, int b,
                          int S, int H, int G, int D, double scale, const int32_t* rank,
                          const int32_t* tau, int s, int w, const int32_t* keys, int64_t nkeys,
                          double* dk, double* dv) {
    (void)b;
    int Hq = H * G;
#pragma omp parallel
    {
        int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
        double* P = (double*)malloc(sizeof(double) * (size_t)S);
        double* dS = (double*)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nkeys; ++i) {
            int bi = keys[3 * i + 0], h = keys[3 * i + 1], t = keys[3 * i + 2];
            const int32_t* rk = rank ? rank + ((size_t)bi * H + h) * S : NULL;
            const int32_t* tu = tau ? tau + ((size_t)bi * H + h) * S : NULL;
            double* ok = dk + (size_t)i * D;
            double* ov = dv + (size_t)i * D;
            for (int d = 0; d < D; ++d) ok[d] = ov[d] = 0.0;
            for (int qp = t; qp < S; ++qp) {
                if (rk && !retained(rk, tu, s, w, qp, t)) continue;
                for (int g = 0; g < G; ++g) {
                    size_t ro = (((size_t)bi * S + qp) * Hq + h * G + g) * D;
                    int n = row_grad(q + ro, dO + ro, k, v, bi, S, H, h, D, scale, rk, tu, s, w, qp, idx, P, dS);
                    for (int u = 0; u < n; ++u) {
                        if (idx[u] != t) continue;
                        for (int d = 0; d < D; ++d) {
                            ok[d] += scale * dS[u] * (double)q[ro + d];
                            ov[d] += P[u] * (double)dO[ro + d];
                        }
                    }
                }
            }
        }
        free(idx);
        free(P);
        free(dS);
    }
}

/* ------------------------------------------------------------------------ */
/* future-attention target                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Route B, Eq. (8) first term summed over the group:
 *   target[b,h,t] = log sum_{g<G} sum_{d=t+w}^{S-1} exp(scale*q_{d,hG+g}.k_t - LSE_{d,hG+g})
 * q [b,S,H*G,D], k [b,S,H,D], lse [b,H*G,S] (fp64; only rows d >= t+w are read).
 * keys [nkeys,3] = (batch index, KV head h, token t).
 */
void oracle_target_lse(const float* q, const float* k, const double* lse, int b, int S, int H, int G,
                       int D, double scale, int w, const int32_t* keys, int64_t nkeys,
                       double* target) {
    (void)b;
    int Hq = H * G;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < nkeys; ++i) {
        int bi = keys[3 * i + 0], h = keys[3 * i + 1], t = keys[3 * i + 2];
        const float* krow = k + (((size_t)bi * S + t) * H + h) * D;
        double sum = 0.0;
        for (int g = 0; g < G; ++g) {
            int j = h * G + g;
            for (int d = t + w; d < S; ++d) {
                const float* qrow = q + (((size_t)bi * S + d) * Hq + j) * D;
                sum += exp(scale * dot_f(qrow, krow, D) - lse[((size_t)bi * Hq + j) * S + d]);
            }
        }
        target[i] = sum > 0.0 ? log(sum) : -INFINITY;
    }
}

/*
 * Route A, the column sum of the attention map: materialise each dense causal
 * row A_{d,.} = softmax(scale * q_d . k_t, t <= d) and add A_{d,t} into
 * column t for every t <= d - w; target = log(column sum over d and g).
 * target [b,H,S].
 */
void oracle_target_colsum(const float* q, const float* k, int b, int S, int H, int G, int D,
                          double scale, int w, double* target) {
    int Hq = H * G;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < b * H; ++bh) {
        int bi = bh / H, h = bh % H;
        double* col = (double*)calloc((size_t)S, sizeof(double));
        double* l = (double*)malloc(sizeof(double) * (size_t)S);
        for (int g = 0; g < G; ++g) {
            int j = h * G + g;
            for (int d = 0; d < S; ++d) {
                const float* qrow = q + (((size_t)bi * S + d) * Hq + j) * D;
                double m = -INFINITY;
                for (int t = 0; t <= d; ++t) {
                    l[t] = scale * dot_f(qrow, k + (((size_t)bi * S + t) * H + h) * D, D);
                    if (l[t] > m) m = l[t];
                }
                double sum = 0.0;
                for (int t = 0; t <= d; ++t) sum += exp(l[t] - m);
                double L = m + log(sum);
                for (int t = 0; t <= d - w; ++t) col[t] += exp(l[t] - L);
            }
        }
        for (int t = 0; t < S; ++t)
            target[((size_t)bi * H + h) * S + t] = col[t] > 0.0 ? log(col[t]) : -INFINITY;
        free(col);
        free(l);
    }
}

/* ------------------------------------------------------------------------ */
/* normalised target, teacher boundary labels, pairwise boundary loss        */
/* ------------------------------------------------------------------------ */

/*
 * [KVpop notes] 2.2: m_t^g = (1/N_t) sum_{d=t+w}^{S-1} A_{d,t}^g and
 * r_t = log(eps + (1/G) sum_g m_t^g), with N_t = S - t - w future queries.
 * Input: the unnormalised target log sum_g sum_d A (fp64), [nbh, S].
 * A key with no future query (N_t <= 0) has mass 0: r = log(eps).
 */
void oracle_target_normalize(const double* target, int64_t nbh, int S, int G, int w, double eps,
                             double* r) {
    for (int64_t i = 0; i < nbh * (int64_t)S; ++i) {
        int t = (int)(i % S);
        int nt = S - t - w;
        double mass = nt > 0 ? exp(target[i]) / ((double)G * nt) : 0.0;
        double x = eps + mass;
        r[i] = x > 0.0 ? log(x) : -INFINITY;
    }
}

/* effective (decayed) score of token t at row q, [KVpop notes] 2.2:
 * r_t + floor((q - t) / n) * log_gamma, in fp32 with one rounding after the
 * product and one after the sum; NaN counts as -inf */
static float decayed(float r, int q, int t, int n, float lg) {
    float m = (float)((q - t) / n);
    float dec = m * lg;
    float sc = r + dec;
    return isnan(sc) ? -INFINITY : sc;
}

typedef struct {
    float v;
    int32_t idx;
} fkeyed_t;

/* (score desc, index asc) */
static int cmp_fkeyed(const void* a, const void* b) {
    const fkeyed_t* x = (const fkeyed_t*)a;
    const fkeyed_t* y = (const fkeyed_t*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

/*
 * Teacher boundary labels, [KVpop notes] 2.2: at row q the token
 * t_new = q - w leaves the window; the teacher ranks E(q) = {s..q-w} by the
 * decayed target score (ties: lower index first) and keeps its top k.
 *   t_bnd[q] = the k-th best token of E(q) minus t_new (the cutoff t_new has to
 *              beat; it is the lowest-scoring member of the teacher top-k whenever
 *              t_new is dropped); -1 if fewer than k other tokens;
 *   y[q]     = +1 if t_new is in the teacher top-k, -1 if not;
 *   rows without a leaving token (q - w < s) get y = 0, t_bnd = -1.
 * Sorting E(q) explicitly for every row: O(S^2 log S).
 */
void oracle_teacher_labels_rows(const float* r, int S, int s, int w, int k, int n, float lg,
                                const int32_t* rows, int nrows, int32_t* t_bnd, int32_t* y) {
#pragma omp parallel
    {
        fkeyed_t* buf = (fkeyed_t*)malloc(sizeof(fkeyed_t) * (size_t)(S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 16)
        for (int i = 0; i < nrows; ++i) {
            int q = rows[i];
            int tn = q - w;
            if (tn < s) {
                t_bnd[i] = -1;
                y[i] = 0;
                continue;
            }
            int m = 0;
            for (int t = s; t < tn; ++t) {
                buf[m].v = decayed(r[t], q, t, n, lg);
                buf[m].idx = t;
                ++m;
            }
            if (k == 0) {
                t_bnd[i] = -1;
                y[i] = -1;
                continue;
            }
            if (m < k) {
                t_bnd[i] = -1;
                y[i] = 1;
                continue;
            }
            qsort(buf, (size_t)m, sizeof(fkeyed_t), cmp_fkeyed);
            fkeyed_t me = {decayed(r[tn], q, tn, n, lg), tn};
            t_bnd[i] = buf[k - 1].idx;
            y[i] = cmp_fkeyed(&me, &buf[k - 1]) < 0 ? 1 : -1;
        }
        free(buf);
    }
}

/* every row q = 0..S-1 */
void oracle_teacher_labels(const float* r, int S, int s, int w, int k, int n, float lg, int32_t* t_bnd,
                           int32_t* y) {
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    for (int q = 0; q < S; ++q) rows[q] = q;
    oracle_teacher_labels_rows(r, S, s, w, k, n, lg, rows, S, t_bnd, y);
    free(rows);
}

static double softplus(double z) { return z > 0.0 ? z + log1p(exp(-z)) : log1p(exp(z)); }
static double sigmoid(double z) { return z >= 0.0 ? 1.0 / (1.0 + exp(-z)) : exp(z) / (1.0 + exp(z)); }

/*
 * Pairwise boundary loss, [KVpop notes] 2.2:
 *   L = mean over rows q with y[q] != 0 and t_bnd[q] >= 0 of
 *       omega[q] * softplus(-y[q] * (rh_new(q) - rh_bnd(q)) / tau),
 *   rh_t(q) = rhat[t] + floor((q - t) / n) * log_gamma[h]  (the decay applies to the
 *   predicted scores as to the targets), t_new = q - w.
 * rhat, omega (NULL = 1), t_bnd, y: [nbh, S] with h = row index mod H.
 * grad [nbh, S] = dL / drhat.  Returns the number of pairs; *loss = 0 when none.
 */
int64_t oracle_boundary_loss(const float* rhat, const int32_t* t_bnd, const int32_t* y, const float* omega,
                             int64_t nbh, int S, int H, int w, int n, const float* lg, double tau,
                             double* loss, double* grad) {
    int64_t pairs = 0;
    double sum = 0.0;
    for (int64_t i = 0; i < nbh * (int64_t)S; ++i) grad[i] = 0.0;
    for (int64_t bh = 0; bh < nbh; ++bh) {
        double l = (double)lg[bh % H];
        const float* rr = rhat + bh * S;
        for (int q = 0; q < S; ++q) {
            int64_t iq = bh * S + q;
            int tb = t_bnd[iq], yy = y[iq];
            if (yy == 0 || tb < 0) continue;
            int tn = q - w;
            double dn = (double)rr[tn] + (double)((q - tn) / n) * l;
            double db = (double)rr[tb] + (double)((q - tb) / n) * l;
            double z = -(double)yy * (dn - db) / tau;
            double om = omega ? (double)omega[iq] : 1.0;
            sum += om * softplus(z);
            double g = om * sigmoid(z) * (-(double)yy / tau);
            grad[bh * S + tn] += g;
            grad[bh * S + tb] -= g;
            ++pairs;
        }
    }
    if (pairs > 0)
        for (int64_t i = 0; i < nbh * (int64_t)S; ++i) grad[i] /= (double)pairs;
    *loss = pairs > 0 ? sum / (double)pairs : 0.0;
    return pairs;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
