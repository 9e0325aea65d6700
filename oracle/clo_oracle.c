/*
 * clo_oracle.c -- plain, slow, fp64 CPU oracle for the CLO decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the libclo CUDA
 * library and its Python binding) may include, link or call this file.  Only
 * the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * Every routine is the plain definition written out with loops in double
 * precision, in the order the method states it:
 *
 *   oracle_thresholds     "CLO: CPU-Light KVCache Offloading", section 2,
 *                         importance-aware adaptive threshold, Eqs. 7-9:
 *                         theta* = arccos(eta), lambda = s^n,
 *                         theta = lambda*theta* + (1-lambda)*pi, tau = cos(theta).
 *   oracle_lookup_update  same page, section 2, head-wise approximate cache
 *                         (hit iff cos(q, q_label) >= tau, otherwise the whole
 *                         head is replaced) and Eq. 10 (importance-weighted
 *                         mean of the group's query-head cosines gives one
 *                         scalar per KV head); section 3, Fig. 7 (an update
 *                         replaces the stored query vector).
 *   oracle_attention_dense  "KVPR: Efficient LLM Inference With I/O-Aware KV
 *                         Cache Partial Recomputation", section A3 (attention
 *                         softmax(Q K^T / sqrt(d_head)) V), two-pass softmax.
 *   oracle_hybrid_attn    CLO page, section 2, hybrid attention kernel: each
 *                         KV head group reads either the top-k Cache Buffer
 *                         (rows chosen by per-head token indices) or the
 *                         full-length Persistent Cache, with no gather first.
 *   oracle_paged_attn     "Neo: Saving GPU Memory Crisis with CPU Offloading
 *                         for Online LLM Inference", method details, system
 *                         implementation and CPU kernel (vLLM-like paged KV
 *                         cache, one decode query per request); same attention.
 *   oracle_plan_persistent  CLO page, section 3.3 and section 2 (selective
 *                         residency): reuse difficulty D_i = tau_i - (s^_i - eps)
 *                         (Eq. 11); the heads one layer's compute time can
 *                         prefetch, N_p = floor(T_comp * B_link / mem_head)
 *                         (Eq. 12); the heads of layer l kept resident,
 *                         N_persist^l = max(N_hard^l - N_p, 0) with N_hard^l the
 *                         heads of the layer with D_i > 0 (Eq. 13).
 *   oracle_topk_retrieve  CLO page, section 2, Eq. 6 (the qk-score ranking of
 *                         the keys does not depend on |q|) and the top-k
 *                         retrieval stage of the decode flow (section 3): the
 *                         k keys of each KV head with the largest score
 *                         against the group's queries.
 *   oracle_fill_cache_buffer  CLO page, section 3, Fig. 7 (an update writes
 *                         the new KV data straight to its final position, no
 *                         staging buffer) and section 2 (only missed heads
 *                         are transferred): for every KV head on the miss
 *                         list, copy the rows of its new top-k token set from
 *                         the full KV copy into the Cache Buffer rows that
 *                         the hybrid attention reads.
 *
 * Readings where the pages are silent:
 *   - GQA grouping is contiguous: query head h belongs to KV head h / G.
 *   - The threshold of a KV head uses the mean importance of its G query heads.
 *   - A zero-norm query or label has cosine 0.
 *   - If the importance weights of a group sum to zero, Eq. 10 falls back to
 *     the plain mean of the cosines.
 *   - sim == tau counts as a hit.
 *   - Persistent KV heads are not looked up: flag 2, labels untouched.
 *   - An empty token set gives output 0 and lse = -inf.
 *   - The final position of a filled row is the Cache Buffer row that the
 *     attention's index names for it; with token-addressed buffers that row
 *     is the token itself.
 *   - Eq. 12 as printed divides T_comp by B_link * mem_head, which is not
 *     dimensionless; the count of heads one layer can prefetch is taken as
 *     T_comp * B_link / mem_head, rounded down.
 *   - Top-k retrieval: the page names HATA hash scoring but gives no algorithm;
 *     the exact ranking is used.  A KV head's score of key t is the dot
 *     product of the sum of its G query vectors with K_t (the group's summed
 *     qk-score); the k largest are taken, equal scores at the cut going to
 *     the lower token index, and listed in ascending token order.
 *   - Of the hard heads (D_i > 0, strictly) of a layer, the N_persist^l with
 *     the largest D_i are kept resident (the rest are prefetched); equal D_i
 *     are taken in increasing head order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* Status codes of this oracle (its own, not the library's). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_INDEX 4

/* IEEE 754 binary16 -> double, from the format's definition:
 * sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Eqs. 7-9, one threshold per KV head.  s holds n_kv*group importance scores
 * (one per query head); the KV head's score is the mean over its group. */
void oracle_thresholds(const double* s, int n_kv, int group, double eta,
                       double n_exp, double* tau) {
    double theta_star = acos(eta); /* Eq. 7 */
    for (int g = 0; g < n_kv; ++g) {
        double sg = 0.0;
        for (int j = 0; j < group; ++j) sg += s[g * group + j];
        sg /= (double)group;
        double lam = pow(sg, n_exp);                             /* Eq. 8 */
        double theta = lam * theta_star + (1.0 - lam) * M_PI;    /* Eq. 9 */
        tau[g] = cos(theta);
    }
}

static double cosine_fp16(const uint16_t* a, const uint16_t* b, int d) {
    double ab = 0.0, aa = 0.0, bb = 0.0;
    for (int i = 0; i < d; ++i) {
        double x = oracle_half_to_double(a[i]);
        double y = oracle_half_to_double(b[i]);
        ab += x * y;
        aa += x * x;
        bb += y * y;
    }
    if (aa == 0.0 || bb == 0.0) return 0.0;
    return ab / (sqrt(aa) * sqrt(bb));
}

/* Head-wise approximate-cache lookup with Eq. 10 aggregation and label update.
 *   q, labels   [B][Hq][d] binary16 bit patterns; labels updated in place.
 *   w_q         [Hq] importance weights of the query heads.
 *   tau_kv      [Hkv] thresholds of the KV heads.
 *   persist     [Hkv] 1 = persistent KV head (may be NULL: none).
 *   flag        [B][Hkv]: 0 hit, 1 miss (labels replaced), 2 persistent.
 *   sim         [B][Hkv] aggregated similarity.
 *   cos_out     [B][Hq] per-query-head cosine (may be NULL).
 *   miss_list   ascending list of b*Hkv+g with flag 1; *miss_count entries. */
int oracle_lookup_update(const uint16_t* q, uint16_t* labels, const double* w_q,
                         const double* tau_kv, const uint8_t* persist, int B,
                         int Hq, int Hkv, int d, uint8_t* flag, double* sim,
                         double* cos_out, int32_t* miss_list,
                         int32_t* miss_count) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || B < 0) return ORACLE_BAD_ARG;
    int G = Hq / Hkv;
    int nmiss = 0;
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hkv; ++g) {
            double sw = 0.0, swc = 0.0, sc = 0.0;
            for (int j = 0; j < G; ++j) {
                int h = g * G + j;
                size_t off = ((size_t)b * Hq + h) * (size_t)d;
                double c = cosine_fp16(q + off, labels + off, d);
                if (cos_out) cos_out[(size_t)b * Hq + h] = c;
                sw += w_q[h];
                swc += w_q[h] * c;
                sc += c;
            }
            double s = (sw != 0.0) ? swc / sw : sc / (double)G; /* Eq. 10 */
            sim[(size_t)b * Hkv + g] = s;
            uint8_t f;
            if (persist && persist[g]) {
                f = 2;
            } else if (s >= tau_kv[g]) {
                f = 0;
            } else {
                f = 1;
                for (int j = 0; j < G; ++j) {
                    size_t off = ((size_t)b * Hq + g * G + j) * (size_t)d;
                    memcpy(labels + off, q + off, (size_t)d * sizeof(uint16_t));
                }
                miss_list[nmiss++] = b * Hkv + g;
            }
            flag[(size_t)b * Hkv + g] = f;
        }
    }
    *miss_count = nmiss;
    return ORACLE_OK;
}

/* softmax(q K^T * scale) V for G query rows over n key/value rows.
 * q [G][d], K/V [n][d] binary16; out [G][d], lse [G] (natural log of the
 * sum of exp(scaled scores)).  Two passes: scores and max, then weights. */
int oracle_attention_dense(const uint16_t* q, const uint16_t* K,
                           const uint16_t* V, int G, int n, int d,
                           double scale, double* out, double* lse) {
    if (G <= 0 || d <= 0 || n < 0) return ORACLE_BAD_ARG;
    if (n == 0) {
        for (int h = 0; h < G; ++h) {
            for (int i = 0; i < d; ++i) out[(size_t)h * d + i] = 0.0;
            lse[h] = -INFINITY;
        }
        return ORACLE_OK;
    }
    double* sc = (double*)malloc((size_t)n * sizeof(double));
    double* qd = (double*)malloc((size_t)d * sizeof(double));
    double* acc = (double*)malloc((size_t)d * sizeof(double));
    if (!sc || !qd || !acc) {
        free(sc); free(qd); free(acc);
        return ORACLE_BAD_ARG;
    }
    for (int h = 0; h < G; ++h) {
        for (int i = 0; i < d; ++i) qd[i] = oracle_half_to_double(q[(size_t)h * d + i]);
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
            double dot = 0.0;
            const uint16_t* kr = K + (size_t)t * d;
            for (int i = 0; i < d; ++i) dot += qd[i] * oracle_half_to_double(kr[i]);
            sc[t] = dot * scale;
            if (sc[t] > m) m = sc[t];
        }
        double l = 0.0;
        for (int i = 0; i < d; ++i) acc[i] = 0.0;
        for (int t = 0; t < n; ++t) {
            double p = exp(sc[t] - m);
            l += p;
            const uint16_t* vr = V + (size_t)t * d;
            for (int i = 0; i < d; ++i) acc[i] += p * oracle_half_to_double(vr[i]);
        }
        for (int i = 0; i < d; ++i) out[(size_t)h * d + i] = acc[i] / l;
        lse[h] = m + log(l);
    }
    free(sc); free(qd); free(acc);
    return ORACLE_OK;
}

/* Gathers the rows of one KV head's token set into contiguous K/V arrays. */
static int gather_rows(const uint16_t* srcK, const uint16_t* srcV,
                       const int32_t* rows, int n, int d, int nrows_src,
                       uint16_t* K, uint16_t* V) {
    for (int t = 0; t < n; ++t) {
        int r = rows ? rows[t] : t;
        if (r < 0 || r >= nrows_src) return ORACLE_BAD_INDEX;
        memcpy(K + (size_t)t * d, srcK + (size_t)r * d, (size_t)d * sizeof(uint16_t));
        memcpy(V + (size_t)t * d, srcV + (size_t)r * d, (size_t)d * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* Hybrid attention over the Cache Buffer and the Persistent Cache.
 *   q        [B][Hq][d]
 *   cbK/cbV  [B][Hkv][C][d]   Cache Buffer (slots of non-persistent heads)
 *   idx      [B][Hkv][k]      rows of the Cache Buffer each head attends to
 *   pK/pV    [B][Np][T][d]    Persistent Cache, slot j holds KV head persist_ids[j]
 *   out      [B][Hq][d], lse [B][Hq]
 * A KV head listed in persist_ids attends to all T persistent rows; every
 * other KV head attends to its k indexed Cache Buffer rows. */
int oracle_hybrid_attn(const uint16_t* q, const uint16_t* cbK,
                       const uint16_t* cbV, const int32_t* idx, int k, int C,
                       const uint16_t* pK, const uint16_t* pV,
                       const int32_t* persist_ids, int Np, int T, int B, int Hq,
                       int Hkv, int d, double scale, double* out, double* lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || B < 0 || k < 0 || k > C ||
        Np < 0 || Np > Hkv || T < 0)
        return ORACLE_BAD_ARG;
    int G = Hq / Hkv;
    size_t nmax = (size_t)(T > k ? T : k);
    uint16_t* K = (uint16_t*)malloc((nmax ? nmax : 1) * (size_t)d * sizeof(uint16_t));
    uint16_t* V = (uint16_t*)malloc((nmax ? nmax : 1) * (size_t)d * sizeof(uint16_t));
    if (!K || !V) { free(K); free(V); return ORACLE_BAD_ARG; }
    int rc = ORACLE_OK;
    for (int b = 0; b < B && rc == ORACLE_OK; ++b) {
        for (int g = 0; g < Hkv && rc == ORACLE_OK; ++g) {
            int slot = -1;
            for (int j = 0; j < Np; ++j)
                if (persist_ids[j] == g) slot = j;
            int n;
            if (slot >= 0) {
                size_t base = (((size_t)b * Np + slot) * (size_t)T) * d;
                rc = gather_rows(pK + base, pV + base, NULL, T, d, T, K, V);
                n = T;
            } else {
                size_t base = (((size_t)b * Hkv + g) * (size_t)C) * d;
                const int32_t* rows = idx + ((size_t)b * Hkv + g) * (size_t)k;
                rc = gather_rows(cbK + base, cbV + base, rows, k, d, C, K, V);
                n = k;
            }
            if (rc != ORACLE_OK) break;
            size_t qo = ((size_t)b * Hq + (size_t)g * G) * d;
            rc = oracle_attention_dense(q + qo, K, V, G, n, d, scale, out + qo,
                                        lse + (size_t)b * Hq + (size_t)g * G);
        }
    }
    free(K); free(V);
    return rc;
}

/* Paged decode attention, one query per request.
 *   q            [B][Hq][d]
 *   kc/vc        [num_blocks][Hkv][block_size][d]
 *   block_table  [B][max_blocks]; token t of request r lives in block
 *                block_table[r][t / block_size], row t % block_size.
 *   ctx_len      [B] number of tokens of each request. */
int oracle_paged_attn(const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                      const int32_t* block_table, int max_blocks,
                      const int32_t* ctx_len, int num_blocks, int B, int Hq,
                      int Hkv, int d, int block_size, double scale, double* out,
                      double* lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || B < 0 || block_size <= 0)
        return ORACLE_BAD_ARG;
    int G = Hq / Hkv;
    int nmax = max_blocks * block_size;
    uint16_t* K = (uint16_t*)malloc((size_t)(nmax ? nmax : 1) * d * sizeof(uint16_t));
    uint16_t* V = (uint16_t*)malloc((size_t)(nmax ? nmax : 1) * d * sizeof(uint16_t));
    if (!K || !V) { free(K); free(V); return ORACLE_BAD_ARG; }
    int rc = ORACLE_OK;
    for (int r = 0; r < B && rc == ORACLE_OK; ++r) {
        int n = ctx_len[r];
        if (n < 0 || n > nmax) { rc = ORACLE_BAD_INDEX; break; }
        for (int h = 0; h < Hkv && rc == ORACLE_OK; ++h) {
            for (int t = 0; t < n; ++t) {
                int blk = block_table[(size_t)r * max_blocks + t / block_size];
                if (blk < 0 || blk >= num_blocks) { rc = ORACLE_BAD_INDEX; break; }
                size_t src = (((size_t)blk * Hkv + h) * block_size + t % block_size) * d;
                memcpy(K + (size_t)t * d, kc + src, (size_t)d * sizeof(uint16_t));
                memcpy(V + (size_t)t * d, vc + src, (size_t)d * sizeof(uint16_t));
            }
            if (rc != ORACLE_OK) break;
            size_t qo = ((size_t)r * Hq + (size_t)h * G) * d;
            rc = oracle_attention_dense(q + qo, K, V, G, n, d, scale, out + qo,
                                        lse + (size_t)r * Hq + (size_t)h * G);
        }
    }
    free(K); free(V);
    return rc;
}

/* Miss-path fill of the Cache Buffer.
 *   srcK/srcV  [B][Hkv][T][d]  full KV copy of every head
 *   tok        [B][Hkv][k]     token of the j-th row of each head's new set
 *   slot       [B][Hkv][k]     its final row in the Cache Buffer; NULL means
 *                              the row is the token itself
 *   cbK/cbV    [B][Hkv][C][d]  Cache Buffer, written in place
 *   miss_list  [miss_count]    entries b * Hkv + g, one per missed KV head
 * Every row of a listed head is copied; rows of heads not on the list and
 * rows not selected are left as they are.  List entries outside [0, B*Hkv),
 * tokens outside [0, T) and slots outside [0, C) are skipped, the rest is
 * still done, and the call returns ORACLE_BAD_INDEX. */
int oracle_fill_cache_buffer(const uint16_t* srcK, const uint16_t* srcV, int T,
                             const int32_t* tok, const int32_t* slot, int k,
                             uint16_t* cbK, uint16_t* cbV, int C,
                             const int32_t* miss_list, int miss_count, int B,
                             int Hkv, int d) {
    if (B < 0 || Hkv <= 0 || d <= 0 || T < 0 || k < 0 || C < 0 || miss_count < 0)
        return ORACLE_BAD_ARG;
    int rc = ORACLE_OK;
    for (int m = 0; m < miss_count; ++m) {
        int e = miss_list[m];
        if (e < 0 || e >= B * Hkv) { rc = ORACLE_BAD_INDEX; continue; }
        for (int j = 0; j < k; ++j) {
            size_t sel = (size_t)e * k + j;
            int t = tok[sel];
            int r = slot ? slot[sel] : t;
            if (t < 0 || t >= T || r < 0 || r >= C) { rc = ORACLE_BAD_INDEX; continue; }
            size_t from = ((size_t)e * T + t) * d;
            size_t to = ((size_t)e * C + r) * d;
            memcpy(cbK + to, srcK + from, (size_t)d * sizeof(uint16_t));
            memcpy(cbV + to, srcV + from, (size_t)d * sizeof(uint16_t));
        }
    }
    return rc;
}

/* Offline persistent-head plan, Eqs. 11-13.
 *   tau, s_hat  [L][Hkv]  per-KV-head threshold and profiled mean cosine
 *   eps         tolerance margin of Eq. 11
 *   t_comp      one layer's compute time (s); b_link the host link's bandwidth
 *               (bytes/s); mem_head the top-k KV bytes of one head
 * Outputs: D [L][Hkv] (Eq. 11), *n_p (Eq. 12), n_persist [L] (Eq. 13) and
 * persist_ids [L][Hkv]: row l lists its n_persist[l] resident heads, largest
 * D first, then -1. */
int oracle_plan_persistent(const double* tau, const double* s_hat, int L, int Hkv,
                           double eps, double t_comp, double b_link, double mem_head,
                           double* D, int* n_p, int* n_persist, int* persist_ids) {
    if (L < 0 || Hkv <= 0 || !(mem_head > 0) || !(t_comp >= 0) || !(b_link >= 0))
        return ORACLE_BAD_ARG;
    double cap = floor(t_comp * b_link / mem_head); /* Eq. 12 */
    if (cap > 2147483647.0) cap = 2147483647.0;
    *n_p = (int)cap;
    for (int l = 0; l < L; ++l) {
        int hard = 0;
        for (int i = 0; i < Hkv; ++i) {
            size_t at = (size_t)l * Hkv + i;
            D[at] = tau[at] - (s_hat[at] - eps); /* Eq. 11 */
            if (D[at] > 0) ++hard;
            persist_ids[at] = -1;
        }
        int keep = hard - *n_p; /* Eq. 13 */
        if (keep < 0) keep = 0;
        n_persist[l] = keep;
        /* Pick the keep hardest heads one at a time: the largest D not yet
         * taken, the lower head index on a tie. */
        for (int j = 0; j < keep; ++j) {
            int best = -1;
            for (int i = 0; i < Hkv; ++i) {
                size_t at = (size_t)l * Hkv + i;
                if (!(D[at] > 0)) continue;
                int taken = 0;
                for (int u = 0; u < j; ++u)
                    if (persist_ids[(size_t)l * Hkv + u] == i) taken = 1;
                if (taken) continue;
                if (best < 0 || D[at] > D[(size_t)l * Hkv + best]) best = i;
            }
            persist_ids[(size_t)l * Hkv + j] = best;
        }
    }
    return ORACLE_OK;
}

/* Top-k retrieval by exact qk-score.
 *   q    [B][Hq][d]       queries (G = Hq / Hkv per KV head)
 *   K    [B][Hkv][T][d]   all keys of each KV head
 *   idx  [B][Hkv][k]      output: the selected tokens, ascending
 * score(t) = (sum of the group's q_h) . K_t in fp64; the k largest scores,
 * ties at the cut to the lower token index. */
static const double* g_topk_scores; /* for the comparator below */

static int by_score_then_index(const void* a, const void* b) {
    int i = *(const int*)a, j = *(const int*)b;
    double si = g_topk_scores[i], sj = g_topk_scores[j];
    if (si > sj) return -1;
    if (si < sj) return 1;
    return i < j ? -1 : (i > j);
}

static int by_index(const void* a, const void* b) {
    int i = *(const int*)a, j = *(const int*)b;
    return (i > j) - (i < j);
}

int oracle_topk_retrieve(const uint16_t* q, const uint16_t* K, int B, int Hq, int Hkv, int T,
                         int d, int k, int32_t* idx) {
    if (B < 0 || Hkv <= 0 || Hq % Hkv != 0 || T < 0 || d <= 0 || k < 0 || k > T)
        return ORACLE_BAD_ARG;
    int G = Hq / Hkv;
    double* qs = (double*)malloc((size_t)d * sizeof(double));
    double* sc = (double*)malloc((size_t)(T ? T : 1) * sizeof(double));
    int* order = (int*)malloc((size_t)(T ? T : 1) * sizeof(int));
    if (!qs || !sc || !order) { free(qs); free(sc); free(order); return ORACLE_BAD_ARG; }
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hkv; ++g) {
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int j = 0; j < G; ++j)
                    acc += oracle_half_to_double(q[((size_t)b * Hq + (size_t)g * G + j) * d + i]);
                qs[i] = acc;
            }
            const uint16_t* Kh = K + (((size_t)b * Hkv + g) * (size_t)T) * d;
            for (int t = 0; t < T; ++t) {
                double dot = 0.0;
                for (int i = 0; i < d; ++i)
                    dot += qs[i] * oracle_half_to_double(Kh[(size_t)t * d + i]);
                sc[t] = dot;
                order[t] = t;
            }
            g_topk_scores = sc;
            qsort(order, (size_t)T, sizeof(int), by_score_then_index);
            qsort(order, (size_t)k, sizeof(int), by_index);
            memcpy(idx + ((size_t)b * Hkv + g) * (size_t)k, order, (size_t)k * sizeof(int32_t));
        }
    }
    free(qs); free(sc); free(order);
    return ORACLE_OK;
}
