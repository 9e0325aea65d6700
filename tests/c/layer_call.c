/*
 * One decode layer through libclo's C ABI alone: a plain C host program with
 * no Python and no torch.  It runs clo_hybrid_decode_layer (the attention of
 * one layer, the next layer's miss-path fill beside it and the lookup of the
 * layer after in its merge launch; "CLO: CPU-Light KVCache Offloading",
 * section 3 Fig. 9) on seeded inputs and checks each part against the fp64
 * oracle (oracle/clo_oracle.c, linked as libclo_oracle.so):
 *   - the attention within 2e-3 max-abs and 1e-3 relative L2, lse within 1e-4;
 *   - the filled Cache Buffer bit for bit;
 *   - the lookup's flags, labels and miss list bit for bit (no group lies
 *     within 1e-4 of its threshold in these inputs; checked).
 * Exit status 0 when every check passes.  Test infrastructure only.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "clo.h"

/* The oracle's routines (oracle/clo_oracle.c). */
double oracle_half_to_double(uint16_t h);
void oracle_thresholds(const double* s, int n_kv, int group, double eta, double n_exp,
                       double* tau);
int oracle_lookup_update(const uint16_t* q, uint16_t* labels, const double* w_q,
                         const double* tau_kv, const uint8_t* persist, int B, int Hq, int Hkv,
                         int d, uint8_t* flag, double* sim, double* cos_out, int32_t* miss_list,
                         int32_t* miss_count);
int oracle_hybrid_attn(const uint16_t* q, const uint16_t* cbK, const uint16_t* cbV,
                       const int32_t* idx, int k, int C, const uint16_t* pK, const uint16_t* pV,
                       const int32_t* persist_ids, int Np, int T, int B, int Hq, int Hkv, int d,
                       double scale, double* out, double* lse);
int oracle_fill_cache_buffer(const uint16_t* srcK, const uint16_t* srcV, int T,
                             const int32_t* tok, const int32_t* slot, int k, uint16_t* cbK,
                             uint16_t* cbV, int C, const int32_t* miss_list, int miss_count, int B,
                             int Hkv, int d);

#define CHECK(x)                                                           \
    do {                                                                   \
        if (!(x)) {                                                        \
            fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #x); \
            return 1;                                                      \
        }                                                                  \
    } while (0)
#define CUDA(x)                                                                        \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "line %d: %s: %s\n", __LINE__, #x, cudaGetErrorString(e_)); \
            return 2;                                                                  \
        }                                                                              \
    } while (0)
#define CLO(x)                                                                          \
    do {                                                                                \
        clo_status s_ = (x);                                                            \
        if (s_ != CLO_OK) {                                                             \
            fprintf(stderr, "line %d: %s: %s\n", __LINE__, #x, clo_status_string(s_)); \
            return 3;                                                                   \
        }                                                                               \
    } while (0)

/* splitmix64 */
static uint64_t rng_state = 0x5EEDu;
static uint64_t next_u64(void) {
    uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static int below(int n) { return (int)(next_u64() % (uint64_t)n); }

/* A random binary16 of magnitude in [1/8, 1): random sign, biased exponent
 * 12..14, random fraction. */
static uint16_t rand_half(void) {
    uint64_t r = next_u64();
    uint16_t sign = (uint16_t)((r & 1u) << 15);
    uint16_t e = (uint16_t)(12 + (int)((r >> 1) % 3));
    uint16_t m = (uint16_t)((r >> 8) & 0x3ffu);
    return (uint16_t)(sign | (uint16_t)(e << 10) | m);
}

static uint16_t* rand_halves(size_t n) {
    uint16_t* a = (uint16_t*)malloc(n * sizeof(uint16_t));
    for (size_t i = 0; a != NULL && i < n; ++i) a[i] = rand_half();
    return a;
}

/* rows[h*k .. h*k+k) = k distinct values of [0, n) in random order, per head. */
static int32_t* distinct_rows(int heads, int n, int k) {
    int32_t* out = (int32_t*)malloc((size_t)heads * k * sizeof(int32_t));
    int32_t* perm = (int32_t*)malloc((size_t)n * sizeof(int32_t));
    if (out == NULL || perm == NULL) return NULL;
    for (int h = 0; h < heads; ++h) {
        for (int i = 0; i < n; ++i) perm[i] = i;
        for (int i = 0; i < k; ++i) { /* Fisher-Yates, first k places */
            int j = i + below(n - i);
            int32_t t = perm[i];
            perm[i] = perm[j];
            perm[j] = t;
            out[(size_t)h * k + i] = perm[i];
        }
    }
    free(perm);
    return out;
}

static void* to_device(const void* h, size_t bytes) {
    void* d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
    if (h != NULL) {
        if (cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    } else if (cudaMemset(d, 0, bytes) != cudaSuccess) {
        return NULL;
    }
    return d;
}

int main(void) {
    enum { B = 2, Hq = 32, Hkv = 8, D = 128, G = Hq / Hkv };
    /* Layer l: the attention (token-addressed Cache Buffer, 2 persistent heads). */
    const int T = 700, k = 70, C = 700, Np = 2;
    const int32_t pid[2] = {5, 2};
    /* Layer l+1: the fill (token-addressed, rows of five missed heads). */
    const int Tf = 500, kf = 50, Cf = 500;
    const int32_t fmiss[5] = {1, 4, 6, 11, 14};
    const int nfmiss = 5;
    /* Layer l+2: the lookup (KV head 3 persistent; s = 1 on even KV heads). */
    const double scale = 1.0 / sqrt((double)D);

    const size_t nq = (size_t)B * Hq * D, ncb = (size_t)B * Hkv * C * D;
    const size_t npc = (size_t)B * Np * T * D, nsrc = (size_t)B * Hkv * Tf * D;
    const size_t ncf = (size_t)B * Hkv * Cf * D;
    uint16_t *q = rand_halves(nq), *cbK = rand_halves(ncb), *cbV = rand_halves(ncb);
    uint16_t *pK = rand_halves(npc), *pV = rand_halves(npc);
    int32_t* idx = distinct_rows(B * Hkv, C, k);
    uint16_t *srcK = rand_halves(nsrc), *srcV = rand_halves(nsrc);
    uint16_t *cfK = rand_halves(ncf), *cfV = rand_halves(ncf);
    int32_t* tok = distinct_rows(B * Hkv, Tf, kf);
    uint16_t *q2 = rand_halves(nq), *lab2 = rand_halves(nq);
    CHECK(q && cbK && cbV && pK && pV && idx && srcK && srcV && cfK && cfV && tok && q2 && lab2);
    float s[Hq], tau[Hkv];
    double sd[Hq], taud[Hkv];
    for (int h = 0; h < Hq; ++h) {
        s[h] = ((h / G) % 2 == 0) ? 1.0f : 0.25f;
        sd[h] = s[h];
    }
    uint8_t pm2[Hkv] = {0, 0, 0, 1, 0, 0, 0, 0};

    /* Thresholds on the host, from the library and from the oracle. */
    CLO(clo_thresholds_host(s, Hkv, G, 0.8f, 3.0f, tau));
    oracle_thresholds(sd, Hkv, G, 0.8, 3.0, taud);
    for (int g = 0; g < Hkv; ++g) {
        CHECK(fabs((double)tau[g] - taud[g]) < 1e-6);
        taud[g] = (double)tau[g]; /* the lookup compares against the same fp32 tau */
    }

    /* Device buffers. */
    void *dq = to_device(q, nq * 2), *dcbK = to_device(cbK, ncb * 2), *dcbV = to_device(cbV, ncb * 2);
    void *didx = to_device(idx, (size_t)B * Hkv * k * 4), *dpK = to_device(pK, npc * 2);
    void *dpV = to_device(pV, npc * 2), *dpid = to_device(pid, sizeof(pid));
    void *dsrcK = to_device(srcK, nsrc * 2), *dsrcV = to_device(srcV, nsrc * 2);
    void *dcfK = to_device(cfK, ncf * 2), *dcfV = to_device(cfV, ncf * 2);
    void* dtok = to_device(tok, (size_t)B * Hkv * kf * 4);
    int32_t fml_host[B * Hkv];
    for (int i = 0; i < B * Hkv; ++i) fml_host[i] = i < nfmiss ? fmiss[i] : -1;
    const int32_t fcount = nfmiss;
    void *dfml = to_device(fml_host, sizeof(fml_host)), *dfmc = to_device(&fcount, 4);
    void *dq2 = to_device(q2, nq * 2), *dlab2 = to_device(lab2, nq * 2);
    void *dw = to_device(s, sizeof(s)), *dtau = to_device(tau, sizeof(tau));
    void* dpm2 = to_device(pm2, sizeof(pm2));
    void *dflag = to_device(NULL, B * Hkv), *dsim = to_device(NULL, B * Hkv * 4);
    void *dml = to_device(NULL, B * Hkv * 4), *dmc = to_device(NULL, 4);
    void *dout = to_device(NULL, nq * 2), *dlse = to_device(NULL, (size_t)B * Hq * 4);
    const size_t ws_bytes = clo_hybrid_workspace_size(B, Hq, Hkv, D, 0);
    void *dws = to_device(NULL, ws_bytes), *derr = to_device(NULL, 4);
    CHECK(ws_bytes > 0 && dq && dcbK && dcbV && didx && dpK && dpV && dpid && dsrcK && dsrcV);
    CHECK(dcfK && dcfV && dtok && dfml && dfmc && dq2 && dlab2 && dw && dtau && dpm2 && dflag);
    CHECK(dsim && dml && dmc && dout && dlse && dws && derr);

    /* The layer call. */
    clo_fill_args fa;
    memset(&fa, 0, sizeof fa);
    fa.srcK = (const clo_half*)dsrcK;
    fa.srcV = (const clo_half*)dsrcV;
    fa.T = Tf;
    fa.tok = (const int32_t*)dtok;
    fa.slot = NULL; /* token-addressed */
    fa.k = kf;
    fa.cbK = (clo_half*)dcfK;
    fa.cbV = (clo_half*)dcfV;
    fa.C = Cf;
    fa.miss_list = (const int32_t*)dfml;
    fa.miss_count = (const int32_t*)dfmc;
    fa.num_ctas = 0;
    clo_lookup_args la;
    la.q = (const clo_half*)dq2;
    la.labels = (clo_half*)dlab2;
    la.w_q = (const float*)dw;
    la.tau = (const float*)dtau;
    la.persist_mask = (const uint8_t*)dpm2;
    la.flag = (uint8_t*)dflag;
    la.sim = (float*)dsim;
    la.miss_list = (int32_t*)dml;
    la.miss_count = (int32_t*)dmc;
    CLO(clo_hybrid_decode_layer((const clo_half*)dq, (const clo_half*)dcbK, (const clo_half*)dcbV,
                                (const int32_t*)didx, k, C, (const clo_half*)dpK,
                                (const clo_half*)dpV, (const int32_t*)dpid, Np, T, B, Hq, Hkv, D,
                                (float)scale, (clo_half*)dout, (float*)dlse, dws, ws_bytes,
                                (int32_t*)derr, &fa, &la, NULL, 0));
    CUDA(cudaDeviceSynchronize());
    int32_t err = -1;
    CUDA(cudaMemcpy(&err, derr, 4, cudaMemcpyDeviceToHost));
    CHECK(clo_check_error_flag(err) == CLO_OK);

    /* The attention of layer l. */
    uint16_t* out = (uint16_t*)malloc(nq * 2);
    float* lse = (float*)malloc((size_t)B * Hq * 4);
    double* ref = (double*)malloc(nq * sizeof(double));
    double* ref_lse = (double*)malloc((size_t)B * Hq * sizeof(double));
    CHECK(out && lse && ref && ref_lse);
    CUDA(cudaMemcpy(out, dout, nq * 2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(lse, dlse, (size_t)B * Hq * 4, cudaMemcpyDeviceToHost));
    CHECK(oracle_hybrid_attn(q, cbK, cbV, idx, k, C, pK, pV, pid, Np, T, B, Hq, Hkv, D, scale,
                             ref, ref_lse) == 0);
    double max_err = 0.0, num = 0.0, den = 0.0, lse_err = 0.0;
    for (size_t i = 0; i < nq; ++i) {
        double e = fabs(oracle_half_to_double(out[i]) - ref[i]);
        max_err = e > max_err ? e : max_err;
        num += e * e;
        den += ref[i] * ref[i];
    }
    for (int i = 0; i < B * Hq; ++i) {
        double e = fabs((double)lse[i] - ref_lse[i]);
        lse_err = e > lse_err ? e : lse_err;
    }
    CHECK(max_err <= 2e-3 && sqrt(num / den) <= 1e-3 && lse_err < 1e-4);

    /* The fill of layer l+1, bit for bit. */
    uint16_t *gK = (uint16_t*)malloc(ncf * 2), *gV = (uint16_t*)malloc(ncf * 2);
    CHECK(gK && gV);
    CUDA(cudaMemcpy(gK, dcfK, ncf * 2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(gV, dcfV, ncf * 2, cudaMemcpyDeviceToHost));
    CHECK(oracle_fill_cache_buffer(srcK, srcV, Tf, tok, NULL, kf, cfK, cfV, Cf, fmiss, nfmiss, B,
                                   Hkv, D) == 0);
    CHECK(memcmp(gK, cfK, ncf * 2) == 0 && memcmp(gV, cfV, ncf * 2) == 0);

    /* The lookup of layer l+2, bit for bit. */
    uint8_t flag[B * Hkv], rflag[B * Hkv];
    int32_t ml[B * Hkv], rml[B * Hkv], mc = -1, rmc = -1;
    float sim[B * Hkv];
    double rsim[B * Hkv];
    uint16_t* glab = (uint16_t*)malloc(nq * 2);
    CHECK(glab != NULL);
    CUDA(cudaMemcpy(flag, dflag, sizeof(flag), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(sim, dsim, sizeof(sim), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(ml, dml, sizeof(ml), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&mc, dmc, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(glab, dlab2, nq * 2, cudaMemcpyDeviceToHost));
    CHECK(oracle_lookup_update(q2, lab2, sd, taud, pm2, B, Hq, Hkv, D, rflag, rsim, NULL, rml,
                               &rmc) == 0);
    for (int i = 0; i < B * Hkv; ++i) {
        if (rflag[i] != 2) CHECK(fabs(rsim[i] - taud[i % Hkv]) > 1e-4);
        CHECK(flag[i] == rflag[i] && fabs((double)sim[i] - rsim[i]) < 1e-5);
    }
    CHECK(mc == rmc && mc > 0 && mc < B * Hkv);
    CHECK(memcmp(ml, rml, (size_t)mc * sizeof(int32_t)) == 0);
    CHECK(memcmp(glab, lab2, nq * 2) == 0);

    printf("layer call from C: attention max err %.2e, rel L2 %.2e; %d filled heads bit-exact; "
           "%d lookup misses exact\n", max_err, sqrt(num / den), nfmiss, mc);
    return 0;
}
