/*
 * clo.h -- C ABI of libclo, the GB300 (sm_103a) decode-attention hot path of
 * CPU-light KV-cache offloading.
 *
 * The operations follow "CLO: CPU-Light KVCache Offloading" (section 2 and
 * section 4): per-head similarity thresholds (Eqs. 7-9), the fused head-wise
 * approximate-cache lookup with GQA aggregation (Eq. 10) and query-label
 * update, and the hybrid attention kernel that reads the top-k Cache Buffer
 * and the full-length Persistent Cache directly.  A plain paged decode
 * attention serves the many-request case of "Neo: Saving GPU Memory Crisis
 * with CPU Offloading for Online LLM Inference" (method details: paged KV
 * cache, one decode attention launch per iteration) and "FastDecode" (R-Part
 * attention over per-request KV).  The attention itself is
 * softmax(q K^T / sqrt(d_head)) V as written in "KVPR: Efficient LLM
 * Inference With I/O-Aware KV Cache Partial Recomputation", section A3.
 * Around them: the miss-path fill that writes missed heads' top-k rows into
 * the Cache Buffer (CLO section 3, Fig. 7), the offline persistent-head plan
 * (CLO Eqs. 11-13), the next layer's lookup carried in an attention launch
 * and one layer of the decode flow in one call, with the next layer's fill
 * beside the attention (CLO section 3, Fig. 9), top-k retrieval by exact
 * qk-score (CLO Eq. 6) and the GPU-centric data-ready synchronisation with a
 * bounded wait (CLO section 2, Fig. 8).
 *
 * Conventions shared by every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller (unless a call
 *    states otherwise), row-major and contiguous in the layouts stated per
 *    call.  fp16 data is IEEE binary16
 *    (clo_half holds the bit pattern).  The library never allocates or frees
 *    device memory; scratch space is caller-provided ("workspace").
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *    return after the launches are enqueued.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns CLO_ERR_INVALID_ARG (or CLO_ERR_UNSUPPORTED for a shape
 *    this build does not implement, CLO_ERR_WORKSPACE for a short workspace)
 *    and launches nothing.  A failed launch returns CLO_ERR_CUDA.
 *  - Data-dependent errors (an index, block-table entry, context length or
 *    persistent-head id out of range) are detected on the device: the kernel
 *    ORs a CLO_FLAG_* bit into *err_flag (a caller-zeroed int32 in device
 *    memory; may be NULL), skips the bad rows, and writes zeros (lse = -inf)
 *    for the affected query heads.  The caller copies err_flag back after the
 *    stream synchronises and maps it with clo_check_error_flag().  No kernel
 *    traps.
 *  - Query head h belongs to KV head h / G with G = Hq / Hkv (contiguous
 *    grouping).  d (head dimension) must be 128 in this build.
 *  - No C++ exception crosses this interface.  There is no global mutable
 *    state besides cached device attributes (and the fixed scratch of
 *    clo_hybrid_decode_attn_noalloc), so independent calls on different
 *    streams may run concurrently provided they do not share output or
 *    workspace buffers.
 */
#ifndef CLO_H_
#define CLO_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t clo_half; /* IEEE binary16 bit pattern */

typedef enum clo_status {
    CLO_OK = 0,
    CLO_ERR_INVALID_ARG = 1,
    CLO_ERR_UNSUPPORTED = 2,
    CLO_ERR_CUDA = 3,
    CLO_ERR_BAD_INDEX = 4,
    CLO_ERR_WORKSPACE = 5,
    CLO_ERR_TIMEOUT = 6
} clo_status;

/* Bits a kernel ORs into *err_flag. */
#define CLO_FLAG_BAD_INDEX 0x1   /* Cache Buffer index, block-table entry, or a fill's
                                    miss-list entry, token or slot out of range */
#define CLO_FLAG_BAD_PERSIST 0x2 /* persist_ids entry out of range or repeated */
#define CLO_FLAG_BAD_CTX 0x4     /* a context length < 0 or > max_blocks*block_size */
#define CLO_FLAG_TIMEOUT 0x8     /* clo_wait_ready gave up before the value arrived */

/* Human-readable name of a status code (static storage, never NULL). */
const char* clo_status_string(clo_status s);

/* Library version, major*10000 + minor*100 + patch. */
int clo_version(void);

/* Maps an err_flag value copied back to the host to a status: CLO_OK when
 * zero, CLO_ERR_TIMEOUT when CLO_FLAG_TIMEOUT is set, else CLO_ERR_BAD_INDEX
 * when any other CLO_FLAG_* bit is set. */
clo_status clo_check_error_flag(int32_t host_err_flag);

/* One copy of `bytes` bytes from src to dst. */
typedef struct clo_copy {
    void* dst;
    const void* src;
    size_t bytes;
} clo_copy;

/*
 * clo_copy_async -- makes the copies copies[0..n) on `stream`, so a caller
 * that holds a step's inputs or results in host memory moves them with one
 * call instead of one per buffer.  The pages have no counterpart: it is the
 * host-buffer edge of this library, and nothing in it computes.
 *  - Copies between memory the GPU can address (device or managed memory,
 *    pinned host memory) are made by a libclo kernel, up to 16 of them a
 *    launch, when both ends are 16-byte aligned (any length) or the copy is at
 *    most 64 KiB; the SMs read and write host memory over the host link.  That
 *    kernel chains with the libclo kernels before and after it like they chain
 *    with each other.  Any other copy is one cudaMemcpyAsync (pageable host
 *    memory makes that wait for the copy).
 *  - The copies of one call may run at the same time: a list in which one
 *    copy writes bytes that another reads or writes (or a copy onto itself)
 *    gives CLO_ERR_INVALID_ARG (checked on the host in O(n log n)).  Calls are
 *    ordered on the stream as usual.
 *  - The caller keeps every buffer alive and unchanged until the stream
 *    reaches the copy.
 *  - Copies with bytes == 0 are skipped.  n < 0, copies == NULL with n > 0,
 *    or a NULL dst/src in a non-empty copy give CLO_ERR_INVALID_ARG before
 *    anything is issued; a failed launch or cudaMemcpyAsync gives
 *    CLO_ERR_CUDA (the copies before it stay issued).
 */
clo_status clo_copy_async(const clo_copy* copies, int n, cudaStream_t stream);

/*
 * clo_thresholds -- per-KV-head similarity thresholds, CLO Eqs. 7-9:
 *     theta* = arccos(eta), lambda = s^n, theta = lambda*theta* + (1-lambda)*pi,
 *     tau = cos(theta).
 * s:    [n_kv * group] fp32 importance scores of the query heads (device).
 *       KV head g uses the mean of s[g*group .. g*group+group-1]; with
 *       group = 1 the map is elementwise.
 * tau:  [n_kv] fp32 output (device).
 * eta:  global similarity bound, in [-1, 1] (the page uses 0.8).
 * n_exp: importance exponent n >= 0 (the page uses 3).
 * Computed in fp32 with the CUDA math library (acosf, powf, cosf).
 */
clo_status clo_thresholds(const float* s, int n_kv, int group, float eta,
                          float n_exp, float* tau, cudaStream_t stream);

/*
 * clo_thresholds_host -- the same thresholds (CLO Eqs. 7-9), computed on the
 * host for callers that set tau once per model or configuration and keep it:
 * s and tau are HOST arrays ([n_kv * group] and [n_kv] fp32), the call is
 * synchronous and touches no GPU.  fp32 arithmetic in the kernel's order (the
 * group mean of s, then Eqs. 7-9 with the host C library's acosf, powf,
 * cosf); it agrees with clo_thresholds and with the fp64 definition within
 * 1e-6.  Same argument rules as clo_thresholds (n_kv == 0 is a no-op).
 */
clo_status clo_thresholds_host(const float* s, int n_kv, int group, float eta, float n_exp,
                               float* tau);

/*
 * clo_lookup_update -- fused head-wise approximate-cache lookup and query-label
 * update (CLO section 2 "head-wise approximate cache" and "fused cache lookup
 * + query label update kernel"; Eq. 10; section 3 Fig. 7).  One launch reads
 * the incoming queries and the stored labels once:
 *     c_h   = q_h . l_h / (|q_h| |l_h|)            (0 if either norm is 0)
 *     sim_g = sum_{h in g} w_h c_h / sum_{h in g} w_h   (plain mean if the
 *             weights of the group sum to 0)                        Eq. 10
 *     hit_g = sim_g >= tau_g
 * On a miss the G labels of the group are overwritten with the G current
 * queries (bit copies) and the head is flagged 1; a hit leaves them (flag 0);
 * a persistent KV head is not cached (flag 2, labels untouched).
 * q:          [B][Hq][d] fp16 (device, read).
 * labels:     [B][Hq][d] fp16 (device, read and updated in place).
 * w_q:        [Hq] fp32 importance weights of the query heads.
 * tau_kv:     [Hkv] fp32 thresholds (e.g. from clo_thresholds).
 * persist_mask: [Hkv] uint8, nonzero = persistent; may be NULL (none).
 * flag:       [B][Hkv] uint8 output.      sim: [B][Hkv] fp32 output.
 * miss_list:  [B*Hkv] int32 output: b*Hkv+g of every miss, ascending.
 * miss_count: [1] int32 output: number of misses.
 * Requires Hq % Hkv == 0, G = Hq/Hkv <= 8, d == 128, 0 <= B*Hkv <= 65536.
 */
clo_status clo_lookup_update(const clo_half* q, clo_half* labels,
                             const float* w_q, const float* tau_kv,
                             const uint8_t* persist_mask, int B, int Hq,
                             int Hkv, int d, uint8_t* flag, float* sim,
                             int32_t* miss_list, int32_t* miss_count,
                             cudaStream_t stream);

/*
 * clo_plan_persistent -- offline persistent-head plan (CLO section 3.3 and
 * section 2, selective residency; Eqs. 11-13).  Host function, no GPU work.
 *     D_i         = tau_i - (s^_i - eps)                          Eq. 11
 *     N_p         = floor(t_comp * link_bytes_per_s / head_bytes) Eq. 12
 *     N_persist^l = max(#{i in layer l : D_i > 0} - N_p, 0)       Eq. 13
 * (Eq. 12 as printed divides T_comp by B_link * mem_head, which is not
 * dimensionless; the number of heads whose top-k rows one layer's compute
 * time can bring over the link is taken.)  Layer l keeps its N_persist^l
 * hardest heads resident (largest D first, ties to the lower head index):
 * these are its persist_ids for clo_hybrid_decode_attn and its persistent
 * mask for clo_lookup_update.
 * tau, s_hat:  [L][Hkv] host fp32: thresholds (e.g. clo_thresholds) and the
 *              offline-profiled mean query cosine of each KV head.
 * eps:         tolerance margin (the page uses 0.1 for Llama3, 0.05 for Qwen2.5).
 * t_comp_s:    one layer's compute time (s); link_bytes_per_s: host-link
 *              bandwidth; head_bytes: top-k K+V bytes of one head (> 0).
 * D:           [L][Hkv] host fp64 output (computed in fp64 from the inputs).
 * n_p:         [1] output.  n_persist: [L] output.
 * persist_ids: [L][Hkv] output; row l holds its n_persist[l] heads, then -1.
 */
clo_status clo_plan_persistent(const float* tau, const float* s_hat, int L, int Hkv,
                               float eps, double t_comp_s, double link_bytes_per_s,
                               double head_bytes, double* D, int32_t* n_p,
                               int32_t* n_persist, int32_t* persist_ids);

/* Optional tuning and instrumentation for the attention and fill calls (may
 * be NULL).  Events recorded while `stream` is being captured into a CUDA
 * graph become external event nodes, so they can time replays. */
typedef struct clo_attn_opts {
    int num_ctas;         /* CTAs of the main kernel; 0 = the default (one full wave) */
    cudaEvent_t ev_begin; /* if non-NULL, recorded on `stream` right before the main kernel */
    cudaEvent_t ev_end;   /* if non-NULL, recorded right after the main kernel */
} clo_attn_opts;

/*
 * clo_fill_cache_buffer -- miss-path fill of the Cache Buffer (CLO section 3
 * Fig. 7: an update writes the new KV data straight to its final position,
 * with no staging buffer and no second copy; section 2: only the KV heads
 * that missed are transferred).  For every entry e = b*Hkv + g of
 * miss_list[0 .. *miss_count) and every j < k:
 *     cbK[e][slot[e][j]] = srcK[e][tok[e][j]]   (and the same for V)
 * srcK, srcV: [B][Hkv][T][d] fp16, the full KV copy.  Either device memory or
 *             pinned host memory mapped into the device's address space
 *             (cudaHostAlloc, a pinned torch tensor): the kernel then reads
 *             the rows in place over the host link (NVLink-C2C on GB300).
 *             Other host memory is accepted only where the device can read
 *             pageable memory; a source the device cannot read gives
 *             CLO_ERR_INVALID_ARG and nothing is launched.
 * tok:        [B][Hkv][k] int32 (device): token of the j-th row of each
 *             head's new top-k set.
 * slot:       [B][Hkv][k] int32 (device): its row in the Cache Buffer, i.e.
 *             the index the hybrid attention will read it through; NULL
 *             means slot = tok (token-addressed buffer, requires C >= T).
 *             The slots of one head must be distinct.
 * cbK, cbV:   [B][Hkv][C][d] fp16 (device), written in place; rows of heads
 *             not on the list and rows not named by a slot are not touched.
 * miss_list, miss_count: device arrays as written by clo_lookup_update (the
 *             count is read on the device; the call does not synchronise).
 * err_flag:   optional (device).  A list entry outside [0, B*Hkv), a token
 *             outside [0, T) or a slot outside [0, C) sets CLO_FLAG_BAD_INDEX
 *             and that row (or head) is skipped; a count outside [0, B*Hkv]
 *             sets it and is clamped.
 * opts:       optional (see clo_attn_opts).  num_ctas sets the fill's grid
 *             (default: one wave of 4 CTAs an SM).  A fill CTA (4 warps, no
 *             shared memory, at most 128 registers a thread) takes no more
 *             room on an SM than an attention CTA, so a fill of N CTAs can run
 *             on a second stream beside an attention launched with N fewer
 *             CTAs than its default grid (3 an SM): the next layer's missed
 *             rows then move while this layer's attention runs.
 * Requires d == 128; pointers to K/V 16-byte aligned.
 */
clo_status clo_fill_cache_buffer(const clo_half* srcK, const clo_half* srcV, int T,
                                 const int32_t* tok, const int32_t* slot, int k,
                                 clo_half* cbK, clo_half* cbV, int C,
                                 const int32_t* miss_list, const int32_t* miss_count,
                                 int B, int Hkv, int d, int32_t* err_flag,
                                 const clo_attn_opts* opts, cudaStream_t stream);

/*
 * clo_topk_retrieve -- top-k retrieval by exact qk-score (CLO section 2,
 * Eq. 6: the ranking of keys by q . k does not depend on |q|; the decode
 * flow's top-k retrieval stage, which the page runs with HATA hashing and no
 * stated algorithm, so the exact ranking is computed).  For each batch row b
 * and KV head g:
 *     score(t) = (sum of the group's query vectors q_h) . K_t   (fp32)
 * and idx[b][g] receives the k tokens with the largest score, equal scores at
 * the cut going to the lower token, in ascending token order.
 * q:         [B][Hq][d] fp16 (device).     K: [B][Hkv][T][d] fp16 (device).
 * idx:       [B][Hkv][k] int32 output (device), e.g. the Cache Buffer index of
 *            a token-addressed buffer.
 * workspace: >= clo_topk_workspace_size(B, Hkv, T) bytes, 16-byte aligned
 *            (the scores).
 * opts:      optional; the events bracket the scoring kernel.
 * Requires 0 <= k <= T <= 385024, d == 128, G <= 8, B*Hkv <= 65535.
 */
size_t clo_topk_workspace_size(int B, int Hkv, int T);
clo_status clo_topk_retrieve(const clo_half* q, const clo_half* K, int B, int Hq, int Hkv,
                             int T, int d, int k, int32_t* idx, void* workspace,
                             size_t ws_bytes, const clo_attn_opts* opts,
                             cudaStream_t stream);

/*
 * Workspace bytes clo_hybrid_decode_attn needs for these sizes when run with
 * num_ctas CTAs (0 = the default grid on the current device).  Returns 0 for
 * invalid sizes.  The workspace holds split-KV partial results; it needs no
 * initialisation and may be reused by later calls on the same stream.
 */
size_t clo_hybrid_workspace_size(int B, int Hq, int Hkv, int d, int num_ctas);

/*
 * clo_hybrid_decode_attn -- GQA decode attention that reads the top-k Cache
 * Buffer and the Persistent Cache in place (CLO section 2 "hybrid attention
 * kernel", section 3 Fig. 9), with no gather into a unified buffer.
 * For each batch row b and KV head g the attended token set is
 *   - all T rows of Persistent Cache slot j if persist_ids[j] == g, else
 *   - the k Cache Buffer rows idx[b][g][0..k-1] of head g.
 * For every query head h of the group:
 *   o_h = sum_t softmax_t(scale * q_h . K_t) V_t,  lse_h = log sum_t exp(scale * q_h . K_t).
 * Split-KV over all SMs with a log-sum-exp merge; fp16 inputs, fp32
 * accumulation, fp16 output rounded to nearest.
 * q:           [B][Hq][d] fp16.
 * cbK, cbV:    [B][Hkv][C][d] fp16 Cache Buffer (slots of persistent heads unused).
 * idx:         [B][Hkv][k] int32 rows in [0, C); any order, duplicates allowed.
 * pK, pV:      [B][Np][T][d] fp16 Persistent Cache; may be NULL when Np == 0.
 * persist_ids: [Np] int32 distinct KV heads in [0, Hkv); may be NULL when Np == 0.
 * out:         [B][Hq][d] fp16 output.    lse: [B][Hq] fp32 output or NULL.
 * workspace:   >= clo_hybrid_workspace_size(B, Hq, Hkv, d, num_ctas) bytes,
 *              16-byte aligned.
 * Requires k >= 1 unless every KV head is persistent, T >= 1 when Np > 0,
 * k <= C, 0 <= Np <= Hkv, G <= 8, d == 128.
 */
clo_status clo_hybrid_decode_attn(const clo_half* q, const clo_half* cbK,
                                  const clo_half* cbV, const int32_t* idx,
                                  int k, int C, const clo_half* pK,
                                  const clo_half* pV,
                                  const int32_t* persist_ids, int Np, int T,
                                  int B, int Hq, int Hkv, int d, float scale,
                                  clo_half* out, float* lse, void* workspace,
                                  size_t ws_bytes, int32_t* err_flag,
                                  const clo_attn_opts* opts,
                                  cudaStream_t stream);

/*
 * clo_hybrid_decode_attn_lookup -- clo_hybrid_decode_attn for layer l and
 * clo_lookup_update for the next layer in one launch sequence (CLO section 3
 * Fig. 9: the next layer's lookup runs while the current layer computes; the
 * separate lookup launch of each layer is saved, CLO section 5's concern with
 * launch overhead).  The results are those of the two calls made separately
 * (the lookup reads nothing the attention writes).  The lookup runs as one
 * 8-CTA cluster while the main attention kernel drains: for up to 64
 * (batch row, KV head) groups inside the attention's merge launch, for more in
 * a launch of its own right after the main kernel.
 * Arguments up to err_flag: as clo_hybrid_decode_attn.  q_next .. miss_count_next:
 * as clo_lookup_update for the next layer (same B, Hq, Hkv, d).  opts: as for
 * clo_hybrid_decode_attn.
 */
clo_status clo_hybrid_decode_attn_lookup(
    const clo_half* q, const clo_half* cbK, const clo_half* cbV, const int32_t* idx, int k, int C,
    const clo_half* pK, const clo_half* pV, const int32_t* persist_ids, int Np, int T, int B,
    int Hq, int Hkv, int d, float scale, clo_half* out, float* lse, void* workspace,
    size_t ws_bytes, int32_t* err_flag, const clo_half* q_next, clo_half* labels_next,
    const float* w_q_next, const float* tau_next, const uint8_t* persist_mask_next,
    uint8_t* flag_next, float* sim_next, int32_t* miss_list_next, int32_t* miss_count_next,
    const clo_attn_opts* opts, cudaStream_t stream);

/* The next layer's miss-path fill carried by clo_hybrid_decode_layer.  Fields
 * as the arguments of clo_fill_cache_buffer with the same names (the batch,
 * KV heads and head dimension are the layer call's B, Hkv and d). */
typedef struct clo_fill_args {
    const clo_half* srcK;
    const clo_half* srcV;
    int T;
    const int32_t* tok;
    const int32_t* slot;
    int k;
    clo_half* cbK;
    clo_half* cbV;
    int C;
    const int32_t* miss_list;
    const int32_t* miss_count;
    int num_ctas; /* CTAs of the fill; 0 = a quarter of the default attention grid's slots,
                     at most as many as the longest possible miss list keeps busy */
} clo_fill_args;

/* A lookup carried by clo_hybrid_decode_layer.  Fields as the arguments of
 * clo_lookup_update with the same names (tau = tau_kv; B, Hq, Hkv and d are
 * the layer call's). */
typedef struct clo_lookup_args {
    const clo_half* q;
    clo_half* labels;
    const float* w_q;
    const float* tau;
    const uint8_t* persist_mask;
    uint8_t* flag;
    float* sim;
    int32_t* miss_list;
    int32_t* miss_count;
} clo_lookup_args;

/*
 * clo_hybrid_decode_layer -- one layer of CLO's decode flow as one call on
 * one stream (CLO section 3, Fig. 9: the lookup for a layer runs a layer
 * ahead of its attention, with an approximate query, and the missed heads'
 * rows move while the layer before it computes).  For layer l it runs
 *   - clo_hybrid_decode_attn of layer l (the arguments up to err_flag);
 *   - fill (may be NULL): clo_fill_cache_buffer for layer l+1, whose miss list
 *     an earlier call's lookup wrote.  Its CTAs run beside the attention's
 *     main kernel in CTA slots that grid leaves free: with opts->num_ctas == 0
 *     the attention takes the default grid less fill->num_ctas CTAs (less the
 *     fill's default share when that is 0);
 *   - lookup (may be NULL): clo_lookup_update for layer l+2, carried as in
 *     clo_hybrid_decode_attn_lookup (in the attention's merge launch, or for
 *     more than 64 groups in a launch of its own after the fill).
 * Called for l = 0, 1, ... this gives each layer's lookup one layer of
 * compute ahead of the layer's attention, and its fill the whole attention of
 * the layer before.  The results are those of the three calls made
 * separately, in any order, so the three must touch disjoint memory: the
 * fill's Cache Buffer is not the one the attention reads, and its miss list
 * and count are not the ones the lookup writes (both checked by pointer:
 * CLO_ERR_INVALID_ARG), and the lookup's labels and outputs are not read by
 * the other two.  The fill reports bad rows in err_flag, like the attention.
 * opts: num_ctas as for clo_hybrid_decode_attn; ev_begin is recorded before
 * the attention's main kernel, ev_end after the fill (after the main kernel
 * when there is none), so the two bracket both kernels.  The workspace size
 * for num_ctas == 0 is enough with or without a fill.
 */
clo_status clo_hybrid_decode_layer(
    const clo_half* q, const clo_half* cbK, const clo_half* cbV, const int32_t* idx, int k, int C,
    const clo_half* pK, const clo_half* pV, const int32_t* persist_ids, int Np, int T, int B,
    int Hq, int Hkv, int d, float scale, clo_half* out, float* lse, void* workspace,
    size_t ws_bytes, int32_t* err_flag, const clo_fill_args* fill, const clo_lookup_args* lookup,
    const clo_attn_opts* opts, cudaStream_t stream);

/*
 * clo_hybrid_decode_attn_noalloc -- clo_hybrid_decode_attn for callers that
 * cannot allocate device memory: serving engines that reserve all free device
 * memory for their own pool at start-up (so a later cudaMalloc fails or
 * fragments that pool), deployments that forbid allocation after start-up,
 * and host programs that reach this library through its C ABI alone, with no
 * allocator of their own.  The pages have no counterpart: this is a
 * deployment variant of the same computation.
 * Same arguments, layouts and results as clo_hybrid_decode_attn, without the
 * workspace: the split-KV scratch is a fixed array of
 * clo_hybrid_noalloc_max_scratch() bytes (8 MiB) compiled into the library,
 * which every GPU that loads the library holds until the process exits.
 *  - Returns CLO_ERR_WORKSPACE, launching nothing, when the problem needs more
 *    than that (clo_hybrid_workspace_size(B, Hq, Hkv, d, num_ctas) > 8 MiB).
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it for that device's context; make that
 *    first call before any stream capture.  A call in a new context on the
 *    device (after cudaDeviceReset) looks it up again, and is then again a
 *    first call.  CLO_ERR_CUDA if the lookup fails.
 *  - It never calls cudaMalloc, cudaFree or any allocating routine.
 *  - All calls share the one array and it keeps the previous call's
 *    contents; nothing in it needs to start at zero.  Calls on one device
 *    that overlap on the GPU (on concurrent streams) race on it: serialise
 *    them.  Each device has its own copy of the array.
 */
clo_status clo_hybrid_decode_attn_noalloc(const clo_half* q, const clo_half* cbK,
                                          const clo_half* cbV, const int32_t* idx, int k, int C,
                                          const clo_half* pK, const clo_half* pV,
                                          const int32_t* persist_ids, int Np, int T, int B,
                                          int Hq, int Hkv, int d, float scale, clo_half* out,
                                          float* lse, int32_t* err_flag,
                                          const clo_attn_opts* opts, cudaStream_t stream);

/* Size in bytes of the fixed scratch used by clo_hybrid_decode_attn_noalloc. */
size_t clo_hybrid_noalloc_max_scratch(void);

/*
 * clo_wait_ready / clo_signal_ready -- GPU-centric data-ready synchronisation
 * ("CLO: CPU-Light KVCache Offloading", section 2 Q1 "GPU-centric
 * synchronisation" and Fig. 8's Data Synchronization Controller): the GPU
 * polls a flag in host memory instead of the host blocking in
 * cudaStreamSynchronize, so the thread that launches kernels can queue the
 * work that needs some data before a host thread has finished moving it.
 *
 * clo_wait_ready queues on `stream` a one-warp kernel that waits until
 * (int32_t)(*ready - expected) >= 0 (sequence numbers; wrap-around safe),
 * then lets the work queued after it run.  The wait is bounded: after
 * timeout_us microseconds (1 .. 10,000,000) it ORs CLO_FLAG_TIMEOUT into
 * *err_flag (a caller-zeroed device int32; may be NULL) and returns, and the
 * work after it runs on whatever the memory holds.  The caller reads the flag
 * after the stream synchronises (clo_check_error_flag gives CLO_ERR_TIMEOUT).
 *  - ready: 4-byte aligned memory the device reads in place: pinned host
 *    memory (cudaHostAlloc, a pinned torch tensor; read through its mapped
 *    address) or device memory.  Anything else gives CLO_ERR_INVALID_ARG.
 *  - The value must be written by a host thread (clo_signal_ready), never by
 *    another GPU kernel: kernels that wait on one another are not guaranteed
 *    to run at the same time.
 *  - The wait is an acquire at system scope: the data the host wrote before
 *    clo_signal_ready published the value is visible to the kernels after it.
 *  - Under lazy module loading (CUDA's default), the first launch of a kernel
 *    in a process can wait for the device to go idle while its code loads.
 *    Such a launch queued behind a wait that the launching thread's own later
 *    work must release would stall until the wait runs out.  Launch every
 *    kernel that follows a wait once beforehand (one call of each libclo
 *    entry point loads its kernels), or set CUDA_MODULE_LOADING=EAGER.
 *
 * clo_signal_ready stores `value` to *ready (host memory) with release
 * ordering, after a release fence: every earlier write of the calling thread
 * is visible to a GPU that has seen the value.  Host code only; no GPU call.
 */
clo_status clo_wait_ready(const uint32_t* ready, uint32_t expected, uint32_t timeout_us,
                          int32_t* err_flag, cudaStream_t stream);
clo_status clo_signal_ready(uint32_t* ready, uint32_t value);

/* Workspace bytes clo_paged_decode_attn needs (same rules as above). */
size_t clo_paged_workspace_size(int B, int Hq, int Hkv, int d, int num_ctas);

/*
 * clo_paged_decode_attn -- dense decode attention over a paged KV cache, one
 * query per request (NEO GPU/CPU paged attention; FastDecode R-Part).
 * Token t < ctx_len[r] of request r is row t % block_size of block
 * block_table[r][t / block_size].
 * q:           [B][Hq][d] fp16.
 * kc, vc:      [num_blocks][Hkv][block_size][d] fp16 block pool.
 * block_table: [B][max_blocks] int32 entries in [0, num_blocks).
 * ctx_len:     [B] int32 in [0, max_blocks*block_size]; 0 gives zeros.
 * out, lse, workspace, err_flag, opts: as for clo_hybrid_decode_attn.
 * Requires block_size == 16, G <= 8, d == 128, B <= 4096,
 * B*Hkv*max_blocks < 2^31.
 */
clo_status clo_paged_decode_attn(const clo_half* q, const clo_half* kc,
                                 const clo_half* vc,
                                 const int32_t* block_table, int max_blocks,
                                 const int32_t* ctx_len, int num_blocks, int B,
                                 int Hq, int Hkv, int d, int block_size,
                                 float scale, clo_half* out, float* lse,
                                 void* workspace, size_t ws_bytes,
                                 int32_t* err_flag, const clo_attn_opts* opts,
                                 cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CLO_H_ */
