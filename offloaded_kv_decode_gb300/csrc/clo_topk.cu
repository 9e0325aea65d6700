// clo_topk.cu -- top-k retrieval by exact qk-score (CLO section 2, Eq. 6: the
// ranking of the keys by q . k does not depend on |q|; the decode flow's
// top-k retrieval stage), for sm_103a.
//
// Per KV head g of batch row b, the score of key t is (sum of the group's G
// query vectors) . K_t, accumulated in fp32; the k largest are selected, equal
// scores at the cut going to the lower token index, and written in ascending
// token order (so the output is deterministic).
//
// Two kernels:
//   topk_score_kernel   streams every key once (HBM-bound: T * 256 bytes a
//                       head).  One resident wave of CTAs, each scoring an
//                       equal share of all heads' keys; each half-warp scores
//                       one 256-byte key row per step (16 bytes a lane, a
//                       16-lane shuffle reduction), with 8 rows in flight per
//                       half-warp.
//   topk_select_kernel  one thread-block cluster per head, each CTA holding a
//                       slice of the head's keys (the order-preserving
//                       integer image of the fp32 scores) in shared memory:
//                       a 4-pass radix select (8 bits a pass, per-warp
//                       histograms summed over the cluster through
//                       distributed shared memory) finds the k-th largest key
//                       and how many of its ties to keep; a last pass walks
//                       each slice in token order and writes the selected
//                       tokens with block-wide prefix sums, offset by the
//                       counts of the lower slices.
#include <algorithm>

#include <cooperative_groups.h>

#include "clo_device.cuh"

namespace clo {

constexpr int TK_D = 128;
constexpr int TK_SCORE_THREADS = 256;
constexpr int TK_UNROLL = 8;                                      // rows in flight a half-warp
constexpr int TK_ROWS_PER_STEP = (TK_SCORE_THREADS / 16) * TK_UNROLL;  // 128 rows a CTA step
#ifndef CLO_TK_SCORE_CTAS_PER_SM
#define CLO_TK_SCORE_CTAS_PER_SM 3
#endif
constexpr int TK_SCORE_CTAS_PER_SM = CLO_TK_SCORE_CTAS_PER_SM;  // the register cap follows
constexpr int TK_SEL_THREADS = 1024;
constexpr int TK_SEL_CACHE = 47 * 1024;  // keys a select CTA keeps in shared memory (188 KB)
constexpr int TK_SEL_SLICE = 8 * 1024;   // aim for about this many keys a select CTA
constexpr int TK_SEL_MAX_CLUSTER = 8;    // portable cluster size
constexpr int TK_MAX_G = 8;

#ifndef CLO_TK_EVICT_FIRST
#define CLO_TK_EVICT_FIRST 1
#endif

// A 16-byte load of a key row, read once: no L1 allocation, and in L2 evicted
// first, so the 512 MB key stream does not push the scores the select kernel
// reads next out of L2.
__device__ __forceinline__ uint4 ld_key_row(const void* p, uint64_t policy) {
    uint4 v;
#if CLO_TK_EVICT_FIRST
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
#else
    (void)policy;
    v = *reinterpret_cast<const uint4*>(p);
#endif
    return v;
}

// The rows of all heads form one line (head-major); CTA c scores an equal
// contiguous share of it, so one resident wave covers every key with no
// ragged last chunk per head.  A share crosses at most a few head boundaries;
// the group's summed query is reloaded at each.
__global__ void __launch_bounds__(TK_SCORE_THREADS, TK_SCORE_CTAS_PER_SM)
    topk_score_kernel(const clo_half* __restrict__ q, const clo_half* __restrict__ K, int Hq,
                      int Hkv, int G, int T, long long rows, float* __restrict__ scores) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31, c = lane & 15, half = lane >> 4;
    const int warp = threadIdx.x >> 5;
    const uint64_t policy = l2_evict_first_policy();
    const long long r0 = rows * blockIdx.x / gridDim.x;
    const long long r1 = rows * (blockIdx.x + 1) / gridDim.x;
    if (r1 <= r0) return;
    // Heads h_first .. h_last, from row t_first of the first to row t_last
    // (exclusive) of the last.
    const int h_first = static_cast<int>(r0 / T), h_last = static_cast<int>((r1 - 1) / T);
    const int t_first = static_cast<int>(r0 - static_cast<long long>(h_first) * T);
    const int t_last = static_cast<int>(r1 - static_cast<long long>(h_last) * T);
    for (int head = h_first; head <= h_last; ++head) {  // head = b * Hkv + g
        const int b = head / Hkv, g = head - b * Hkv;
        // Lane c holds dims [8c, 8c + 8) of the group's summed query.
        float qs[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qs[i] = 0.f;
        const clo_half* qg = q + (static_cast<size_t>(b) * Hq + static_cast<size_t>(g) * G) * TK_D + c * 8;
        for (int j = 0; j < G; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(qg + static_cast<size_t>(j) * TK_D);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
                qs[2 * i] += f.x;
                qs[2 * i + 1] += f.y;
            }
        }
        const clo_half* Kh = K + static_cast<size_t>(head) * T * TK_D + c * 8;
        float* sh = scores + static_cast<size_t>(head) * T;
        const int t0 = head == h_first ? t_first : 0;
        const int t1 = head == h_last ? t_last : T;
        // The loop runs on a warp-uniform base (the shuffles below need the
        // whole warp); half-warp h of warp w takes rows base + h + 16 u.
        for (int base = t0 + 2 * warp; base < t1; base += TK_ROWS_PER_STEP) {
            uint4 kv[TK_UNROLL];
#pragma unroll
            for (int u = 0; u < TK_UNROLL; ++u) {
                const int t = base + half + u * (TK_SCORE_THREADS / 16);
                if (t < t1) kv[u] = ld_key_row(Kh + static_cast<size_t>(t) * TK_D, policy);
            }
#pragma unroll
            for (int u = 0; u < TK_UNROLL; ++u) {
                const int t = base + half + u * (TK_SCORE_THREADS / 16);
                float acc = 0.f;
                if (t < t1) {
                    const uint32_t w[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
                        acc = fmaf(qs[2 * i], f.x, acc);
                        acc = fmaf(qs[2 * i + 1], f.y, acc);
                    }
                }
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, off);
                if (c == 0 && t < t1) sh[t] = acc;
            }
        }
    }
}

// Order-preserving image of an fp32 score (larger score, larger key; +0 and
// -0 map to the same key).
__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of a per-thread count over the CTA (thread order) and
// the CTA total: a warp scan, then warp 0 scans the warp totals.
// wsum: TK_SEL_THREADS / 32 ints; woff: TK_SEL_THREADS / 32 + 1 ints.
__device__ __forceinline__ int block_scan(int v, int* wsum, int* woff, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < TK_SEL_THREADS / 32 ? wsum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(FULL_MASK, wi, off);
            if (lane >= off) wi += u;
        }
        if (lane < TK_SEL_THREADS / 32) woff[lane] = wi - w;
        if (lane == 31) woff[TK_SEL_THREADS / 32] = wi;
    }
    __syncthreads();
    total = woff[TK_SEL_THREADS / 32];
    return woff[warp] + incl - v;
}

// One cluster of `cs` CTAs per head (cs = gridDim.x / heads); CTA r of the
// cluster caches keys [r * slice, (r + 1) * slice) in shared memory and every
// pass sums the cluster's histograms through distributed shared memory, so
// every CTA takes the same digit decisions.  Registers are held to 32 a
// thread so two 1024-thread CTAs share an SM: at 64 a thread one CTA fills
// the register file, and 64 heads of 4 CTAs took two waves on 152 SMs.
__global__ void __launch_bounds__(TK_SEL_THREADS, 2)
    topk_select_kernel(const float* __restrict__ scores, int T, int k, int slice,
                       int32_t* __restrict__ idx) {
    namespace cg = cooperative_groups;
    pdl_launch_dependents();
    pdl_wait();
    constexpr int kWarps = TK_SEL_THREADS / 32;
    __shared__ int hist[kWarps][256];  // one histogram per warp (no contention between warps)
    __shared__ int total[2][256];      // this CTA's counts, read by the whole cluster (by pass parity)
    __shared__ int gtotal[256];
    __shared__ int wsum[kWarps];
    __shared__ int woff[kWarps + 1];
    __shared__ int counts[2];          // this CTA's keys above and equal to the k-th
    __shared__ uint32_t sel_prefix;
    __shared__ int sel_need;
    extern __shared__ uint32_t keys_sm[];  // this CTA's slice of the row
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int row = blockIdx.x / cs;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lo = min(T, rank * slice), hi = min(T, lo + slice), n = hi - lo;
    const float* s = scores + static_cast<size_t>(row) * T + lo;
    // The slice is read from L2 once, 8 loads in flight a thread.
    for (int t0 = threadIdx.x; t0 < n; t0 += 8 * TK_SEL_THREADS) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = t0 + u * TK_SEL_THREADS;
            v[u] = t < n ? s[t] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = t0 + u * TK_SEL_THREADS;
            if (t < n) keys_sm[t] = order_key(v[u]);
        }
    }
    if (threadIdx.x == 0) {
        sel_prefix = 0u;
        sel_need = k;
    }
    uint32_t mask = 0u;
    int last_digit = 0, par = 0;
    // Pass p writes total[p & 1].  The other CTAs read it between this pass's
    // cluster barrier and the next one, and pass p + 2 writes it only after
    // that next barrier, so one cluster barrier a pass is enough.
    for (int shift = 24; shift >= 0; shift -= 8, par ^= 1) {
        for (int i = lane; i < 256; i += 32) hist[warp][i] = 0;
        __syncthreads();
        const uint32_t prefix = sel_prefix;
        // Four keys a lane per trip; the adds are shared-memory atomics on
        // the warp's own histogram (nothing waits on them, and lanes that hit
        // the same bin are resolved by the atomic unit).
        for (int t0 = warp * 32; t0 < n; t0 += 4 * TK_SEL_THREADS) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int t = t0 + u * TK_SEL_THREADS + lane;
                if (t < n) {
                    const uint32_t key = keys_sm[t];
                    if ((key & mask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1);
                }
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 256; i += TK_SEL_THREADS) {
            int c = 0;
            for (int w = 0; w < kWarps; ++w) c += hist[w][i];
            total[par][i] = c;
        }
        cluster.sync();  // every CTA's counts are final
        for (int i = threadIdx.x; i < 256; i += TK_SEL_THREADS) {
            int c = 0;
            for (int r = 0; r < cs; ++r) c += cluster.map_shared_rank(&total[par][0], r)[i];
            gtotal[i] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // Lane l owns digits 255 - 8l - 7 .. 255 - 8l (from the top): find
            // the digit where the count from the top first reaches need.
            const int need = sel_need;
            int own = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) own += gtotal[255 - 8 * lane - j];
            int incl = own;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(FULL_MASK, incl, off);
                if (lane >= off) incl += v;
            }
            const unsigned reach = __ballot_sync(FULL_MASK, incl >= need);
            const int l = __ffs(reach) - 1;  // need <= the bucket's count, so some lane reaches it
            if (lane == l) {
                int cum = incl - own;
                int digit = 255 - 8 * l;
                for (int j = 0; j < 8; ++j) {
                    const int dgt = 255 - 8 * l - j;
                    if (cum + gtotal[dgt] >= need) {
                        digit = dgt;
                        break;
                    }
                    cum += gtotal[dgt];
                }
                sel_need = need - cum;
                sel_prefix = prefix | (static_cast<uint32_t>(digit) << shift);
            }
        }
        mask |= 255u << shift;
        __syncthreads();
        last_digit = static_cast<int>((sel_prefix >> shift) & 255u);
    }
    const int last_par = par ^ 1;  // the buffer of the last pass
    // kth = the k-th largest key of the row; the row keeps every larger key
    // and the first `ties` keys equal to it, in token order.
    const uint32_t kth = sel_prefix;
    const int ties = sel_need;
    // This CTA's keys above the k-th and equal to it.
    int above = 0;
    for (int t = threadIdx.x; t < n; t += TK_SEL_THREADS) above += keys_sm[t] > kth ? 1 : 0;
    int above_total;
    (void)block_scan(above, wsum, woff, above_total);
    if (threadIdx.x == 0) {
        counts[0] = above_total;
        counts[1] = total[last_par][last_digit];  // the last pass counted exactly the keys equal to kth
    }
    cluster.sync();
    int out_base = 0, ties_before = 0;
    for (int r = 0; r < rank; ++r) {
        const int* c = cluster.map_shared_rank(counts, r);
        const int eq = c[1];
        const int take = min(eq, max(ties - ties_before, 0));
        out_base += c[0] + take;
        ties_before += eq;
    }
    cluster.sync();  // the other CTAs' counts are no longer read
    const int my_ties = min(counts[1], max(ties - ties_before, 0));
    const bool all_ties = my_ties == counts[1];  // the usual case: no tie rank needed
    // Thread i takes keys 4i .. 4i + 3 of each 4096-key chunk, so thread
    // order is token order.
    int32_t* out = idx + static_cast<size_t>(row) * k;
    int taken = out_base, ties_seen = 0;
    for (int t0 = 0; t0 < n; t0 += 4 * TK_SEL_THREADS) {
        const int tb = t0 + 4 * threadIdx.x;
        uint32_t key[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) key[u] = tb + u < n ? keys_sm[tb + u] : 0u;
        bool sel[4];
        if (all_ties) {
#pragma unroll
            for (int u = 0; u < 4; ++u) sel[u] = tb + u < n && key[u] >= kth;
        } else {
            int nt = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) nt += (tb + u < n && key[u] == kth) ? 1 : 0;
            int tie_total;
            int rnk = ties_seen + block_scan(nt, wsum, woff, tie_total);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool in = tb + u < n;
                const bool tie = in && key[u] == kth;
                sel[u] = in && (key[u] > kth || (tie && rnk < my_ties));
                rnk += tie ? 1 : 0;
            }
            ties_seen += tie_total;
        }
        int ns = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) ns += sel[u] ? 1 : 0;
        int sel_total;
        int pos = taken + block_scan(ns, wsum, woff, sel_total);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (sel[u]) {
                if (pos < k) out[pos] = lo + tb + u;  // exactly k are selected; the test guards the store
                ++pos;
            }
        }
        taken += sel_total;
    }
}

}  // namespace clo

using namespace clo;

extern "C" size_t clo_topk_workspace_size(int B, int Hkv, int T) {
    if (B < 0 || Hkv <= 0 || T < 0) return 0;
    return static_cast<size_t>(B) * Hkv * T * sizeof(float);
}

extern "C" clo_status clo_topk_retrieve(const clo_half* q, const clo_half* K, int B, int Hq,
                                        int Hkv, int T, int d, int k, int32_t* idx,
                                        void* workspace, size_t ws_bytes,
                                        const clo_attn_opts* opts, cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || T < 0 || k < 0 || k > T)
        return CLO_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != TK_D || G > TK_MAX_G) return CLO_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Hkv > 65535 || T > TK_SEL_MAX_CLUSTER * TK_SEL_CACHE)
        return CLO_ERR_UNSUPPORTED;
    if (B == 0 || k == 0) return CLO_OK;
    if (q == nullptr || K == nullptr || idx == nullptr) return CLO_ERR_INVALID_ARG;
    const auto aligned = [](const void* p, size_t a) {
        return (reinterpret_cast<uintptr_t>(p) % a) == 0;
    };
    if (!aligned(q, 16) || !aligned(K, 16) || !aligned(idx, 4)) return CLO_ERR_INVALID_ARG;
    const size_t need = clo_topk_workspace_size(B, Hkv, T);
    if (workspace == nullptr || ws_bytes < need || !aligned(workspace, 16)) return CLO_ERR_WORKSPACE;
    float* scores = static_cast<float*>(workspace);
    const int heads = B * Hkv;
    const int sms = device_sm_count();
    if (sms <= 0) return CLO_ERR_CUDA;
    // One resident wave of score CTAs, each with at least one CTA step of rows.
    const long long rows = static_cast<long long>(heads) * T;
    long long score_ctas = static_cast<long long>(sms) * TK_SCORE_CTAS_PER_SM;
    score_ctas = std::max(1ll, std::min(score_ctas, rows / TK_ROWS_PER_STEP));
    if (opts != nullptr && opts->ev_begin != nullptr && !record_event(opts->ev_begin, stream))
        return CLO_ERR_CUDA;
    if (launch_pdl(topk_score_kernel, dim3(static_cast<unsigned>(score_ctas)),
                   dim3(TK_SCORE_THREADS), 0, stream, q, K, Hq, Hkv, G, T, rows, scores) !=
        cudaSuccess)
        return CLO_ERR_CUDA;
    if (opts != nullptr && opts->ev_end != nullptr && !record_event(opts->ev_end, stream))
        return CLO_ERR_CUDA;
    // Cluster of cs CTAs per head, each caching a slice of at most
    // TK_SEL_CACHE keys; at least 4 when the row is long enough, so one head's
    // passes are spread over several SMs.
    int cs = static_cast<int>((static_cast<long long>(T) + TK_SEL_SLICE - 1) / TK_SEL_SLICE);
    cs = std::max(1, std::min(TK_SEL_MAX_CLUSTER, cs));
    const int slice = (T + cs - 1) / cs;
    if (slice > TK_SEL_CACHE) return CLO_ERR_UNSUPPORTED;
    const size_t sel_smem = static_cast<size_t>(slice) * sizeof(uint32_t);
    if (!prepare_kernel(reinterpret_cast<const void*>(topk_select_kernel),
                        static_cast<int>(TK_SEL_CACHE * sizeof(uint32_t))))
        return CLO_ERR_CUDA;
    if (launch_pdl_cluster(topk_select_kernel, dim3(heads * cs), dim3(TK_SEL_THREADS), sel_smem,
                           stream, static_cast<unsigned>(cs), static_cast<const float*>(scores), T,
                           k, slice, idx) != cudaSuccess)
        return CLO_ERR_CUDA;
    return CLO_OK;
}
