// clo_lookup.cuh -- the head-wise approximate-cache lookup + query-label update
// (CLO section 2, Eq. 10, section 3 Fig. 7) as a device routine run by one
// thread-block cluster, shared by the stand-alone lookup kernel, by the
// attention's merge kernel when a small next-layer lookup rides in its launch,
// and by the lookup launched beside the attention's main kernel.
//
// One cluster of LK_CLUSTER CTAs covers all (batch row, KV head) groups: each
// CTA takes a contiguous share and one warp scores one group; every lane holds
// 4 of the 128 dimensions of each of the G query heads, so q and the labels
// are read from HBM exactly once with 8-byte loads, and the three dot
// products per head are finished with warp shuffles.  On a miss the same
// registers are written back as the new labels.  The compact miss list is
// deterministic (ascending b*Hkv+g) without a second launch or global
// scratch: after a cluster barrier every CTA reads the miss counts of the
// lower-ranked CTAs from their shared memory (DSMEM) and writes its own misses
// at that offset.
#pragma once

#include <cooperative_groups.h>

#include "clo_device.cuh"

namespace clo {

constexpr int LK_CLUSTER = 8;
constexpr int LK_MAX_G = 8;
constexpr int LK_MAX_GROUPS = 65536;

struct LookupParams {
    const clo_half* q;
    clo_half* labels;
    const float* w;
    const float* tau;
    const uint8_t* pmask;
    uint8_t* flag;
    float* sim;
    int32_t* miss_list;
    int32_t* miss_count;
    int B, Hq, Hkv, G;
};

__device__ __forceinline__ float2 h2f(uint32_t v) {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
}

// Run by every thread of every CTA of one LK_CLUSTER-CTA cluster; kWarps is
// the warps per CTA.  miss_sm: at least ceil(B*Hkv / LK_CLUSTER) bytes of
// this CTA's shared memory; cta_misses: one int of it.
template <int kWarps>
__device__ void lookup_cluster(const LookupParams& p, uint8_t* miss_sm, int* cta_misses) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int ngroups = p.B * p.Hkv;
    const int g0 = static_cast<int>(static_cast<long long>(ngroups) * rank / LK_CLUSTER);
    const int g1 = static_cast<int>(static_cast<long long>(ngroups) * (rank + 1) / LK_CLUSTER);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    for (int gi = g0 + warp; gi < g1; gi += kWarps) {
        const int b = gi / p.Hkv;
        const int g = gi - b * p.Hkv;
        const size_t base = (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * p.G) * 128 +
                            static_cast<size_t>(lane) * 4;
        // Every load of the group is issued before the first use.
        uint2 qv[LK_MAX_G], lv[LK_MAX_G];
        float wv[LK_MAX_G];
#pragma unroll
        for (int j = 0; j < LK_MAX_G; ++j) {
            if (j < p.G) {
                qv[j] = *reinterpret_cast<const uint2*>(p.q + base + j * 128);
                lv[j] = *reinterpret_cast<const uint2*>(p.labels + base + j * 128);
                wv[j] = __ldg(p.w + g * p.G + j);
            }
        }
        const float tau_g = __ldg(p.tau + g);
        const bool persistent = p.pmask != nullptr && __ldg(p.pmask + g) != 0;
        float sw = 0.f, swc = 0.f, sc = 0.f;
#pragma unroll
        for (int j = 0; j < LK_MAX_G; ++j) {
            if (j < p.G) {
                const float2 qa = h2f(qv[j].x), qb = h2f(qv[j].y);
                const float2 la = h2f(lv[j].x), lb = h2f(lv[j].y);
                float dot = qa.x * la.x;
                dot = fmaf(qa.y, la.y, dot);
                dot = fmaf(qb.x, lb.x, dot);
                dot = fmaf(qb.y, lb.y, dot);
                float qq = qa.x * qa.x;
                qq = fmaf(qa.y, qa.y, qq);
                qq = fmaf(qb.x, qb.x, qq);
                qq = fmaf(qb.y, qb.y, qq);
                float ll = la.x * la.x;
                ll = fmaf(la.y, la.y, ll);
                ll = fmaf(lb.x, lb.x, ll);
                ll = fmaf(lb.y, lb.y, ll);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    dot += __shfl_xor_sync(FULL_MASK, dot, off);
                    qq += __shfl_xor_sync(FULL_MASK, qq, off);
                    ll += __shfl_xor_sync(FULL_MASK, ll, off);
                }
                const float c = (qq > 0.f && ll > 0.f) ? dot / (sqrtf(qq) * sqrtf(ll)) : 0.f;
                const float w = wv[j];
                sw += w;
                swc = fmaf(w, c, swc);
                sc += c;
            }
        }
        const float s = (sw != 0.f) ? swc / sw : sc / static_cast<float>(p.G);  // Eq. 10
        uint8_t f;
        if (persistent) {
            f = 2;  // persistent: always resident, never looked up
        } else if (s >= tau_g) {
            f = 0;  // hit: keep the label
        } else {
            f = 1;  // miss: the whole KV head is replaced, labels <- current queries
#pragma unroll
            for (int j = 0; j < LK_MAX_G; ++j)
                if (j < p.G) *reinterpret_cast<uint2*>(p.labels + base + j * 128) = qv[j];
        }
        if (lane == 0) {
            p.flag[gi] = f;
            p.sim[gi] = s;
            miss_sm[gi - g0] = (f == 1);
        }
    }
    __syncthreads();
    if (warp == 0) {
        int cnt = 0;
        for (int i = lane; i < g1 - g0; i += 32) cnt += miss_sm[i];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) cnt += __shfl_xor_sync(FULL_MASK, cnt, off);
        if (lane == 0) *cta_misses = cnt;
    }
    cluster.sync();
    if (warp == 0) {
        int pos = 0;
        for (int r = 0; r < rank; ++r) pos += *cluster.map_shared_rank(cta_misses, r);
        for (int i0 = 0; i0 < g1 - g0; i0 += 32) {
            const int i = i0 + lane;
            const bool m = (i < g1 - g0) && miss_sm[i] != 0;
            const unsigned bal = __ballot_sync(FULL_MASK, m);
            if (m) p.miss_list[pos + __popc(bal & ((1u << lane) - 1u))] = g0 + i;
            pos += __popc(bal);
        }
        if (rank == LK_CLUSTER - 1 && lane == 0) *p.miss_count = pos;
    }
    cluster.sync();  // keep every CTA's shared memory alive until all reads are done
}

// Host-side checks of a lookup's arguments (B > 0); fills p on success.
inline clo_status make_lookup_params(const clo_half* q, clo_half* labels, const float* w_q,
                                     const float* tau_kv, const uint8_t* persist_mask, int B,
                                     int Hq, int Hkv, int d, uint8_t* flag, float* sim,
                                     int32_t* miss_list, int32_t* miss_count, LookupParams& p) {
    const auto aligned = [](const void* x, size_t a) {
        return (reinterpret_cast<uintptr_t>(x) % a) == 0;
    };
    if (miss_count == nullptr || !aligned(miss_count, 4)) return CLO_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return CLO_ERR_INVALID_ARG;
    if (q == nullptr || labels == nullptr || w_q == nullptr || tau_kv == nullptr ||
        flag == nullptr || sim == nullptr || miss_list == nullptr)
        return CLO_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(labels, 16) || !aligned(w_q, 4) || !aligned(tau_kv, 4) ||
        !aligned(sim, 4) || !aligned(miss_list, 4))
        return CLO_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != 128 || G > LK_MAX_G) return CLO_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Hkv > LK_MAX_GROUPS) return CLO_ERR_UNSUPPORTED;
    p = LookupParams{q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list, miss_count,
                     B, Hq, Hkv, G};
    return CLO_OK;
}

// Shared-memory bytes lookup_cluster needs a CTA for B*Hkv groups.
inline int lookup_smem_bytes(int B, int Hkv) { return (B * Hkv + LK_CLUSTER - 1) / LK_CLUSTER; }

// Launches the lookup as one cluster directly after a libclo main kernel,
// beside it (see lookup_beside_kernel in clo_lookup.cu).
cudaError_t launch_lookup_beside(const LookupParams& p, cudaStream_t stream);

// A lookup of at least this many (batch row, KV head) groups is carried beside
// the attention's main kernel; a smaller one rides in the attention's merge
// launch.  A launch of
// its own adds a step to the chain, which a small lookup does not repay (per
// layer-step, one box: the B1 128K step with 8 groups 32.7 us in the merge
// launch, 36.2 us beside; the B8 32K layer with 64 groups 58.4 and 59.6 us),
// while a large one, left to run after the drain, delays the next layer (the
// Qwen2.5-14B batch-16 step with 128 groups: 138.5 us in the merge launch,
// 135.8 us beside).
constexpr int LK_BESIDE_MIN_GROUPS = 65;

}  // namespace clo
