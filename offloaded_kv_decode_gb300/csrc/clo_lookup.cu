// clo_lookup.cu -- per-head thresholds (CLO Eqs. 7-9) and the fused head-wise
// approximate-cache lookup + query-label update (CLO section 2, Eq. 10,
// section 3 Fig. 7), for sm_103a.  The lookup is one launch of a single
// 8-CTA thread-block cluster running lookup_cluster (clo_lookup.cuh).
#include "clo_lookup.cuh"

namespace clo {

// 4 warps per CTA: small enough (with <= 64 registers per thread) to be
// resident next to an attention CTA, so a lookup can overlap attention.
constexpr int LK_THREADS = 128;
constexpr int LK_WARPS = LK_THREADS / 32;
constexpr float PI_F = 3.14159265358979323846f;

__global__ void thresholds_kernel(const float* __restrict__ s, int n_kv, int group, float eta,
                                  float n_exp, float* __restrict__ tau) {
    pdl_launch_dependents();
    pdl_wait();
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n_kv) return;
    float acc = 0.f;
    for (int j = 0; j < group; ++j) acc += s[g * group + j];
    const float sg = acc / static_cast<float>(group);
    const float theta_star = acosf(eta);                              // Eq. 7
    const float lam = powf(sg, n_exp);                                // Eq. 8
    const float theta = lam * theta_star + (1.f - lam) * PI_F;        // Eq. 9
    tau[g] = cosf(theta);
}

__global__ void __cluster_dims__(LK_CLUSTER, 1, 1) __launch_bounds__(LK_THREADS, 8)
    lookup_update_kernel(const LookupParams p) {
    extern __shared__ uint8_t miss_sm[];  // miss bit of each group of this CTA
    __shared__ int cta_misses;
    pdl_launch_dependents();
    pdl_wait();
    lookup_cluster<LK_WARPS>(p, miss_sm, &cta_misses);
}

// The same with 16 warps per CTA, for more groups than the narrow form has
// warps: every warp then scores at most one group per CTA pass, so the
// launch is one round trip for the queries and labels instead of several.
constexpr int LK_WIDE_THREADS = 512;
__global__ void __cluster_dims__(LK_CLUSTER, 1, 1) __launch_bounds__(LK_WIDE_THREADS, 1)
    lookup_update_wide_kernel(const LookupParams p) {
    extern __shared__ uint8_t miss_sm[];
    __shared__ int cta_misses;
    pdl_launch_dependents();
    pdl_wait();
    lookup_cluster<LK_WIDE_THREADS / 32>(p, miss_sm, &cta_misses);
}

// The lookup launched beside the kernel before it: a main kernel that lets
// its dependents start only after its own dependency wait, and writes nothing
// the lookup reads or writes.  Every kernel before that one has then
// finished, so the lookup reads its inputs at once; it waits for that kernel
// at its end, so a kernel launched after the lookup still finds both
// finished.  16-warp CTAs held to 64 registers a thread (32K registers, half
// an SM's) fit on an SM once two attention CTAs there have finished, so a
// large lookup runs in the main kernel's drain.  (8- and 4-warp CTAs, which
// fit earlier but score several groups a warp, measured slower: Qwen2.5-14B
// batch-16 step 142.1 / 141.1 / 135.8 us a layer-step with 4 / 8 / 16 warps.)
constexpr int LK_BESIDE_THREADS = 512;

__global__ void __cluster_dims__(LK_CLUSTER, 1, 1) __launch_bounds__(LK_BESIDE_THREADS, 2)
    lookup_beside_kernel(const LookupParams p) {
    extern __shared__ uint8_t miss_sm[];
    __shared__ int cta_misses;
    pdl_launch_dependents();
    lookup_cluster<LK_BESIDE_THREADS / 32>(p, miss_sm, &cta_misses);
    pdl_wait();
}

cudaError_t launch_lookup_beside(const LookupParams& p, cudaStream_t stream) {
    const int per_cta = lookup_smem_bytes(p.B, p.Hkv);
    if (!prepare_kernel(reinterpret_cast<const void*>(lookup_beside_kernel), per_cta))
        return cudaErrorUnknown;
    return launch_pdl(lookup_beside_kernel, dim3(LK_CLUSTER), dim3(LK_BESIDE_THREADS),
                      static_cast<size_t>(per_cta), stream, p);
}

}  // namespace clo

using namespace clo;

extern "C" clo_status clo_thresholds(const float* s, int n_kv, int group, float eta, float n_exp,
                                     float* tau, cudaStream_t stream) {
    if (s == nullptr || tau == nullptr || n_kv < 0 || group < 1) return CLO_ERR_INVALID_ARG;
    if (!(eta >= -1.f && eta <= 1.f) || !(n_exp >= 0.f)) return CLO_ERR_INVALID_ARG;
    if (n_kv == 0) return CLO_OK;
    const int threads = 128;
    const int blocks = (n_kv + threads - 1) / threads;
    if (!prepare_kernel(reinterpret_cast<const void*>(thresholds_kernel), 0)) return CLO_ERR_CUDA;
    return launch_pdl(thresholds_kernel, dim3(blocks), dim3(threads), 0, stream, s, n_kv, group,
                      eta, n_exp, tau) == cudaSuccess
               ? CLO_OK
               : CLO_ERR_CUDA;
}

// The same map on the host in fp32, in the kernel's order: the group mean of
// s, then Eqs. 7-9 with the host C library's acosf, powf and cosf.
extern "C" clo_status clo_thresholds_host(const float* s, int n_kv, int group, float eta,
                                          float n_exp, float* tau) {
    if (n_kv < 0 || group < 1) return CLO_ERR_INVALID_ARG;
    if (!(eta >= -1.f && eta <= 1.f) || !(n_exp >= 0.f)) return CLO_ERR_INVALID_ARG;
    if (n_kv == 0) return CLO_OK;
    if (s == nullptr || tau == nullptr) return CLO_ERR_INVALID_ARG;
    const float theta_star = acosf(eta);                              // Eq. 7
    for (int g = 0; g < n_kv; ++g) {
        float acc = 0.f;
        for (int j = 0; j < group; ++j) acc += s[static_cast<size_t>(g) * group + j];
        const float sg = acc / static_cast<float>(group);
        const float lam = powf(sg, n_exp);                            // Eq. 8
        const float theta = lam * theta_star + (1.f - lam) * PI_F;    // Eq. 9
        tau[g] = cosf(theta);
    }
    return CLO_OK;
}

extern "C" clo_status clo_lookup_update(const clo_half* q, clo_half* labels, const float* w_q,
                                        const float* tau_kv, const uint8_t* persist_mask, int B,
                                        int Hq, int Hkv, int d, uint8_t* flag, float* sim,
                                        int32_t* miss_list, int32_t* miss_count,
                                        cudaStream_t stream) {
    if (miss_count == nullptr || (reinterpret_cast<uintptr_t>(miss_count) % 4) != 0)
        return CLO_ERR_INVALID_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return CLO_ERR_INVALID_ARG;
    if (B == 0) {  // nothing to look up: only the miss count is written
        return cudaMemsetAsync(miss_count, 0, sizeof(int32_t), stream) == cudaSuccess
                   ? CLO_OK
                   : CLO_ERR_CUDA;
    }
    LookupParams p;
    const clo_status st = make_lookup_params(q, labels, w_q, tau_kv, persist_mask, B, Hq, Hkv, d,
                                             flag, sim, miss_list, miss_count, p);
    if (st != CLO_OK) return st;
    const int per_cta = lookup_smem_bytes(B, Hkv);
    const bool wide = static_cast<long long>(B) * Hkv > static_cast<long long>(LK_CLUSTER) * LK_WARPS;
    auto* kern = wide ? lookup_update_wide_kernel : lookup_update_kernel;
    if (!prepare_kernel(reinterpret_cast<const void*>(kern), per_cta)) return CLO_ERR_CUDA;
    return launch_pdl(kern, dim3(LK_CLUSTER), dim3(wide ? LK_WIDE_THREADS : LK_THREADS),
                      static_cast<size_t>(per_cta), stream, p) == cudaSuccess
               ? CLO_OK
               : CLO_ERR_CUDA;
}
