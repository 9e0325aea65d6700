// clo_plan.cu -- offline persistent-head plan (CLO section 3.3 and section 2,
// selective residency; Eqs. 11-13), on the host.
//
// A KV head whose profiled mean query cosine s^ falls short of its threshold
// tau by more than the margin eps will miss most steps: its reuse difficulty
// is D = tau - (s^ - eps) (Eq. 11) and it is "hard" when D > 0.  One layer's
// compute time T_comp hides the transfer of N_p = floor(T_comp * B_link /
// mem_head) heads' top-k rows over the host link (Eq. 12; the printed ratio
// is not dimensionless and this is the dimensionless reading).  The hard
// heads beyond that are kept whole in HBM: N_persist = max(N_hard - N_p, 0)
// (Eq. 13), the hardest first, ties to the lower head index.
#include <math.h>

#include <algorithm>
#include <vector>

#include "clo.h"

extern "C" clo_status clo_plan_persistent(const float* tau, const float* s_hat, int L, int Hkv,
                                          float eps, double t_comp_s, double link_bytes_per_s,
                                          double head_bytes, double* D, int32_t* n_p,
                                          int32_t* n_persist, int32_t* persist_ids) {
    if (L < 0 || Hkv <= 0 || !(head_bytes > 0.0) || !(t_comp_s >= 0.0) ||
        !(link_bytes_per_s >= 0.0) || !isfinite(t_comp_s) || !isfinite(link_bytes_per_s) ||
        !isfinite(head_bytes) || !isfinite(eps))
        return CLO_ERR_INVALID_ARG;
    if (n_p == nullptr || (L > 0 && (tau == nullptr || s_hat == nullptr || D == nullptr ||
                                     n_persist == nullptr || persist_ids == nullptr)))
        return CLO_ERR_INVALID_ARG;
    const double heads = floor(t_comp_s * link_bytes_per_s / head_bytes);  // Eq. 12
    const int cap = heads >= 2147483647.0 ? 2147483647 : static_cast<int>(heads);
    *n_p = cap;
    std::vector<int> hard;
    hard.reserve(Hkv);
    for (int l = 0; l < L; ++l) {
        const size_t row = static_cast<size_t>(l) * Hkv;
        hard.clear();
        for (int i = 0; i < Hkv; ++i) {
            const double d = static_cast<double>(tau[row + i]) -
                             (static_cast<double>(s_hat[row + i]) - static_cast<double>(eps));
            D[row + i] = d;  // Eq. 11
            if (d > 0.0) hard.push_back(i);
        }
        std::stable_sort(hard.begin(), hard.end(),
                         [&](int a, int b) { return D[row + a] > D[row + b]; });
        const int keep = std::max(static_cast<int>(hard.size()) - cap, 0);  // Eq. 13
        n_persist[l] = keep;
        for (int j = 0; j < Hkv; ++j) persist_ids[row + j] = j < keep ? hard[j] : -1;
    }
    return CLO_OK;
}
