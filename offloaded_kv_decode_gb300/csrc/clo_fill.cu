// clo_fill.cu -- miss-path fill of the Cache Buffer (CLO section 3, Fig. 7:
// an update writes the new KV rows straight to their final position, with no
// staging buffer; section 2: only the heads that missed are transferred), for
// sm_103a.
//
// For every KV head on the miss list (as written by the lookup) the rows of
// its new top-k token set are copied from the full KV copy into the Cache
// Buffer rows the hybrid attention reads.  The full copy may sit in pinned
// host memory: the kernel then reads it in place over NVLink-C2C, which takes
// the place of CLO's GDRCopy transfer engine (the GPU pulls the rows itself,
// so no CPU thread gathers or pushes them).
//
// Work is a flat line of rows (miss m, row j), m < *miss_count (read on the
// device, so the launch does not wait for the lookup's result on the host).
// A warp takes 16 rows at a time: lanes 0..15 load the rows' list entry,
// token and slot in parallel, then each half-warp moves 8 rows of K and 8 of
// V (256 bytes each, 16 bytes a lane), all loads before any store, so every
// lane has 16 independent 16-byte loads in flight across the host link.
#include "clo_fill.cuh"

namespace clo {

// 4-warp CTAs, 4 an SM: the same 16 warps an SM and register cap as larger
// CTAs, and one fill CTA fits in the room of one attention CTA, so a fill
// launched beside an attention grid that leaves a few CTA slots free runs
// alongside it (a caller overlapping the next layer's fill with this layer's
// attention).
constexpr int FILL_THREADS = 128;
constexpr int FILL_WARPS = FILL_THREADS / 32;
constexpr int FILL_ROWS = 16;  // rows a warp moves per step
constexpr int FILL_CTAS_PER_SM = 4;

// A 16-byte load that does not allocate in L1 (the source is read once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// A 16-byte store of a Cache Buffer row, evicted from L2 first.  The fill of
// a layer runs while the layer before it computes (the lookup is one layer
// ahead), so the hundreds of MB that attention streams would evict the rows
// before their own attention reads them anyway; the hint keeps them from
// pushing out what the kernels around the fill reuse.  (On the B8 32K
// full-miss fill from HBM it measured 35.0 -> 34.6 us; the same hint on the
// loads measured 35.8 us.)
__device__ __forceinline__ void st_row(void* p, const uint4& v, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;\n" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

// The rows of the miss list, moved by the grid's warps.
__device__ __forceinline__ void fill_rows(const FillParams& p) {
    int count = *p.miss_count;
    if (count < 0 || count > p.n_heads) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report_error(p.err_flag, CLO_FLAG_BAD_INDEX);
        count = count < 0 ? 0 : p.n_heads;
    }
    const long long rows = static_cast<long long>(count) * p.k;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, chunk = lane & 15;
    const long long warp0 = static_cast<long long>(blockIdx.x) * FILL_WARPS + (threadIdx.x >> 5);
    const long long nwarps = static_cast<long long>(gridDim.x) * FILL_WARPS;
    const uint64_t policy = l2_evict_first_policy();
    bool bad = false;
    for (long long base = warp0 * FILL_ROWS; base < rows; base += nwarps * FILL_ROWS) {
        // Lane i < 16 resolves row base + i: its head entry, token and slot.
        long long src_row = -1, dst_row = -1;
        const long long i = base + chunk;
        if (lane < FILL_ROWS && i < rows) {
            const int m = static_cast<int>(i / p.k);
            const int j = static_cast<int>(i - static_cast<long long>(m) * p.k);
            const int e = __ldg(p.miss_list + m);
            if (e >= 0 && e < p.n_heads) {
                const long long sel = static_cast<long long>(e) * p.k + j;
                const int t = __ldg(p.tok + sel);
                const int r = p.slot != nullptr ? __ldg(p.slot + sel) : t;
                if (t >= 0 && t < p.T && r >= 0 && r < p.C) {
                    src_row = static_cast<long long>(e) * p.T + t;
                    dst_row = static_cast<long long>(e) * p.C + r;
                } else {
                    bad = true;
                }
            } else {
                bad = true;
            }
        }
        // Half-warp h moves rows h, h + 2, ..., h + 14 of the 16.
        uint4 vk[FILL_ROWS / 2], vv[FILL_ROWS / 2];
        long long dst[FILL_ROWS / 2];
#pragma unroll
        for (int u = 0; u < FILL_ROWS / 2; ++u) {
            const int r = 2 * u + half;
            const long long s = __shfl_sync(FULL_MASK, src_row, r);
            dst[u] = __shfl_sync(FULL_MASK, dst_row, r);
            if (s >= 0) {
                vk[u] = ld_stream(p.srcK + s * FILL_D + chunk * 8);
                vv[u] = ld_stream(p.srcV + s * FILL_D + chunk * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < FILL_ROWS / 2; ++u) {
            if (dst[u] >= 0) {
                st_row(p.cbK + dst[u] * FILL_D + chunk * 8, vk[u], policy);
                st_row(p.cbV + dst[u] * FILL_D + chunk * 8, vv[u], policy);
            }
        }
    }
    if (bad) report_error(p.err_flag, CLO_FLAG_BAD_INDEX);
}

__global__ void __launch_bounds__(FILL_THREADS, FILL_CTAS_PER_SM) fill_kernel(const FillParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the miss list comes from the kernel before
    fill_rows(p);
}

// The fill launched beside the kernel before it (see launch_fill): the miss
// list was written before that kernel started, so the rows move at once, and
// the wait at the end keeps this grid from finishing before that kernel, so
// the kernels after it see both finished.
__global__ void __launch_bounds__(FILL_THREADS, FILL_CTAS_PER_SM)
    fill_beside_kernel(const FillParams p) {
    pdl_launch_dependents();
    fill_rows(p);
    pdl_wait();
}

// Resolves the address the device reads a source buffer through.  Device and
// managed memory are used as they are; pinned host memory through its mapped
// device address; other host memory only where the device can read pageable
// memory (address translation services).  Returns false if the device cannot
// read it, so no kernel is launched on an unreachable pointer.
static bool device_readable(const void*& p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    if (a.type == cudaMemoryTypeHost) {
        if (a.devicePointer == nullptr) return false;
        p = a.devicePointer;
        return true;
    }
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess)
        return false;
    return pageable != 0;
}

clo_status make_fill_params(const clo_half* srcK, const clo_half* srcV, int T, const int32_t* tok,
                            const int32_t* slot, int k, clo_half* cbK, clo_half* cbV, int C,
                            const int32_t* miss_list, const int32_t* miss_count, int B, int Hkv,
                            int d, int32_t* err_flag, FillParams& p, bool& nothing) {
    nothing = false;
    if (B < 0 || Hkv <= 0 || T < 0 || k < 0 || C < 0) return CLO_ERR_INVALID_ARG;
    if (d != FILL_D) return CLO_ERR_UNSUPPORTED;
    if (miss_count == nullptr) return CLO_ERR_INVALID_ARG;
    const long long n_heads = static_cast<long long>(B) * Hkv;
    if (n_heads > (1ll << 30) || static_cast<long long>(T) * n_heads > (1ll << 40) ||
        static_cast<long long>(C) * n_heads > (1ll << 40))
        return CLO_ERR_UNSUPPORTED;
    if (B == 0 || k == 0) {  // nothing to move
        nothing = true;
        return CLO_OK;
    }
    if (srcK == nullptr || srcV == nullptr || tok == nullptr || cbK == nullptr ||
        cbV == nullptr || miss_list == nullptr)
        return CLO_ERR_INVALID_ARG;
    if (slot == nullptr && C < T) return CLO_ERR_INVALID_ARG;  // token-addressed needs C >= T
    const auto aligned = [](const void* q, size_t a) {
        return (reinterpret_cast<uintptr_t>(q) % a) == 0;
    };
    if (!aligned(srcK, 16) || !aligned(srcV, 16) || !aligned(cbK, 16) || !aligned(cbV, 16) ||
        !aligned(tok, 4) || !aligned(slot, 4) || !aligned(miss_list, 4) || !aligned(miss_count, 4))
        return CLO_ERR_INVALID_ARG;

    const void* rK = srcK;
    const void* rV = srcV;
    if (!device_readable(rK) || !device_readable(rV)) return CLO_ERR_INVALID_ARG;

    p.srcK = static_cast<const clo_half*>(rK);
    p.srcV = static_cast<const clo_half*>(rV);
    p.tok = tok;
    p.slot = slot;
    p.cbK = cbK;
    p.cbV = cbV;
    p.miss_list = miss_list;
    p.miss_count = miss_count;
    p.err_flag = err_flag;
    p.T = T;
    p.k = k;
    p.C = C;
    p.n_heads = static_cast<int>(n_heads);
    return CLO_OK;
}

long long fill_max_grid(const FillParams& p) {
    const int sms = device_sm_count();
    if (sms <= 0) return 0;
    const long long max_steps = (static_cast<long long>(p.n_heads) * p.k + FILL_ROWS - 1) / FILL_ROWS;
    long long grid = (max_steps + FILL_WARPS - 1) / FILL_WARPS;
    if (grid > static_cast<long long>(sms) * FILL_CTAS_PER_SM) grid = static_cast<long long>(sms) * FILL_CTAS_PER_SM;
    return grid < 1 ? 1 : grid;
}

// A quarter of the wave (114 of 456 CTA slots on 152 SMs).  Layer calls with
// misses fetched over the host link, µs per layer-step on one box: the B8 32K
// layer 95.2 / 93.8 / 93.5 / 96.1 and the B1 128K step 58.5 / 57.1 / 56.1 /
// 56.0 with 64 / 96 / 128 / 160 fill CTAs.  Fewer CTAs keep too little in
// flight on the link; more take too many slots from the attention.
constexpr int FILL_BESIDE_SHARE = 4;

long long fill_beside_default_ctas(const FillParams& p, int wave) {
    long long n = wave / FILL_BESIDE_SHARE;
    const long long most = fill_max_grid(p);
    if (n > most) n = most;
    return n < 1 ? 1 : n;
}

cudaError_t launch_fill(const FillParams& p, int grid, bool beside, cudaStream_t stream) {
    return launch_pdl(beside ? fill_beside_kernel : fill_kernel, dim3(static_cast<unsigned>(grid)),
                      dim3(FILL_THREADS), 0, stream, p);
}

}  // namespace clo

using namespace clo;

extern "C" clo_status clo_fill_cache_buffer(const clo_half* srcK, const clo_half* srcV, int T,
                                            const int32_t* tok, const int32_t* slot, int k,
                                            clo_half* cbK, clo_half* cbV, int C,
                                            const int32_t* miss_list, const int32_t* miss_count,
                                            int B, int Hkv, int d, int32_t* err_flag,
                                            const clo_attn_opts* opts, cudaStream_t stream) {
    FillParams p;
    bool nothing = false;
    const clo_status st = make_fill_params(srcK, srcV, T, tok, slot, k, cbK, cbV, C, miss_list,
                                           miss_count, B, Hkv, d, err_flag, p, nothing);
    if (st != CLO_OK || nothing) return st;
    long long grid = fill_max_grid(p);
    if (grid <= 0) return CLO_ERR_CUDA;
    if (opts != nullptr && opts->num_ctas > 0) grid = opts->num_ctas;
    if (opts != nullptr && opts->ev_begin != nullptr && !record_event(opts->ev_begin, stream))
        return CLO_ERR_CUDA;
    if (launch_fill(p, static_cast<int>(grid), false, stream) != cudaSuccess) return CLO_ERR_CUDA;
    if (opts != nullptr && opts->ev_end != nullptr && !record_event(opts->ev_end, stream))
        return CLO_ERR_CUDA;
    return CLO_OK;
}
