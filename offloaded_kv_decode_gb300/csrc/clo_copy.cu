// clo_copy.cu -- clo_copy_async: a list of copies between device memory and
// pinned host memory, for callers that keep a step's inputs or results on
// the host.  The pages have no counterpart; nothing here computes.
//
// Copies whose two sides the GPU can address (device or managed memory, or
// pinned host memory through its mapped device address), 16-byte aligned
// and a multiple of 16 bytes long, are made by one kernel launch per run of
// up to COPY_MAX such copies: the SMs read and write host memory over the
// host link themselves.  That launch takes part in programmatic dependent
// launch like every other libclo kernel, so it chains with the kernels
// around it; a copy-engine copy between two kernels would make the second
// wait for the first to drain and for the copy before it could start.  Any
// other copy goes to cudaMemcpyAsync.  The copies of one call may run at the
// same time, so the call refuses lists whose copies overlap.
#include <algorithm>

#include "clo_device.cuh"

namespace clo {

constexpr int COPY_MAX = 16;       // copies a launch
constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;     // independent 16-byte loads a thread keeps in flight
constexpr int COPY_CTAS_PER_SM = 8;

struct CopyList {
    uint4* dst[COPY_MAX];
    const uint4* src[COPY_MAX];
    long long n16[COPY_MAX];  // 16-byte units
};

// Copy blockIdx.y of the list; the CTAs along x stride over its units.
__global__ void __launch_bounds__(COPY_THREADS) copy_kernel(const CopyList c) {
    pdl_launch_dependents();
    pdl_wait();  // the source may come from the kernel before
    const int i = blockIdx.y;
    const uint4* __restrict__ src = c.src[i];
    uint4* __restrict__ dst = c.dst[i];
    const long long n = c.n16[i];
    const long long stride = static_cast<long long>(gridDim.x) * COPY_THREADS;
    for (long long base = static_cast<long long>(blockIdx.x) * COPY_THREADS + threadIdx.x;
         base < n; base += stride * COPY_UNROLL) {
        uint4 v[COPY_UNROLL];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const long long j = base + u * stride;
            if (j < n) v[u] = src[j];
        }
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const long long j = base + u * stride;
            if (j < n) dst[j] = v[u];
        }
    }
}

// The address the GPU reaches p through, or nullptr if it cannot (pageable
// host memory, unknown pointers): device and managed memory as they are,
// pinned host memory through its mapped device address.
static void* device_address(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged)
        return const_cast<void*>(p);
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static clo_status launch_copies(const CopyList& c, int n, long long most16, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (sms <= 0) return CLO_ERR_CUDA;
    long long gx = (most16 + static_cast<long long>(COPY_THREADS) * COPY_UNROLL - 1) /
                   (static_cast<long long>(COPY_THREADS) * COPY_UNROLL);
    const long long cap = static_cast<long long>(sms) * COPY_CTAS_PER_SM / n;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    if (launch_pdl(copy_kernel, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(n)),
                   dim3(COPY_THREADS), 0, stream, c) != cudaSuccess)
        return CLO_ERR_CUDA;
    return CLO_OK;
}

}  // namespace clo

using namespace clo;

extern "C" clo_status clo_copy_async(const clo_copy* copies, int n, cudaStream_t stream) {
    if (n < 0 || (n > 0 && copies == nullptr)) return CLO_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (copies[i].bytes > 0 && (copies[i].dst == nullptr || copies[i].src == nullptr))
            return CLO_ERR_INVALID_ARG;
    // Copies of one call may run at the same time: none may write bytes that
    // another one reads or writes (all pointers share the unified address space).
    const auto overlap = [](const void* a, const void* b, size_t na, size_t nb) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + nb && y < x + na;
    };
    for (int i = 0; i < n; ++i) {
        const clo_copy& a = copies[i];
        if (a.bytes == 0) continue;
        if (overlap(a.dst, a.src, a.bytes, a.bytes)) return CLO_ERR_INVALID_ARG;
        for (int j = i + 1; j < n; ++j) {
            const clo_copy& b = copies[j];
            if (b.bytes == 0) continue;
            if (overlap(a.dst, b.dst, a.bytes, b.bytes) || overlap(a.dst, b.src, a.bytes, b.bytes) ||
                overlap(a.src, b.dst, a.bytes, b.bytes))
                return CLO_ERR_INVALID_ARG;
        }
    }
    CopyList batch{};
    int nb = 0;
    long long most16 = 0;
    for (int i = 0; i < n; ++i) {
        const clo_copy& cp = copies[i];
        if (cp.bytes == 0) continue;
        void* d = device_address(cp.dst);
        const void* s = device_address(cp.src);
        const bool by_kernel = d != nullptr && s != nullptr && aligned16(d) && aligned16(s) &&
                               cp.bytes % 16 == 0;
        if (by_kernel) {
            batch.dst[nb] = static_cast<uint4*>(d);
            batch.src[nb] = static_cast<const uint4*>(s);
            batch.n16[nb] = static_cast<long long>(cp.bytes / 16);
            most16 = std::max(most16, batch.n16[nb]);
            if (++nb == COPY_MAX) {
                const clo_status st = launch_copies(batch, nb, most16, stream);
                if (st != CLO_OK) return st;
                nb = 0;
                most16 = 0;
            }
            continue;
        }
        if (nb > 0) {  // keep the list order
            const clo_status st = launch_copies(batch, nb, most16, stream);
            if (st != CLO_OK) return st;
            nb = 0;
            most16 = 0;
        }
        if (cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDefault, stream) != cudaSuccess)
            return CLO_ERR_CUDA;
    }
    if (nb > 0) return launch_copies(batch, nb, most16, stream);
    return CLO_OK;
}
