// clo_copy.cu -- clo_copy_async: a list of copies between device memory and
// pinned host memory, for callers that keep a step's inputs or results on
// the host.  The pages have no counterpart; nothing here computes.
//
// Copies whose two sides the GPU can address (device or managed memory, or
// pinned host memory through its mapped device address) are made by one
// kernel launch per run of up to COPY_MAX such copies: the SMs read and write
// host memory over the host link themselves.  Copies with both ends 16-byte
// aligned move 16 bytes a thread, any others (up to COPY_SMALL bytes) a byte
// a thread.  That launch takes part in programmatic dependent launch like
// every other libclo kernel, so it chains with the kernels around it; a
// copy-engine copy between two kernels would make the second wait for the
// first to drain and for the copy before it could start.  Any other copy
// goes to cudaMemcpyAsync.  The copies of one call may run at the same time,
// so the call refuses lists whose copies overlap.
#include <algorithm>
#include <vector>

#include "clo_device.cuh"

namespace clo {

constexpr int COPY_MAX = 16;       // copies a launch
constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;     // independent 16-byte loads a thread keeps in flight
constexpr int COPY_CTAS_PER_SM = 8;
constexpr size_t COPY_SMALL = 64 * 1024;  // largest copy the kernel makes a byte at a time

struct CopyList {
    char* dst[COPY_MAX];
    const char* src[COPY_MAX];
    long long bytes[COPY_MAX];
};

__device__ __forceinline__ bool both_aligned16(const void* a, const void* b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}

// Copy blockIdx.y of the list; the CTAs along x stride over it: 16-byte
// units when both ends are 16-byte aligned, then the bytes past the last
// whole unit (all of them otherwise).
__global__ void __launch_bounds__(COPY_THREADS) copy_kernel(const CopyList c) {
    pdl_launch_dependents();
    pdl_wait();  // the source may come from the kernel before
    const int i = blockIdx.y;
    const char* __restrict__ src = c.src[i];
    char* __restrict__ dst = c.dst[i];
    const long long bytes = c.bytes[i];
    const long long n = both_aligned16(dst, src) ? bytes / 16 : 0;
    const uint4* __restrict__ src16 = reinterpret_cast<const uint4*>(src);
    uint4* __restrict__ dst16 = reinterpret_cast<uint4*>(dst);
    const long long stride = static_cast<long long>(gridDim.x) * COPY_THREADS;
    const long long first = static_cast<long long>(blockIdx.x) * COPY_THREADS + threadIdx.x;
    for (long long base = first; base < n; base += stride * COPY_UNROLL) {
        uint4 v[COPY_UNROLL];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const long long j = base + u * stride;
            if (j < n) v[u] = src16[j];
        }
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u) {
            const long long j = base + u * stride;
            if (j < n) dst16[j] = v[u];
        }
    }
    for (long long b = n * 16 + first; b < bytes; b += stride) dst[b] = src[b];
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

// most: the largest copy of the batch in work units (16-byte units, or bytes
// for a byte copy).
static clo_status launch_copies(const CopyList& c, int n, long long most, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (sms <= 0) return CLO_ERR_CUDA;
    long long gx = (most + static_cast<long long>(COPY_THREADS) * COPY_UNROLL - 1) /
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
    // another one (or itself) reads or writes; reads may overlap reads.  The
    // byte ranges (all pointers share the unified address space) are swept in
    // address order: a range that starts below the end of an earlier write,
    // or a write that starts below the end of any earlier range, overlaps it.
    struct Range {
        uintptr_t lo, hi;
        bool write;
    };
    std::vector<Range> ranges;
    try {
        ranges.reserve(2 * static_cast<size_t>(n));
    } catch (...) {  // no exception leaves the library
        return CLO_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < n; ++i) {
        const clo_copy& cp = copies[i];
        if (cp.bytes == 0) continue;
        const uintptr_t d = reinterpret_cast<uintptr_t>(cp.dst);
        const uintptr_t r = reinterpret_cast<uintptr_t>(cp.src);
        if (d + cp.bytes < d || r + cp.bytes < r) return CLO_ERR_INVALID_ARG;  // wraps around
        ranges.push_back({d, d + cp.bytes, true});
        ranges.push_back({r, r + cp.bytes, false});
    }
    std::sort(ranges.begin(), ranges.end(),
              [](const Range& a, const Range& b) { return a.lo < b.lo; });
    uintptr_t end_any = 0, end_write = 0;
    for (const Range& g : ranges) {
        if (g.lo < end_write || (g.write && g.lo < end_any)) return CLO_ERR_INVALID_ARG;
        end_any = std::max(end_any, g.hi);
        if (g.write) end_write = std::max(end_write, g.hi);
    }
    CopyList batch{};
    int nb = 0;
    long long most = 0;
    for (int i = 0; i < n; ++i) {
        const clo_copy& cp = copies[i];
        if (cp.bytes == 0) continue;
        void* d = device_address(cp.dst);
        const void* s = device_address(cp.src);
        const bool vec = d != nullptr && s != nullptr && aligned16(d) && aligned16(s);
        const bool by_kernel = d != nullptr && s != nullptr && (vec || cp.bytes <= COPY_SMALL);
        if (by_kernel) {
            batch.dst[nb] = static_cast<char*>(d);
            batch.src[nb] = static_cast<const char*>(s);
            batch.bytes[nb] = static_cast<long long>(cp.bytes);
            most = std::max(most, static_cast<long long>(vec ? (cp.bytes + 15) / 16 : cp.bytes));
            if (++nb == COPY_MAX) {
                const clo_status st = launch_copies(batch, nb, most, stream);
                if (st != CLO_OK) return st;
                nb = 0;
                most = 0;
            }
            continue;
        }
        if (nb > 0) {  // keep the list order
            const clo_status st = launch_copies(batch, nb, most, stream);
            if (st != CLO_OK) return st;
            nb = 0;
            most = 0;
        }
        if (cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDefault, stream) != cudaSuccess)
            return CLO_ERR_CUDA;
    }
    if (nb > 0) return launch_copies(batch, nb, most, stream);
    return CLO_OK;
}
