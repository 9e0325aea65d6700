// clo_sync.cu -- GPU-centric data-ready synchronisation ("CLO: CPU-Light
// KVCache Offloading", section 2 Q1 "GPU-centric synchronisation" and Fig. 8's
// Data Synchronization Controller): a host thread that moves data for the GPU
// publishes a sequence number in host memory the GPU can read, and a kernel
// already queued on the stream polls it, so the thread that launches kernels
// never blocks in cudaStreamSynchronize and the launches run ahead of the
// data.
//
// The poll is bounded.  It gives up after the caller's time limit (read from
// %globaltimer) or an iteration cap derived from it, whichever comes first,
// ORs CLO_FLAG_TIMEOUT into the error flag and returns; the kernels queued
// after it then run on whatever the memory holds, and the caller reads the
// flag after the stream synchronises.  No wait in this library is unbounded.
#include <atomic>

#include "clo_device.cuh"

namespace clo {

constexpr unsigned WAIT_SLEEP_NS = 256;          // back-off between polls
constexpr uint32_t WAIT_MAX_US = 10u * 1000u * 1000u;  // longest limit a call may ask for

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Acquire load at system scope: every write the host made before it stored
// the value (with release ordering) is visible to this GPU afterwards.
__device__ __forceinline__ uint32_t load_acquire_sys(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One warp; lane 0 polls until (int32_t)(*ready - expected) >= 0 (sequence
// numbers, so the comparison survives wrap-around) or the limit passes.
__global__ void __launch_bounds__(32, 1)
    wait_ready_kernel(const uint32_t* ready, uint32_t expected, uint64_t limit_ns,
                      uint64_t max_polls, int32_t* err_flag) {
    pdl_wait();  // ordered after everything queued before it
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_ns();
        bool ok = false;
        for (uint64_t i = 0; i < max_polls; ++i) {
            if (static_cast<int32_t>(load_acquire_sys(ready) - expected) >= 0) {
                ok = true;
                break;
            }
            if (global_ns() - t0 >= limit_ns) break;
            __nanosleep(WAIT_SLEEP_NS);
        }
        if (!ok) report_error(err_flag, CLO_FLAG_TIMEOUT);
    }
    __syncwarp();
    // Dependents may start only now; they still wait, at their own
    // dependency wait, for this grid to finish and flush.
    pdl_launch_dependents();
}

}  // namespace clo

using namespace clo;

extern "C" clo_status clo_wait_ready(const uint32_t* ready, uint32_t expected,
                                     uint32_t timeout_us, int32_t* err_flag,
                                     cudaStream_t stream) {
    if (ready == nullptr || (reinterpret_cast<uintptr_t>(ready) % 4) != 0)
        return CLO_ERR_INVALID_ARG;
    if (timeout_us == 0 || timeout_us > WAIT_MAX_US) return CLO_ERR_INVALID_ARG;
    // The flag must be memory the device reads in place: device or managed
    // memory, or pinned host memory through its mapped address.
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ready) != cudaSuccess) {
        (void)cudaGetLastError();
        return CLO_ERR_INVALID_ARG;
    }
    const uint32_t* dptr = ready;
    if (a.type == cudaMemoryTypeHost) {
        if (a.devicePointer == nullptr) return CLO_ERR_INVALID_ARG;
        dptr = static_cast<const uint32_t*>(a.devicePointer);
    } else if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) {
        return CLO_ERR_INVALID_ARG;
    }
    const uint64_t limit_ns = static_cast<uint64_t>(timeout_us) * 1000u;
    // A poll (an acquire load over the host link plus the back-off) takes
    // well over 100 ns, so this cap is never the binding limit unless the
    // clock misbehaves.
    const uint64_t max_polls = limit_ns / 100u + 1024u;
    if (!prepare_kernel(reinterpret_cast<const void*>(wait_ready_kernel), 0)) return CLO_ERR_CUDA;
    return launch_pdl(wait_ready_kernel, dim3(1), dim3(32), 0, stream, dptr, expected, limit_ns,
                      max_polls, err_flag) == cudaSuccess
               ? CLO_OK
               : CLO_ERR_CUDA;
}

extern "C" clo_status clo_signal_ready(uint32_t* ready, uint32_t value) {
    if (ready == nullptr || (reinterpret_cast<uintptr_t>(ready) % 4) != 0)
        return CLO_ERR_INVALID_ARG;
    // Release: the caller's earlier writes (the data the GPU is waiting for)
    // are ordered before the value becomes visible.
    std::atomic_thread_fence(std::memory_order_release);
    __atomic_store_n(ready, value, __ATOMIC_RELEASE);
    return CLO_OK;
}
