// Host-side helpers shared by the fp8q entry points: argument checks that
// run before any launch, launch sizing, and CUDA error capture.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "fp8q.h"

// Optional NVTX ranges around every entry point that queues GPU work, for
// timelines in Nsight tools ("FP8 Transmission Optimization for VLA
// Training", Other Technical Findings: the transfer path was instrumented
// with NVTX).  Compiled in only when the library is built with FP8Q_NVTX
// defined (FP8Q_NVTX=1 in the environment of weight_transfer_gb300/build.py);
// off by default, and then the macro expands to nothing.  NVTX v3 is
// header-only: without a tool attached a range costs one branch.
#ifdef FP8Q_NVTX
#include <nvtx3/nvToolsExt.h>
namespace fp8q {
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace fp8q
#define FP8Q_NVTX_RANGE(name) ::fp8q::NvtxRange fp8q_nvtx_range_(name)
#else
#define FP8Q_NVTX_RANGE(name) ((void)0)
#endif

namespace fp8q {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) overlap (empty ranges never do).
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline bool valid_fmt(fp8q_format_t f) { return f == FP8Q_E4M3 || f == FP8Q_E5M2; }

// Records and maps a CUDA error (thread-local, see fp8q_last_cuda_error).
fp8q_status_t cuda_status(cudaError_t e);

// Status of the launch just made on this thread.
inline fp8q_status_t launch_status() { return cuda_status(cudaGetLastError()); }

// Error bits raised by the kernels of each translation unit since the last
// clear (read after the caller has synchronized the device).
unsigned unit_errors_quantize(bool clear);
unsigned unit_errors_reduce(bool clear);
unsigned unit_errors_ring_hop(bool clear);
unsigned unit_errors_mxfp8(bool clear);
unsigned unit_errors_selftest(bool clear);
unsigned unit_errors_tensorwise(bool clear);

// Devices whose per-device state is cached; others are set up on every call.
constexpr int kMaxDevices = 64;

// The calling thread's current device, or -1.
int current_device();

// SM count of the current device (cached per device).
int sm_count();

// Blocks of `threads` threads of `kernel` that fit on one SM.
template <class K>
int resident_blocks(K kernel, int threads, size_t smem = 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

// One-time preparation of a kernel on each device: the opt-in to more than
// 48 KB of dynamic shared memory (a function attribute that applies to the
// device current when it is set) and the kernel's resident blocks per SM.
// Cached per device, so that one process may drive several GPUs; concurrent
// first calls repeat the same idempotent work.  A cache object must have
// static storage duration (its counters start at zero).
struct KernelCache {
    std::atomic<int> resident[kMaxDevices];
};

template <class K>
fp8q_status_t prepare_kernel(KernelCache& kc, K kernel, int threads, size_t smem, size_t smem_optin, int* resident) {
    const int dev = current_device();
    const bool cached = dev >= 0 && dev < kMaxDevices;
    int r = cached ? kc.resident[dev].load(std::memory_order_acquire) : 0;
    if (r == 0) {
        if (smem_optin > 0) {
            const cudaError_t e =
                cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_optin);
            if (e != cudaSuccess) return cuda_status(e);
        }
        r = resident_blocks(kernel, threads, smem);
        if (cached) kc.resident[dev].store(r, std::memory_order_release);
    }
    *resident = r;
    return FP8Q_OK;
}

// Persistent grid: enough blocks to fill every SM `resident` deep, but never
// more than there is work for.
inline unsigned grid_for(size_t work_blocks, int resident) {
    size_t cap = (size_t)sm_count() * (size_t)(resident > 0 ? resident : 1);
    size_t g = work_blocks < cap ? work_blocks : cap;
    return (unsigned)(g > 0 ? g : 1);
}

// The all-gather decode of the simulated ring AllReduce: n codes and their
// scales decoded once, the bf16 values written to each of the `count`
// outputs (count <= FP8Q_MAX_HOP_GROUP); with mean_divisor > 0 each decoded
// value is divided by it (true division) before the bf16 rounding.
fp8q_status_t gather_decode_entry(const uint8_t* codes, const float* scales, size_t n, fp8q_format_t fmt,
                                  void* const* outs, int count, int mean_divisor, fp8q_stream_t stream);

// Process-wide switch of programmatic dependent launch (fp8q_set_launch_overlap).
bool launch_overlap();

// Launches `kernel` on `stream`, with programmatic stream serialization when
// the switch is on (the kernel then waits on the device for its predecessor,
// see dependency_wait), and returns the launch status.
template <typename... KArgs, typename... Args>
fp8q_status_t launch(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = launch_overlap() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) (void)cudaGetLastError();     // leave no error behind for later launches
    return cuda_status(e);
}

}  // namespace fp8q
