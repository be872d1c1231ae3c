// Entry points with no kernel of their own: size helpers, status strings,
// CUDA error capture and the cached device query used for launch sizing.
#include "fp8q_host.cuh"

#include <atomic>

namespace fp8q {

static thread_local int g_last_cuda_error = 0;
static std::atomic<int> g_launch_overlap{1};

bool launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }

fp8q_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FP8Q_OK;
    g_last_cuda_error = (int)e;
    return FP8Q_ERR_CUDA;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return 1;
    if (dev < kMaxDevices) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace fp8q

extern "C" size_t fp8q_num_scales(size_t n) { return n / FP8Q_BLOCK + (n % FP8Q_BLOCK != 0); }

extern "C" int fp8q_set_launch_overlap(int enable) {
    return fp8q::g_launch_overlap.exchange(enable != 0 ? 1 : 0);
}

extern "C" int fp8q_last_cuda_error(void) { return fp8q::g_last_cuda_error; }

extern "C" const char* fp8q_status_string(fp8q_status_t status) {
    switch (status) {
        case FP8Q_OK: return "ok";
        case FP8Q_ERR_NULL: return "a required pointer is NULL";
        case FP8Q_ERR_SIZE: return "size out of range";
        case FP8Q_ERR_ALIGN: return "pointer not 16-byte aligned";
        case FP8Q_ERR_FORMAT: return "unknown FP8 format";
        case FP8Q_ERR_K: return "shard count or MXFP8 K out of range";
        case FP8Q_ERR_CUDA: return "CUDA launch error (see fp8q_last_cuda_error)";
        case FP8Q_ERR_ALIAS: return "an output overlaps an input or another output";
        case FP8Q_ERR_FLAGS: return "unknown bits in a flags argument";
    }
    return "unknown status";
}

extern "C" fp8q_status_t fp8q_device_errors(unsigned int* flags, int clear) {
    if (!flags) return FP8Q_ERR_NULL;
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fp8q::cuda_status(e);
    *flags = fp8q::unit_errors_quantize(clear != 0) | fp8q::unit_errors_reduce(clear != 0) |
             fp8q::unit_errors_ring_hop(clear != 0) | fp8q::unit_errors_mxfp8(clear != 0) |
             fp8q::unit_errors_selftest(clear != 0) | fp8q::unit_errors_tensorwise(clear != 0);
    return FP8Q_OK;
}
