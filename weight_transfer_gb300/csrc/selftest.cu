// Self-test of the bounded copy wait that every staged kernel relies on.
//
// Each staged kernel waits for its shared-memory copies on an mbarrier, and
// gives up after a wall-clock limit instead of hanging: the CTA votes, raises
// the copy time-out error bit, and returns (fail loudly rather than hang or
// return garbage silently -- "perf: Reduce MXFP8 refit weight-transfer
// overheads", Safety).  A copy that never lands cannot be produced on
// purpose without a fault, so this kernel makes the same wait run out the
// one safe way: it arms its barrier for 16 transaction bytes and issues no
// copy, so nothing is ever in flight into its shared memory and the phase
// never completes.  Given a source, it issues the 16-byte copy instead and
// the wait completes.
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kSelftestThreads = 64;

__global__ void __launch_bounds__(kSelftestThreads)
copy_wait_selftest_kernel(const uint4* src, uint4* dst, unsigned long long limit_ns) {
    __shared__ __align__(16) uint4 stage;
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, 16);
        if (src != nullptr) bulk_g2s(&stage, src, 16, &bar);
    }
    const bool ok = mbar_wait(&bar, 0u, limit_ns);
    // the staged kernels' give-up path: a CTA-wide vote, one error bit
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) raise_error(kErrCopyTimeout);
        return;
    }
    if (threadIdx.x == 0 && dst != nullptr) *dst = stage;
}

unsigned unit_errors_selftest(bool clear) { return read_unit_errors(clear); }

}  // namespace fp8q

extern "C" fp8q_status_t fp8q_selftest_copy_wait(const void* src, void* dst, uint64_t limit_ns,
                                                 fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_selftest_copy_wait");
    using namespace fp8q;
    if ((src == nullptr) != (dst == nullptr)) return FP8Q_ERR_NULL;
    if (src != nullptr && (!aligned16(src) || !aligned16(dst))) return FP8Q_ERR_ALIGN;
    if (src != nullptr && overlaps(src, 16, dst, 16)) return FP8Q_ERR_ALIAS;
    if (limit_ns < FP8Q_SELFTEST_MIN_WAIT_NS || limit_ns > FP8Q_SELFTEST_MAX_WAIT_NS) return FP8Q_ERR_SIZE;
    return launch(copy_wait_selftest_kernel, 1, kSelftestThreads, 0, stream, static_cast<const uint4*>(src),
                  static_cast<uint4*>(dst), (unsigned long long)limit_ns);
}
