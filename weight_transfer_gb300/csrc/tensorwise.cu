// Per-tensor ("tensorwise") FP8 scaling: one amax and one scale for the
// whole tensor.
//
// "How to Speed Up VLA Training Step by Step", FP8 paragraph: TorchAO's
// Float8Linear tensorwise recipe computes amax, scale and cast over the
// whole tensor.  The same arithmetic as the blockwise quantizer with a single
// block spanning all n elements:
//   amax = max |x_i|,  s = RN(amax / Fmax),  c_i = satfinite RNE_fp8(RN(x_i / s)).
// Two passes over x: an amax kernel (bf16 magnitudes compared as integers,
// which orders them exactly; one atomicMax per CTA) and an encode kernel
// that derives s from the amax and converts with the per-tensor reciprocal
// and one Markstein step (exact for bf16 dividends, see block_quotients).
// Both stage their tiles with bulk copies on one-pass grids, like the
// blockwise quantizer (the earlier register-load grid-stride kernels took
// about 85-88 us on the 8 x 13.1M bucket).
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

// Both passes stage tiles of 8192 elements (16 KB of bf16) with one bulk
// copy each, two consecutive tiles per CTA of 256 threads on a grid that
// covers the tensor once -- the blockwise quantizer's layout.  A tile's
// ragged end is read from global memory with guarded loads.
constexpr int kTwThreads = 256;
constexpr int kTwTile = 8192;
constexpr int kTwStageBytes = 2 * kTwTile;
constexpr int kTwTilesPerCta = 2;
constexpr size_t kTwSmem = (size_t)kTwTilesPerCta * kTwStageBytes + 8 * kTwTilesPerCta;

// Largest bf16 magnitude bits among the 8 elements of v.
__device__ __forceinline__ uint32_t amax_bits8(const uint4& v, uint32_t m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, max(w[q] & 0x7FFFu, (w[q] >> 16) & 0x7FFFu));
    return m;
}

// The CTA's two tiles requested into their stages (thread 0); returns the
// number of tiles the CTA owns.
__device__ __forceinline__ int tw_request(const uint16_t* x, size_t n, uint8_t* smem, uint64_t* full, size_t t0) {
    const size_t nstaged = n / kTwTile;
    int owned = 0;
    for (int s = 0; s < kTwTilesPerCta; ++s) {
        const size_t t = t0 + s;
        if (t * kTwTile >= n) break;
        owned = s + 1;
        if (threadIdx.x == 0 && t < nstaged) {
            mbar_arrive_expect_tx(&full[s], kTwStageBytes);
            bulk_g2s(smem + (size_t)s * kTwStageBytes, x + t * kTwTile, kTwStageBytes, &full[s]);
        }
    }
    return owned;
}

// Round r of a tile: this thread's 8 elements [e, e + 8) of the tile,
// e = r * 2048 + 8 * tid, from shared memory or (ragged tile) global memory.
__device__ __forceinline__ uint4 tw_load8(const uint8_t* st, bool staged, const uint16_t* x, size_t n, size_t t,
                                          unsigned e) {
    if (staged) return *reinterpret_cast<const uint4*>(st + 2 * e);
    const size_t g = t * kTwTile + e;
    return ld_bf16x8_tail(x + g, (long long)n - (long long)g);
}

// scale_amax[1] accumulates the amax as binary32 bits (non-negative floats
// order like their bit patterns): one atomicMax per CTA.
__global__ void __launch_bounds__(kTwThreads)
tensor_amax_kernel(const uint16_t* __restrict__ x, size_t n, float* scale_amax) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint32_t warp_max[kTwThreads / 32];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTwTilesPerCta * kTwStageBytes);
    const size_t t0 = (size_t)blockIdx.x * kTwTilesPerCta;
    const size_t nstaged = n / kTwTile;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTwTilesPerCta; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    dependency_wait();
    allow_dependents();
    __syncthreads();
    const int owned = tw_request(x, n, smem, full, t0);
    uint32_t m = 0;
    bool ok = true;
    int s = 0;
    for (; s < owned; ++s) {
        const size_t t = t0 + s;
        const bool staged = t < nstaged;
        if (staged && !mbar_wait(&full[s], 0u)) {
            ok = false;
            break;
        }
        const uint8_t* st = smem + (size_t)s * kTwStageBytes;
#pragma unroll
        for (int r = 0; r < kTwTile / (8 * kTwThreads); ++r)
            m = amax_bits8(tw_load8(st, staged, x, n, t, r * 8 * kTwThreads + 8 * threadIdx.x), m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31u) == 0) warp_max[threadIdx.x >> 5] = m;
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) {
            raise_error(kErrCopyTimeout);
            for (int r = s; r < owned; ++r)
                if (t0 + r < nstaged) mbar_wait(&full[r], 0u);
        }
        return;
    }
    if (threadIdx.x == 0) {
        uint32_t c = 0;
        for (int i = 0; i < kTwThreads / 32; ++i) c = max(c, warp_max[i]);
        if (c) atomicMax(reinterpret_cast<unsigned*>(scale_amax) + 1, c << 16);
    }
}

// s from the amax (as the blockwise scale), then each element's code with
// the tensor's reciprocal and one Markstein step (exact for bf16 dividends,
// see block_quotients).
template <int FMT>
__global__ void __launch_bounds__(kTwThreads)
tensor_encode_kernel(const uint16_t* __restrict__ x, size_t n, uint8_t* __restrict__ codes, float* scale_amax) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTwTilesPerCta * kTwStageBytes);
    const size_t t0 = (size_t)blockIdx.x * kTwTilesPerCta;
    const size_t nstaged = n / kTwTile;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTwTilesPerCta; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    // x is an input of the whole call, and the amax kernel before this one
    // does not write it: the tiles may be requested before the wait
    const int owned = tw_request(x, n, smem, full, t0);
    dependency_wait();
    allow_dependents();
    __syncthreads();
    const float amax = scale_amax[1];
    const float s = block_scale<FMT>(amax);
    int si = 0;
    bool ok = true;
    for (; si < owned; ++si) {
        const size_t t = t0 + si;
        const bool staged = t < nstaged;
        if (staged && !mbar_wait(&full[si], 0u)) {
            ok = false;
            break;
        }
        const uint8_t* st = smem + (size_t)si * kTwStageBytes;
#pragma unroll
        for (int r = 0; r < kTwTile / (8 * kTwThreads); ++r) {
            const unsigned e = r * 8 * kTwThreads + 8 * threadIdx.x;
            const uint4 v = tw_load8(st, staged, x, n, t, e);
            float f[8], q[8];
            unpack8(v, f);
            block_quotients<1, 8>(f, s, q);
            const uint32_t w[2] = {cvt_fp8x4<FMT>(q[0], q[1], q[2], q[3]), cvt_fp8x4<FMT>(q[4], q[5], q[6], q[7])};
            const size_t g = t * kTwTile + e;
            if (staged)
                st_stream(codes + g, make_uint2(w[0], w[1]));
            else
                st_u8_tail(codes + g, w, 2, (long long)n - (long long)g);
        }
    }
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) {
            raise_error(kErrCopyTimeout);
            for (int r = si; r < owned; ++r)
                if (t0 + r < nstaged) mbar_wait(&full[r], 0u);
        }
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_amax[0] = s;
}

template <int FMT>
static fp8q_status_t launch_tensorwise(const uint16_t* x, size_t n, uint8_t* codes, float* scale_amax,
                                       cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(scale_amax + 1, 0, sizeof(float), s);
    if (e != cudaSuccess) return cuda_status(e);
    static KernelCache kc1, kc2;
    int r1 = 0, r2 = 0;
    fp8q_status_t pst = prepare_kernel(kc1, tensor_amax_kernel, kTwThreads, kTwSmem, kTwSmem, &r1);
    if (pst == FP8Q_OK) pst = prepare_kernel(kc2, tensor_encode_kernel<FMT>, kTwThreads, kTwSmem, kTwSmem, &r2);
    if (pst != FP8Q_OK) return pst;
    const size_t tiles = (n + kTwTile - 1) / kTwTile;
    const size_t grid = (tiles + kTwTilesPerCta - 1) / kTwTilesPerCta;
    if (grid > 0x7FFFFFFFu) return FP8Q_ERR_SIZE;
    const fp8q_status_t st = launch(tensor_amax_kernel, (unsigned)grid, kTwThreads, kTwSmem, s, x, n, scale_amax);
    if (st != FP8Q_OK) return st;
    return launch(tensor_encode_kernel<FMT>, (unsigned)grid, kTwThreads, kTwSmem, s, x, n, codes, scale_amax);
}

unsigned unit_errors_tensorwise(bool clear) { return read_unit_errors(clear); }

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status_t fp8q_quantize_tensorwise(const void* x_bf16, size_t n, fp8q_format_t fmt, uint8_t* codes,
                                                  float* scale_amax, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_quantize_tensorwise");
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!x_bf16 || !codes || !scale_amax) return FP8Q_ERR_NULL;
    if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(scale_amax)) return FP8Q_ERR_ALIGN;
    if (overlaps(codes, n, x_bf16, 2 * n) || overlaps(scale_amax, 8, x_bf16, 2 * n) || overlaps(scale_amax, 8, codes, n))
        return FP8Q_ERR_ALIAS;
    const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3 ? launch_tensorwise<kE4M3>(x, n, codes, scale_amax, s)
                            : launch_tensorwise<kE5M2>(x, n, codes, scale_amax, s);
}
