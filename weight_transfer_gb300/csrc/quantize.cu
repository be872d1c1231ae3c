// (a) Blockwise FP8 quantize, and the plain fp32 -> FP8 element conversion.
//
// "FP8 Transmission Optimization for VLA Training", intro ("blockwise
// scaling") and "FP8 Transmission Optimization and Bottlenecks" (e4m3/e5m2):
// one fp32 scale per 128-element block, scale = amax / Fmax, codes are the
// satfinite round-to-nearest-even conversion of x / scale.
//
// Work split: 8 lanes own one 128-element block; lane j holds elements
// [8j, 8j+8) and [64+8j, 64+8j+8), so each of the two 16-byte load
// instructions of a warp reads four whole 128-byte half-blocks.  A warp covers
// 4 blocks per step and U steps are loaded before any is processed (2U
// independent 16-byte loads in flight per lane).  The block amax is a 3-step
// xor-shuffle inside the 8-lane group; the quotients x / s use the per-block
// reciprocal with one Markstein correction (exact for bf16 dividends, see
// block_quotients).  The grid is persistent (SM count x resident blocks).
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 2;

template <int FMT, int U>
__global__ void __launch_bounds__(kQuantThreads)
quantize_blockwise_kernel(const uint16_t* __restrict__ x, size_t n, uint8_t* __restrict__ codes,
                          float* __restrict__ scales) {
    const size_t nb = (n + 127) >> 7;       // blocks, the last one possibly partial
    const size_t nfull = n >> 7;            // full blocks
    const unsigned lane = threadIdx.x & 31u;
    const unsigned j = lane & 7u;           // lane inside the block's 8-lane group
    const unsigned sub = lane >> 3;         // which of the warp's 4 blocks
    const size_t warp = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;

    // the loop bound is warp-uniform so every shuffle below has all 32 lanes
    for (size_t base = warp; 4 * base < nb; base += nwarps * U) {
        uint4 va[U], vb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t b = 4 * (base + (size_t)u * nwarps) + sub;
            const size_t e0 = (b << 7) + 8 * j;
            if (b < nfull) {
                va[u] = ld_stream(x + e0);
                vb[u] = ld_stream(x + e0 + 64);
            } else if (b < nb) {
                va[u] = ld_bf16x8_tail(x + e0, (long long)n - (long long)e0);
                vb[u] = ld_bf16x8_tail(x + e0 + 64, (long long)n - (long long)e0 - 64);
            } else {
                va[u] = make_uint4(0u, 0u, 0u, 0u);
                vb[u] = va[u];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t b = 4 * (base + (size_t)u * nwarps) + sub;
            const size_t e0 = (b << 7) + 8 * j;
            float f[16];
            unpack8(va[u], *reinterpret_cast<float(*)[8]>(f));
            unpack8(vb[u], *reinterpret_cast<float(*)[8]>(f + 8));
            float a = fabsf(f[0]);
#pragma unroll
            for (int i = 1; i < 16; ++i) a = fmaxf(a, fabsf(f[i]));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
            const float s = block_scale<FMT>(a);
            float q[16];
            block_quotients<1, 16>(f, s, q);
            uint32_t wa[2] = {cvt_fp8x4<FMT>(q[0], q[1], q[2], q[3]), cvt_fp8x4<FMT>(q[4], q[5], q[6], q[7])};
            uint32_t wb[2] = {cvt_fp8x4<FMT>(q[8], q[9], q[10], q[11]), cvt_fp8x4<FMT>(q[12], q[13], q[14], q[15])};
            if (b < nfull) {
                st_stream(codes + e0, make_uint2(wa[0], wa[1]));
                st_stream(codes + e0 + 64, make_uint2(wb[0], wb[1]));
            } else if (b < nb) {
                st_u8_tail(codes + e0, wa, 2, (long long)n - (long long)e0);
                st_u8_tail(codes + e0 + 64, wb, 2, (long long)n - (long long)e0 - 64);
            }
            if (b < nb && j == 0) scales[b] = s;
        }
    }
}

// Elementwise conversion: 4 floats per lane per step.
template <int FMT>
__global__ void __launch_bounds__(256)
encode_f32_kernel(const float* __restrict__ x, size_t n, uint8_t* __restrict__ codes) {
    const size_t n4 = n >> 2;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const uint4 v = ld_stream(x + 4 * i);
        const uint32_t c = cvt_fp8x4<FMT>(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                                          __uint_as_float(v.w));
        asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(codes + 4 * i), "r"(c) : "memory");
    }
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < (n & 3)) {
        const size_t i = (n4 << 2) + t;
        codes[i] = (uint8_t)cvt_fp8x2<FMT>(x[i], 0.0f);
    }
}

template <int FMT>
static fp8q_status_t launch_quantize(const uint16_t* x, size_t n, uint8_t* codes, float* scales,
                                     cudaStream_t stream) {
    static int resident = resident_blocks(quantize_blockwise_kernel<FMT, kQuantUnroll>, kQuantThreads);
    const size_t nb = (n + 127) / 128;
    const size_t blocks_per_cta = (kQuantThreads / 8) * kQuantUnroll;
    const unsigned grid = grid_for((nb + blocks_per_cta - 1) / blocks_per_cta, resident);
    quantize_blockwise_kernel<FMT, kQuantUnroll><<<grid, kQuantThreads, 0, stream>>>(x, n, codes, scales);
    return launch_status();
}

template <int FMT>
static fp8q_status_t launch_encode(const float* x, size_t n, uint8_t* codes, cudaStream_t stream) {
    static int resident = resident_blocks(encode_f32_kernel<FMT>, 256);
    const size_t units = (n + 3) / 4;
    const unsigned grid = grid_for((units + 255) / 256, resident * 2);
    encode_f32_kernel<FMT><<<grid, 256, 0, stream>>>(x, n, codes);
    return launch_status();
}

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status_t fp8q_quantize_blockwise(const void* x_bf16, size_t n, fp8q_format_t fmt,
                                                 uint8_t* codes, float* scales, fp8q_stream_t stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!x_bf16 || !codes || !scales) return FP8Q_ERR_NULL;
    if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(scales)) return FP8Q_ERR_ALIGN;
    const size_t nb = fp8q_num_scales(n);
    if (overlaps(codes, n, x_bf16, 2 * n) || overlaps(scales, 4 * nb, x_bf16, 2 * n) ||
        overlaps(codes, n, scales, 4 * nb))
        return FP8Q_ERR_ALIAS;
    const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3 ? launch_quantize<kE4M3>(x, n, codes, scales, s)
                            : launch_quantize<kE5M2>(x, n, codes, scales, s);
}

extern "C" fp8q_status_t fp8q_encode_f32(const float* x, size_t n, fp8q_format_t fmt, uint8_t* codes,
                                         fp8q_stream_t stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!x || !codes) return FP8Q_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes)) return FP8Q_ERR_ALIGN;
    if (overlaps(codes, n, x, 4 * n)) return FP8Q_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3 ? launch_encode<kE4M3>(x, n, codes, s) : launch_encode<kE5M2>(x, n, codes, s);
}
