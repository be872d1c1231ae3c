// Per-tensor ("tensorwise") FP8 scaling: one amax and one scale for the
// whole tensor.
//
// "How to Speed Up VLA Training Step by Step", FP8 paragraph: TorchAO's
// Float8Linear tensorwise recipe computes amax, scale and cast over the
// whole tensor.  The same arithmetic as the blockwise quantizer with a single
// block spanning all n elements:
//   amax = max |x_i|,  s = RN(amax / Fmax),  c_i = satfinite RNE_fp8(RN(x_i / s)).
// Two passes over x: an amax kernel (bf16 magnitudes compared as integers,
// which orders them exactly; one atomicMax per warp) and an encode kernel
// that derives s from the amax and converts with the per-tensor reciprocal
// and one Markstein step (exact for bf16 dividends, see block_quotients).
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

// Largest bf16 magnitude bits among the 8 elements of v.
__device__ __forceinline__ uint32_t amax_bits8(const uint4& v, uint32_t m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, max(w[q] & 0x7FFFu, (w[q] >> 16) & 0x7FFFu));
    return m;
}

// scale_amax[1] accumulates the amax as binary32 bits (non-negative floats
// order like their bit patterns).  Each thread keeps four 16-byte loads in
// flight: with one, the loads a GPU can hold in flight do not cover HBM's
// latency at full bandwidth.
__global__ void __launch_bounds__(256)
tensor_amax_kernel(const uint16_t* __restrict__ x, size_t n, float* scale_amax) {
    dependency_wait();
    allow_dependents();
    uint32_t m = 0;
    const size_t n8 = n / 8;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t i = t0;
    for (; i + 3 * stride < n8; i += 4 * stride) {
        const uint4 v0 = ld_stream(x + 8 * i);
        const uint4 v1 = ld_stream(x + 8 * (i + stride));
        const uint4 v2 = ld_stream(x + 8 * (i + 2 * stride));
        const uint4 v3 = ld_stream(x + 8 * (i + 3 * stride));
        m = amax_bits8(v3, amax_bits8(v2, amax_bits8(v1, amax_bits8(v0, m))));
    }
    for (; i < n8; i += stride) m = amax_bits8(ld_stream(x + 8 * i), m);
    for (size_t i = 8 * n8 + t0; i < n; i += stride) m = max(m, (uint32_t)(x[i] & 0x7FFFu));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31u) == 0 && m) atomicMax(reinterpret_cast<unsigned*>(scale_amax) + 1, m << 16);
}

template <int FMT>
__global__ void __launch_bounds__(256)
tensor_encode_kernel(const uint16_t* __restrict__ x, size_t n, uint8_t* __restrict__ codes, float* scale_amax) {
    dependency_wait();
    allow_dependents();
    const float amax = scale_amax[1];
    const float s = block_scale<FMT>(amax);
    const size_t n8 = n / 8;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    auto encode8 = [&](const uint4& v, size_t i) {
        float f[8], q[8];
        unpack8(v, f);
        block_quotients<1, 8>(f, s, q);
        st_stream(codes + 8 * i, make_uint2(cvt_fp8x4<FMT>(q[0], q[1], q[2], q[3]), cvt_fp8x4<FMT>(q[4], q[5], q[6], q[7])));
    };
    size_t i = t0;
    for (; i + stride < n8; i += 2 * stride) {     // two loads in flight per thread
        const uint4 v0 = ld_stream(x + 8 * i);
        const uint4 v1 = ld_stream(x + 8 * (i + stride));
        encode8(v0, i);
        encode8(v1, i + stride);
    }
    for (; i < n8; i += stride) encode8(ld_stream(x + 8 * i), i);
    for (size_t i = 8 * n8 + t0; i < n; i += stride) {
        float f[1] = {__uint_as_float((uint32_t)x[i] << 16)}, q[1];
        block_quotients<1, 1>(f, s, q);
        codes[i] = (uint8_t)cvt_fp8x2<FMT>(q[0], 0.0f);
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
    fp8q_status_t pst = prepare_kernel(kc1, tensor_amax_kernel, 256, 0, 0, &r1);
    if (pst == FP8Q_OK) pst = prepare_kernel(kc2, tensor_encode_kernel<FMT>, 256, 0, 0, &r2);
    if (pst != FP8Q_OK) return pst;
    const size_t units = (n + 7) / 8;
    const fp8q_status_t st = launch(tensor_amax_kernel, grid_for((units + 255) / 256, r1), 256, 0, s, x, n, scale_amax);
    if (st != FP8Q_OK) return st;
    return launch(tensor_encode_kernel<FMT>, grid_for((units + 255) / 256, r2), 256, 0, s, x, n, codes, scale_amax);
}

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
