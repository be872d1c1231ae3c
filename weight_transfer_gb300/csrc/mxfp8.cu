// (d) BF16 -> MXFP8 weight prequantization with the 128x4-tiled E8M0 scale
// layout.
//
// "perf: Reduce MXFP8 refit weight-transfer overheads", Summary (eligible
// trainer weights are quantized before the transfer and reuse MXFP8 shuffle
// buffers), self-review (E8M0 zero-scale clamp; 2D and 3D expert tensors)
// and inline review (a K/32 scale dimension of 1 is real).  Block rule from
// the OCP MX v1.0 specification: e = floor(log2 amax) - 8 + 127 for E4M3.
//
// Work split: a CTA owns one 128-row x 128-column tile of one matrix, which
// is exactly one 512-byte tile of the swizzled scale buffer (128 rows x 4
// scale columns).  Each warp covers 16 rows, two rows per 16-byte load
// instruction (16 lanes x 8 bf16 = 128 columns); 4 lanes share a 32-element
// block and reduce its amax with two xor-shuffles.  The 512 scale bytes are
// placed at their swizzled positions in shared memory and leave the CTA as
// one contiguous 512-byte store; codes are written row-major.
//
// The exponent needs no floating-point log: for a finite amax >= 0 with
// biased binary32 exponent E, floor(log2 amax) - 8 + 127 = E - 8 when amax
// is normal, and every subnormal or zero amax clamps to 0 -- so
// e = max(E - 8, 0).  The scaling by 2^(127 - e) is exact (a power of two in
// the normal range, 2^-119 .. 2^127).
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kMxThreads = 256;
constexpr int kMxRowsPerWarp = 16;

__global__ void __launch_bounds__(kMxThreads)
mxfp8_quantize_kernel(const uint16_t* __restrict__ w, int64_t m, int64_t k, int64_t row_tiles,
                      int64_t col_tiles, int64_t total_tiles, uint8_t* __restrict__ codes,
                      uint8_t* __restrict__ scales) {
    __shared__ __align__(16) uint8_t sbuf[2][512];
    const unsigned lane = threadIdx.x & 31u;
    const unsigned warp = threadIdx.x >> 5;
    const unsigned c = lane & 15u;                 // 8-column chunk inside the tile
    const unsigned jl = c >> 2;                    // scale column inside the tile
    const int64_t tiles_per_mat = row_tiles * col_tiles;
    int buf = 0;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, buf ^= 1) {
        const int64_t bt = t / tiles_per_mat;
        const int64_t rem = t - bt * tiles_per_mat;
        const int64_t rt = rem / col_tiles;
        const int64_t ct = rem - rt * col_tiles;
        const int64_t col = ct * 128 + c * 8;
        const bool col_ok = col < k;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = rt * 128 + warp * kMxRowsPerWarp + 2 * i + (lane >> 4);
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            if (col_ok && row < m) v[i] = ld_stream(w + ((bt * m + row) * k + col));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rl = warp * kMxRowsPerWarp + 2 * i + (lane >> 4);    // row inside the tile
            const int64_t row = rt * 128 + rl;
            float f[8];
            unpack8(v[i], f);
            float a = fabsf(f[0]);
#pragma unroll
            for (int e = 1; e < 8; ++e) a = fmaxf(a, fabsf(f[e]));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
            const int E = (int)(__float_as_uint(a) >> 23);           // a >= 0: no sign bit
            const int e8 = E > 8 ? E - 8 : 0;                          // E8M0 byte
            const float factor = __uint_as_float((uint32_t)(254 - e8) << 23);   // 2^(127 - e8)
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = __fmul_rn(f[e], factor);
            if (col_ok && row < m)
                st_stream(codes + ((bt * m + row) * k + col),
                          make_uint2(cvt_fp8x4<kE4M3>(q[0], q[1], q[2], q[3]), cvt_fp8x4<kE4M3>(q[4], q[5], q[6], q[7])));
            if ((c & 3u) == 0)   // padded rows / columns keep e8 == 0
                sbuf[buf][(rl & 31) * 16 + (rl >> 5) * 4 + jl] = (uint8_t)e8;
        }
        __syncthreads();
        if (threadIdx.x < 32)
            st_stream(scales + t * 512 + threadIdx.x * 16, *reinterpret_cast<const uint4*>(&sbuf[buf][threadIdx.x * 16]));
    }
}

}  // namespace fp8q

using namespace fp8q;

extern "C" size_t mxfp8_swizzled_scale_bytes(int64_t batch, int64_t m, int64_t k) {
    if (batch < 0 || m < 0 || k <= 0 || k % MXFP8_BLOCK != 0) return 0;
    const int64_t kb = k / MXFP8_BLOCK;
    return (size_t)batch * (size_t)((m + 127) / 128) * (size_t)((kb + 3) / 4) * 512u;
}

extern "C" fp8q_status_t mxfp8_quantize_swizzled(const void* w_bf16, int64_t batch, int64_t m, int64_t k,
                                                 uint8_t* codes, uint8_t* scales_swizzled, fp8q_stream_t stream) {
    if (batch < 0 || m < 0) return FP8Q_ERR_SIZE;
    if (k <= 0 || k % MXFP8_BLOCK != 0) return FP8Q_ERR_K;
    if (m > 0 && batch > 0 && (uint64_t)k > FP8Q_MAX_ELEMENTS / (uint64_t)m / (uint64_t)batch) return FP8Q_ERR_SIZE;
    const size_t n = (size_t)batch * (size_t)m * (size_t)k;
    if (n == 0) return FP8Q_OK;
    if (!w_bf16 || !codes || !scales_swizzled) return FP8Q_ERR_NULL;
    if (!aligned16(w_bf16) || !aligned16(codes) || !aligned16(scales_swizzled)) return FP8Q_ERR_ALIGN;
    const size_t sbytes = mxfp8_swizzled_scale_bytes(batch, m, k);
    if (overlaps(codes, n, w_bf16, 2 * n) || overlaps(scales_swizzled, sbytes, w_bf16, 2 * n) ||
        overlaps(codes, n, scales_swizzled, sbytes))
        return FP8Q_ERR_ALIAS;
    static int resident = resident_blocks(mxfp8_quantize_kernel, kMxThreads);
    const int64_t row_tiles = (m + 127) / 128;
    const int64_t col_tiles = (k / MXFP8_BLOCK + 3) / 4;
    const int64_t total = batch * row_tiles * col_tiles;
    const unsigned grid = grid_for((size_t)total, resident);
    mxfp8_quantize_kernel<<<grid, kMxThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(w_bf16), m, k, row_tiles, col_tiles, total, codes, scales_swizzled);
    return launch_status();
}
