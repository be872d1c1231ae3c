// The receiving side of a prequantized MXFP8 transfer.
//
// "perf: Reduce MXFP8 refit weight-transfer overheads": the receiver loads
// the E4M3 weights with their *_scale_from_checkpoint (Safety), rearranges
// scales for its GEMMs (the "MXFP8 shuffle", whose result is checked
// bit-exactly by NRL_MXFP8_SHUFFLE_VERIFY in the 30B / 235B reproductions)
// and, in the review of the sm100 fast path, expects scales shaped
// [M, K/32].  Three small kernels serve that side:
//   mxfp8_dequantize_swizzled  w = RNE_bf16(decode_e4m3(c) * 2^(e - 127))
//   mxfp8_unswizzle_scales     swizzled E8M0 bytes -> row-major [batch, m, k/32]
//   fp8q_count_mismatches      number of differing bytes of two buffers
// None of them is on the sender's hot path.  The dequantize walks whole
// 128 x 128 tiles, whose scales are one contiguous 512-byte tile; the other
// two are grid-stride kernels.
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

__device__ __forceinline__ int64_t swizzle_offset(int64_t bt, int64_t r, int64_t j, int64_t m, int64_t kb) {
    const int64_t col_tiles = (kb + 3) / 4, row_tiles = (m + 127) / 128;
    return bt * row_tiles * col_tiles * 512 + ((r / 128) * col_tiles + j / 4) * 512 + (r % 32) * 16 +
           ((r % 128) / 32) * 4 + (j % 4);
}

// Dequantize by whole 128 x 128 tiles of the [batch * m, k] code matrix: the
// tiles of the swizzled scale layout, so tile t's 512 E8M0 bytes are the
// contiguous bytes [512 t, 512 t + 512) of the scale buffer.  256 threads
// per tile: 8 per row, 32 rows per pass, 4 passes.  Thread c of a row takes
// codes [8c, 8c + 8) and [64 + 8c, 64 + 8c + 8) (two 8-byte loads, two
// 16-byte bf16 stores), so that each store instruction of a warp writes
// whole 128-byte runs; with 16 consecutive codes per thread a store covered
// only half of each 32-byte sector it touched.  The tile index is split into
// (matrix, row tile, column tile) once per tile, in 32-bit arithmetic (the
// entry point rejects tensors of 2^32 tiles or more).
__global__ void __launch_bounds__(256)
mxfp8_dequantize_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int64_t m,
                        int64_t k, uint32_t total_tiles, uint32_t tiles_per_mat, uint32_t col_tiles,
                        uint16_t* __restrict__ out) {
    dependency_wait();
    allow_dependents();
    const unsigned tid = threadIdx.x;
    const unsigned chunk = tid & 7u;               // codes [8 chunk, +8) and [64 + 8 chunk, +8) of the tile row
    const unsigned rsub = tid >> 3;                // row inside a 32-row pass
    const unsigned j = chunk >> 2;                 // scale column of the first 8 codes; the second's is j + 2
    for (uint32_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        const uint32_t bt = t / tiles_per_mat;
        const uint32_t rem = t - bt * tiles_per_mat;
        const uint32_t rt = rem / col_tiles;
        const uint32_t ct = rem - rt * col_tiles;
        const int64_t col = (int64_t)ct * 128 + chunk * 8;
        if (col >= k) continue;                    // k % 32 == 0: both 8-code runs are in, or the first only, or none
        const bool second = col + 64 < k;
        const uint8_t* stile = scales + (size_t)t * 512;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const unsigned r = p * 32 + rsub;      // row inside the tile
            const int64_t row = (int64_t)rt * 128 + r;
            if (row >= m) break;                   // later passes are further down
            const size_t e0 = (size_t)((int64_t)bt * m + row) * (size_t)k + (size_t)col;
            const unsigned sb = (r & 31u) * 16 + (r >> 5) * 4;
            const uint32_t e8a = __ldg(stile + sb + j);
            const uint32_t e8b = second ? __ldg(stile + sb + j + 2) : 0u;
            // 2^(e8 - 127): a normal binary32 for e8 >= 1, the subnormal 2^-127 for e8 == 0
            const float fa = __uint_as_float(e8a ? (e8a << 23) : 0x00400000u);
            const float fb = __uint_as_float(e8b ? (e8b << 23) : 0x00400000u);
            const uint2 ca = ld_stream8(codes + e0);
            const uint2 cb = second ? ld_stream8(codes + e0 + 64) : make_uint2(0u, 0u);
            float d[16];
            decode_fp8x4<kE4M3>(ca.x, d);
            decode_fp8x4<kE4M3>(ca.y, d + 4);
            decode_fp8x4<kE4M3>(cb.x, d + 8);
            decode_fp8x4<kE4M3>(cb.y, d + 12);
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {   // the products are exact; only the bf16 rounding rounds
                h[i] = pack_bf16x2(__fmul_rn(d[2 * i], fa), __fmul_rn(d[2 * i + 1], fa));
                h[4 + i] = pack_bf16x2(__fmul_rn(d[8 + 2 * i], fb), __fmul_rn(d[8 + 2 * i + 1], fb));
            }
            st_stream(out + e0, make_uint4(h[0], h[1], h[2], h[3]));
            if (second) st_stream(out + e0 + 64, make_uint4(h[4], h[5], h[6], h[7]));
        }
    }
}

__global__ void __launch_bounds__(256)
mxfp8_unswizzle_kernel(const uint8_t* __restrict__ scales, int64_t m, int64_t kb, size_t total,
                       uint8_t* __restrict__ out) {
    dependency_wait();
    allow_dependents();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int64_t j = (int64_t)(i % (size_t)kb);
        const int64_t row = (int64_t)(i / (size_t)kb);
        const int64_t bt = row / m, r = row - bt * m;
        out[i] = scales[swizzle_offset(bt, r, j, m, kb)];
    }
}

// Adds the number of differing bytes of a and b to *count.
__global__ void __launch_bounds__(256)
count_mismatches_kernel(const uint8_t* __restrict__ a, const uint8_t* __restrict__ b, size_t n,
                        unsigned long long* count) {
    dependency_wait();
    allow_dependents();
    unsigned long long mine = 0;
    const size_t n16 = n / 16;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (size_t i = t0; i < n16; i += stride) {
        const uint4 x = ld_stream(a + 16 * i), y = ld_stream(b + 16 * i);
        // __vcmpne4: 0xFF in every byte lane that differs
        mine += __popc(__vcmpne4(x.x, y.x)) / 8 + __popc(__vcmpne4(x.y, y.y)) / 8 +
                __popc(__vcmpne4(x.z, y.z)) / 8 + __popc(__vcmpne4(x.w, y.w)) / 8;
    }
    for (size_t i = 16 * n16 + t0; i < n; i += stride) mine += a[i] != b[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xFFFFFFFFu, mine, o);
    if ((threadIdx.x & 31u) == 0 && mine) atomicAdd(count, mine);
}

static fp8q_status_t check_mx_shape(int64_t batch, int64_t m, int64_t k) {
    if (batch < 0 || m < 0) return FP8Q_ERR_SIZE;
    if (k <= 0 || k % MXFP8_BLOCK != 0) return FP8Q_ERR_K;
    if (m > 0 && batch > 0 && (uint64_t)k > FP8Q_MAX_ELEMENTS / (uint64_t)m / (uint64_t)batch) return FP8Q_ERR_SIZE;
    return FP8Q_OK;
}

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status_t mxfp8_dequantize_swizzled(const uint8_t* codes, const uint8_t* scales_swizzled, int64_t batch,
                                                   int64_t m, int64_t k, void* out_bf16, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("mxfp8_dequantize_swizzled");
    fp8q_status_t st = check_mx_shape(batch, m, k);
    if (st != FP8Q_OK) return st;
    const size_t n = (size_t)batch * (size_t)m * (size_t)k;
    if (n == 0) return FP8Q_OK;
    if (!codes || !scales_swizzled || !out_bf16) return FP8Q_ERR_NULL;
    if (!aligned16(codes) || !aligned16(scales_swizzled) || !aligned16(out_bf16)) return FP8Q_ERR_ALIGN;
    const size_t sb = mxfp8_swizzled_scale_bytes(batch, m, k);
    if (overlaps(out_bf16, 2 * n, codes, n) || overlaps(out_bf16, 2 * n, scales_swizzled, sb)) return FP8Q_ERR_ALIAS;
    const int64_t row_tiles = (m + 127) / 128, col_tiles = (k / MXFP8_BLOCK + 3) / 4;
    const uint64_t tiles = (uint64_t)batch * (uint64_t)row_tiles * (uint64_t)col_tiles;
    if (tiles > 0xFFFFFFFFull) return FP8Q_ERR_SIZE;       // the kernel indexes tiles in 32 bits
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t pst = prepare_kernel(kc, mxfp8_dequantize_kernel, 256, 0, 0, &resident);
    if (pst != FP8Q_OK) return pst;
    return launch(mxfp8_dequantize_kernel, grid_for((size_t)tiles, resident), 256, 0,
                  reinterpret_cast<cudaStream_t>(stream), codes, scales_swizzled, m, k, (uint32_t)tiles,
                  (uint32_t)(row_tiles * col_tiles), (uint32_t)col_tiles, static_cast<uint16_t*>(out_bf16));
}

extern "C" fp8q_status_t mxfp8_unswizzle_scales(const uint8_t* scales_swizzled, int64_t batch, int64_t m, int64_t k,
                                                uint8_t* scales_rowmajor, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("mxfp8_unswizzle_scales");
    fp8q_status_t st = check_mx_shape(batch, m, k);
    if (st != FP8Q_OK) return st;
    const size_t total = (size_t)batch * (size_t)m * (size_t)(k / MXFP8_BLOCK);
    if (total == 0) return FP8Q_OK;
    if (!scales_swizzled || !scales_rowmajor) return FP8Q_ERR_NULL;
    if (!aligned16(scales_swizzled) || !aligned16(scales_rowmajor)) return FP8Q_ERR_ALIGN;
    if (overlaps(scales_rowmajor, total, scales_swizzled, mxfp8_swizzled_scale_bytes(batch, m, k)))
        return FP8Q_ERR_ALIAS;
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t pst = prepare_kernel(kc, mxfp8_unswizzle_kernel, 256, 0, 0, &resident);
    if (pst != FP8Q_OK) return pst;
    return launch(mxfp8_unswizzle_kernel, grid_for((total + 255) / 256, resident), 256, 0,
                  reinterpret_cast<cudaStream_t>(stream), scales_swizzled, m, (int64_t)(k / MXFP8_BLOCK), total,
                  scales_rowmajor);
}

extern "C" fp8q_status_t fp8q_count_mismatches(const void* a, const void* b, size_t nbytes, unsigned long long* count,
                                               fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_count_mismatches");
    if (nbytes > 16 * FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (nbytes == 0) return FP8Q_OK;
    if (!a || !b || !count) return FP8Q_ERR_NULL;
    if (!aligned16(a) || !aligned16(b) || (reinterpret_cast<uintptr_t>(count) & 7u)) return FP8Q_ERR_ALIGN;
    if (overlaps(count, 8, a, nbytes) || overlaps(count, 8, b, nbytes)) return FP8Q_ERR_ALIAS;
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t pst = prepare_kernel(kc, count_mismatches_kernel, 256, 0, 0, &resident);
    if (pst != FP8Q_OK) return pst;
    return launch(count_mismatches_kernel, grid_for((nbytes / 16 + 255) / 256 + 1, resident), 256, 0,
                  reinterpret_cast<cudaStream_t>(stream), static_cast<const uint8_t*>(a),
                  static_cast<const uint8_t*>(b), nbytes, count);
}
