// (a) Blockwise FP8 quantize, and the plain fp32 -> FP8 element conversion.
//
// "FP8 Transmission Optimization for VLA Training", intro ("blockwise
// scaling") and "FP8 Transmission Optimization and Bottlenecks" (e4m3/e5m2):
// one fp32 scale per 128-element block, scale = amax / Fmax, codes are the
// satfinite round-to-nearest-even conversion of x / scale.
//
// Work split: tiles of 64 blocks (8192 elements, 16 KB of bf16), two
// consecutive tiles per CTA of 256 threads, on a grid that covers the array
// once (not persistent).  Thread 0 requests both tiles at once, each one bulk
// copy (cp.async.bulk) into its own shared-memory stage armed on that
// stage's mbarrier, so the loads in flight are not bounded by registers.
// Once a stage has landed, 8 lanes own one block: lane j reads elements
// [8j, 8j+8) and [64+8j, 64+8j+8) from shared memory (each 8-lane phase reads
// 128 contiguous bytes, no bank conflicts), a warp covers 4 blocks per round,
// the CTA 32 blocks per round, 2 rounds per tile.  The block amax is a 3-step
// xor-shuffle inside the 8-lane group; the quotients x / s use the per-block
// reciprocal with one Markstein correction (exact for bf16 dividends, see
// block_quotients).  The ragged last tile (n not a multiple of 8192) is read
// straight from global memory.
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kQuantThreads = 256;
constexpr int kQuantTileBlocks = 64;
constexpr int kQuantTile = kQuantTileBlocks * 128;        // elements
constexpr int kQuantStageBytes = kQuantTile * 2;
constexpr int kQuantTilesPerCta = 2;
constexpr size_t kQuantSmem = (size_t)kQuantTilesPerCta * kQuantStageBytes + 8 * kQuantTilesPerCta;

// One block's worth of work for one lane: 16 bf16 in two 8-element halves
// (va, vb) -> amax over the 8-lane group, scale, 16 codes.
template <int FMT>
__device__ __forceinline__ void quantize_block16(const uint4& va, const uint4& vb, uint32_t (&wa)[2],
                                                 uint32_t (&wb)[2], float& scale) {
    float f[16];
    unpack8(va, *reinterpret_cast<float(*)[8]>(f));
    unpack8(vb, *reinterpret_cast<float(*)[8]>(f + 8));
    float a = fabsf(f[0]);
#pragma unroll
    for (int i = 1; i < 16; ++i) a = fmaxf(a, fabsf(f[i]));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    const float s = block_scale<FMT>(a);
    float q[16];
    block_quotients<1, 16>(f, s, q);
    wa[0] = cvt_fp8x4<FMT>(q[0], q[1], q[2], q[3]);
    wa[1] = cvt_fp8x4<FMT>(q[4], q[5], q[6], q[7]);
    wb[0] = cvt_fp8x4<FMT>(q[8], q[9], q[10], q[11]);
    wb[1] = cvt_fp8x4<FMT>(q[12], q[13], q[14], q[15]);
    scale = s;
}

// Tile `lt` (kQuantTile elements from lt * kQuantTile) of one array: staged
// from shared memory `st`, or, for the array's ragged last tile, read
// straight from global memory with guarded loads and stores.
template <int FMT>
__device__ __forceinline__ void quantize_tile(const uint8_t* st, bool staged, const uint16_t* x, size_t n,
                                              uint8_t* codes, float* scales, size_t lt) {
    const unsigned tid = threadIdx.x;
    const unsigned lane = tid & 31u, warp = tid >> 5;
    const unsigned j = lane & 7u, sub = lane >> 3;
    const size_t nb = (n + 127) >> 7;
#pragma unroll
    for (int m = 0; m < kQuantTileBlocks / 32; ++m) {
        const unsigned bl = m * 32 + warp * 4 + sub;          // block inside the tile
        const size_t b = lt * kQuantTileBlocks + bl;           // block inside the array
        const size_t e0 = (b << 7) + 8 * j;
        uint4 va, vb;
        if (staged) {
            va = *reinterpret_cast<const uint4*>(st + bl * 256 + j * 16);
            vb = *reinterpret_cast<const uint4*>(st + bl * 256 + 128 + j * 16);
        } else {
            va = ld_bf16x8_tail(x + e0, (long long)n - (long long)e0);
            vb = ld_bf16x8_tail(x + e0 + 64, (long long)n - (long long)e0 - 64);
        }
        uint32_t wa[2], wb[2];
        float sc;
        quantize_block16<FMT>(va, vb, wa, wb, sc);
        if (staged) {
            st_stream(codes + e0, make_uint2(wa[0], wa[1]));
            st_stream(codes + e0 + 64, make_uint2(wb[0], wb[1]));
            if (j == 0) scales[b] = sc;
        } else if (b < nb) {
            st_u8_tail(codes + e0, wa, 2, (long long)n - (long long)e0);
            st_u8_tail(codes + e0 + 64, wb, 2, (long long)n - (long long)e0 - 64);
            if (j == 0) scales[b] = sc;
        }
    }
}

// CTA c quantizes tiles 2c and 2c + 1; both are requested at once, one
// shared-memory stage each.  The grid is not persistent: the hardware
// dispatches CTAs in index order as earlier ones retire, so the tiles in
// flight always cover one narrow, advancing address window.  (A persistent
// grid-stride loop over the same tiles let the CTAs drift apart: it ran at
// 6.2 TB/s on 10.6 GB against 7.3 TB/s for this form, and 47.1 against
// 45.1 us on 8 x 13.1M elements.)
template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
quantize_blockwise_kernel(const uint16_t* __restrict__ x, size_t n, uint8_t* __restrict__ codes,
                          float* __restrict__ scales, int inputs_ready) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuantTilesPerCta * kQuantStageBytes);
    const size_t ntiles = (n + kQuantTile - 1) / kQuantTile;
    const size_t nstaged = n / kQuantTile;                // tiles entirely inside the array
    const size_t t0 = (size_t)blockIdx.x * kQuantTilesPerCta;
    const unsigned tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < kQuantTilesPerCta; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto request = [&]() {                        // thread 0 only: both tiles
        for (int s = 0; s < kQuantTilesPerCta; ++s) {
            const size_t t = t0 + s;
            if (t < nstaged) {
                mbar_arrive_expect_tx(&full[s], kQuantStageBytes);
                bulk_g2s(smem + (size_t)s * kQuantStageBytes, x + t * kQuantTile, kQuantStageBytes, &full[s]);
            }
        }
    };
    // with inputs_ready the caller guarantees that no kernel still running
    // writes x: the tiles are requested before the grid-dependency wait
    if (tid == 0 && inputs_ready) request();
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && !inputs_ready) request();

    int s = 0;
    bool failed = false;
    for (; s < kQuantTilesPerCta; ++s) {
        const size_t t = t0 + s;
        if (t >= ntiles) break;
        const bool staged = t < nstaged;
        const bool ok = staged ? mbar_wait(&full[s], 0u) : true;
        quantize_tile<FMT>(smem + (size_t)s * kQuantStageBytes, staged, x, n, codes, scales, t);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
    }
    if (failed && tid == 0) {
        // report, and let the copies still in flight land before the CTA's
        // shared memory is released
        raise_error(kErrCopyTimeout);
        for (int r = s; r < kQuantTilesPerCta; ++r)
            if (t0 + r < nstaged) mbar_wait(&full[r], 0u);
    }
}

// Up to kQuantMaxGroup independent blockwise quantizations in one launch
// (for instance every rank's chunk of a simulated ring, or several gradient
// buckets).  Item i owns the global tiles [tile_start[i], tile_start[i + 1]).
constexpr int kQuantMaxGroup = FP8Q_MAX_QUANT_GROUP;

struct QuantGroup {
    const uint16_t* x[kQuantMaxGroup];
    uint8_t* codes[kQuantMaxGroup];
    float* scales[kQuantMaxGroup];
    size_t n[kQuantMaxGroup];
    int64_t tile_start[kQuantMaxGroup + 1];
    int count;
    int inputs_ready;
};

// The work split of quantize_blockwise_kernel over the tiles of all items:
// CTA c takes global tiles 2c and 2c + 1, which may belong to different
// items.  An item's ragged last tile is read from global memory.
template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
quantize_group_kernel(const __grid_constant__ QuantGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuantTilesPerCta * kQuantStageBytes);
    const int64_t total_tiles = g.tile_start[g.count];
    const int64_t t0 = (int64_t)blockIdx.x * kQuantTilesPerCta;
    const unsigned tid = threadIdx.x;

    // item of each of the CTA's tiles (CTA-uniform)
    int item[kQuantTilesPerCta];
    {
        int i = 0;
#pragma unroll
        for (int s = 0; s < kQuantTilesPerCta; ++s) {
            while (i + 1 < g.count && t0 + s >= g.tile_start[i + 1]) ++i;
            item[s] = i;
        }
    }
    // a tile is staged when it lies entirely inside its item's array
    auto staged_tile = [&](int s) {
        const int64_t t = t0 + s;
        return t < total_tiles && (size_t)(t - g.tile_start[item[s]] + 1) * kQuantTile <= g.n[item[s]];
    };
    if (tid == 0) {
        for (int s = 0; s < kQuantTilesPerCta; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto request = [&]() {                        // thread 0 only: both tiles
#pragma unroll
        for (int s = 0; s < kQuantTilesPerCta; ++s) {
            if (!staged_tile(s)) continue;
            const size_t lt = (size_t)(t0 + s - g.tile_start[item[s]]);
            mbar_arrive_expect_tx(&full[s], kQuantStageBytes);
            bulk_g2s(smem + (size_t)s * kQuantStageBytes, g.x[item[s]] + lt * kQuantTile, kQuantStageBytes,
                     &full[s]);
        }
    };
    if (tid == 0 && g.inputs_ready) request();
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && !g.inputs_ready) request();

    int s = 0;
    bool failed = false;
#pragma unroll
    for (; s < kQuantTilesPerCta; ++s) {
        const int64_t t = t0 + s;
        if (t >= total_tiles) break;
        const int i = item[s];
        const bool staged = staged_tile(s);
        const bool ok = staged ? mbar_wait(&full[s], 0u) : true;
        quantize_tile<FMT>(smem + (size_t)s * kQuantStageBytes, staged, g.x[i], g.n[i], g.codes[i], g.scales[i],
                           (size_t)(t - g.tile_start[i]));
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
    }
    if (failed && tid == 0) {
        raise_error(kErrCopyTimeout);
#pragma unroll
        for (int r = 0; r < kQuantTilesPerCta; ++r)
            if (r >= s && staged_tile(r)) mbar_wait(&full[r], 0u);
    }
}

// Elementwise conversion: 4 floats per lane per step.
template <int FMT>
__global__ void __launch_bounds__(256)
encode_f32_kernel(const float* __restrict__ x, size_t n, uint8_t* __restrict__ codes) {
    dependency_wait();
    allow_dependents();
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
                                     cudaStream_t stream, int inputs_ready) {
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, quantize_blockwise_kernel<FMT>, kQuantThreads, kQuantSmem,
                                            kQuantSmem, &resident);
    if (st != FP8Q_OK) return st;
    const size_t tiles = (n + kQuantTile - 1) / kQuantTile;
    const size_t grid = (tiles + kQuantTilesPerCta - 1) / kQuantTilesPerCta;
    return launch(quantize_blockwise_kernel<FMT>, (unsigned)grid, kQuantThreads, kQuantSmem, stream, x, n, codes,
                  scales, inputs_ready);
}

template <int FMT>
static fp8q_status_t launch_encode(const float* x, size_t n, uint8_t* codes, cudaStream_t stream) {
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, encode_f32_kernel<FMT>, 256, 0, 0, &resident);
    if (st != FP8Q_OK) return st;
    const size_t units = (n + 3) / 4;
    const unsigned grid = grid_for((units + 255) / 256, resident * 2);
    return launch(encode_f32_kernel<FMT>, grid, 256, 0, stream, x, n, codes);
}

// Byte ranges of a group item: input 0, outputs 1..2.
static void item_ranges(const fp8q_quant_t& q, const void* p[3], size_t sz[3]) {
    p[0] = q.x_bf16;  sz[0] = 2 * q.n;
    p[1] = q.codes;   sz[1] = q.n;
    p[2] = q.scales;  sz[2] = 4 * fp8q_num_scales(q.n);
}

template <int FMT>
static fp8q_status_t launch_quantize_group(const QuantGroup& g, size_t tiles, cudaStream_t stream) {
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, quantize_group_kernel<FMT>, kQuantThreads, kQuantSmem, kQuantSmem,
                                            &resident);
    if (st != FP8Q_OK) return st;
    const size_t grid = (tiles + kQuantTilesPerCta - 1) / kQuantTilesPerCta;
    if (grid > 0x7FFFFFFFu) return FP8Q_ERR_SIZE;        // beyond the grid limit (about 2^44 elements)
    return launch(quantize_group_kernel<FMT>, (unsigned)grid, kQuantThreads, kQuantSmem, stream, g);
}

}  // namespace fp8q

namespace fp8q {
unsigned unit_errors_quantize(bool clear) { return read_unit_errors(clear); }
}  // namespace fp8q

using namespace fp8q;

static fp8q_status_t quantize_entry(const void* x_bf16, size_t n, fp8q_format_t fmt, uint8_t* codes, float* scales,
                                    unsigned flags, fp8q_stream_t stream) {
    if (flags & ~FP8Q_INPUTS_READY) return FP8Q_ERR_FLAGS;
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
    const int ready = (flags & FP8Q_INPUTS_READY) ? 1 : 0;
    return fmt == FP8Q_E4M3 ? launch_quantize<kE4M3>(x, n, codes, scales, s, ready)
                            : launch_quantize<kE5M2>(x, n, codes, scales, s, ready);
}

extern "C" fp8q_status_t fp8q_quantize_blockwise(const void* x_bf16, size_t n, fp8q_format_t fmt,
                                                 uint8_t* codes, float* scales, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_quantize_blockwise");
    return quantize_entry(x_bf16, n, fmt, codes, scales, 0, stream);
}

extern "C" fp8q_status_t fp8q_quantize_blockwise_ex(const void* x_bf16, size_t n, fp8q_format_t fmt,
                                                    uint8_t* codes, float* scales, unsigned int flags,
                                                    fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_quantize_blockwise_ex");
    return quantize_entry(x_bf16, n, fmt, codes, scales, flags, stream);
}

extern "C" fp8q_status_t fp8q_encode_f32(const float* x, size_t n, fp8q_format_t fmt, uint8_t* codes,
                                         fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_encode_f32");
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!x || !codes) return FP8Q_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes)) return FP8Q_ERR_ALIGN;
    if (overlaps(codes, n, x, 4 * n)) return FP8Q_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3 ? launch_encode<kE4M3>(x, n, codes, s) : launch_encode<kE5M2>(x, n, codes, s);
}

extern "C" fp8q_status_t fp8q_quantize_blockwise_group(const fp8q_quant_t* items, int count, fp8q_format_t fmt,
                                                       unsigned int flags, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_quantize_blockwise_group");
    if (flags & ~FP8Q_INPUTS_READY) return FP8Q_ERR_FLAGS;
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (!items) return FP8Q_ERR_NULL;
    if (count < 1 || count > kQuantMaxGroup) return FP8Q_ERR_SIZE;
    for (int i = 0; i < count; ++i) {                  // each item as fp8q_quantize_blockwise checks it
        const fp8q_quant_t& q = items[i];
        if (q.n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
        if (q.n == 0) continue;
        if (!q.x_bf16 || !q.codes || !q.scales) return FP8Q_ERR_NULL;
        if (!aligned16(q.x_bf16) || !aligned16(q.codes) || !aligned16(q.scales)) return FP8Q_ERR_ALIGN;
    }
    // no output overlaps any input or output of the group
    for (int i = 0; i < count; ++i) {
        if (items[i].n == 0) continue;
        const void* pi[3];
        size_t si[3];
        item_ranges(items[i], pi, si);
        for (int j = 0; j < count; ++j) {
            if (items[j].n == 0) continue;
            const void* pj[3];
            size_t sj[3];
            item_ranges(items[j], pj, sj);
            for (int a = 1; a < 3; ++a)
                for (int b = 0; b < 3; ++b) {
                    if (i == j && a == b) continue;
                    if (overlaps(pi[a], si[a], pj[b], sj[b])) return FP8Q_ERR_ALIAS;
                }
        }
    }
    QuantGroup g;
    int used = 0;
    int64_t start = 0;
    for (int i = 0; i < count; ++i) {
        const fp8q_quant_t& q = items[i];
        if (q.n == 0) continue;
        g.x[used] = static_cast<const uint16_t*>(q.x_bf16);
        g.codes[used] = q.codes;
        g.scales[used] = q.scales;
        g.n[used] = q.n;
        g.tile_start[used] = start;
        start += (int64_t)((q.n + kQuantTile - 1) / kQuantTile);
        ++used;
    }
    if (used == 0) return FP8Q_OK;
    g.tile_start[used] = start;
    g.count = used;
    g.inputs_ready = (flags & FP8Q_INPUTS_READY) ? 1 : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return fmt == FP8Q_E4M3 ? launch_quantize_group<kE4M3>(g, (size_t)start, s)
                            : launch_quantize_group<kE5M2>(g, (size_t)start, s);
}
