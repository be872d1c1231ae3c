// (a) Blockwise FP8 quantize, and the plain fp32 -> FP8 element conversion.
//
// "FP8 Transmission Optimization for VLA Training", intro ("blockwise
// scaling") and "FP8 Transmission Optimization and Bottlenecks" (e4m3/e5m2):
// one fp32 scale per 128-element block, scale = amax / Fmax, codes are the
// satfinite round-to-nearest-even conversion of x / scale.
//
// Work split: a persistent CTA of 256 threads walks tiles of 64 blocks
// (8192 elements, 16 KB of bf16).  Thread 0 keeps up to kQuantStages tiles
// in flight, each one bulk copy (cp.async.bulk) into a shared-memory stage
// armed on that stage's mbarrier, so the loads in flight are not bounded by
// registers.  Once a stage has landed, 8 lanes own one block: lane j reads
// elements [8j, 8j+8) and [64+8j, 64+8j+8) from shared memory (each 8-lane
// phase reads 128 contiguous bytes, no bank conflicts), a warp covers 4
// blocks per round, the CTA 32 blocks per round, 2 rounds per tile.  The
// block amax is a 3-step xor-shuffle inside the 8-lane group; the quotients
// x / s use the per-block reciprocal with one Markstein correction (exact for
// bf16 dividends, see block_quotients).  The ragged last tile (n not a
// multiple of 8192) is read straight from global memory.
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kQuantThreads = 256;
constexpr int kQuantTileBlocks = 64;
constexpr int kQuantTile = kQuantTileBlocks * 128;        // elements
constexpr int kQuantStageBytes = kQuantTile * 2;
constexpr int kQuantStages = 3;
constexpr size_t kQuantSmem = (size_t)kQuantStages * kQuantStageBytes + 8 * kQuantStages;

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

template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
quantize_blockwise_kernel(const uint16_t* __restrict__ x, size_t n, uint8_t* __restrict__ codes,
                          float* __restrict__ scales, int inputs_ready) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuantStages * kQuantStageBytes);
    const size_t nb = (n + 127) >> 7;
    const size_t ntiles = (n + kQuantTile - 1) / kQuantTile;
    const size_t nstaged = n / kQuantTile;                // tiles entirely inside the array
    const unsigned tid = threadIdx.x;
    const unsigned lane = tid & 31u, warp = tid >> 5;
    const unsigned j = lane & 7u, sub = lane >> 3;

    if (tid == 0) {
        for (int s = 0; s < kQuantStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto issue = [&](size_t t, int s) {           // thread 0 only
        mbar_arrive_expect_tx(&full[s], kQuantStageBytes);
        bulk_g2s(smem + (size_t)s * kQuantStageBytes, x + t * kQuantTile, kQuantStageBytes, &full[s]);
    };
    auto prologue = [&]() {                       // thread 0 only: the first tiles
        for (int s = 0; s < kQuantStages; ++s) {
            const size_t t = blockIdx.x + (size_t)s * gridDim.x;
            if (t < nstaged) issue(t, s);
        }
    };
    // with inputs_ready the caller guarantees that no kernel still running
    // writes x: the first tiles are requested before the grid-dependency wait
    if (tid == 0 && inputs_ready) prologue();
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && !inputs_ready) prologue();

    int it = 0;
    bool failed = false;
    for (size_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = it % kQuantStages;
        const bool staged = t < nstaged;
        const bool ok = staged ? mbar_wait(&full[s], (uint32_t)(it / kQuantStages) & 1u) : true;
        const uint8_t* st = smem + (size_t)s * kQuantStageBytes;
#pragma unroll
        for (int m = 0; m < kQuantTileBlocks / 32; ++m) {
            const unsigned bl = m * 32 + warp * 4 + sub;          // block inside the tile
            const size_t b = t * kQuantTileBlocks + bl;            // block inside the array
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
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            const size_t tn = t + (size_t)kQuantStages * gridDim.x;
            if (tn < nstaged) {
                fence_proxy_async_smem();
                issue(tn, s);
            }
        }
    }
    if (failed && tid == 0) {
        raise_error(kErrCopyTimeout);
        for (int jj = it; jj < it + kQuantStages; ++jj) {
            const size_t tj = blockIdx.x + (size_t)jj * gridDim.x;
            if (tj < nstaged) mbar_wait(&full[jj % kQuantStages], (uint32_t)(jj / kQuantStages) & 1u);
        }
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

// The work split of quantize_blockwise_kernel over the tiles of all items.
// An item's ragged last tile is not staged and can sit between staged tiles,
// so each stage's barrier parity is tracked explicitly: bit s of `parity` is
// the phase to wait for on stage s, flipped each time a staged tile of that
// stage has been consumed; `pending` (thread 0) marks stages with a copy
// issued and not yet consumed.
template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
quantize_group_kernel(const __grid_constant__ QuantGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuantStages * kQuantStageBytes);
    const int64_t total_tiles = g.tile_start[g.count];
    const unsigned tid = threadIdx.x;
    const unsigned lane = tid & 31u, warp = tid >> 5;
    const unsigned j = lane & 7u, sub = lane >> 3;

    auto item_of = [&](int64_t t) {                        // CTA-uniform
        int i = 0;
        while (i + 1 < g.count && t >= g.tile_start[i + 1]) ++i;
        return i;
    };
    // a tile is staged when it lies entirely inside its item's array
    auto staged_tile = [&](int64_t t, int i) { return (size_t)(t - g.tile_start[i] + 1) * kQuantTile <= g.n[i]; };
    if (tid == 0) {
        for (int s = 0; s < kQuantStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto issue = [&](int64_t t, int i, int s) {   // thread 0 only
        const size_t lt = (size_t)(t - g.tile_start[i]);
        mbar_arrive_expect_tx(&full[s], kQuantStageBytes);
        bulk_g2s(smem + (size_t)s * kQuantStageBytes, g.x[i] + lt * kQuantTile, kQuantStageBytes, &full[s]);
    };
    uint32_t parity = 0;
    uint32_t pending = 0;
    auto prologue = [&]() {                       // thread 0 only: the first tiles
        for (int s = 0; s < kQuantStages; ++s) {
            const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
            if (t < total_tiles) {
                const int i = item_of(t);
                if (staged_tile(t, i)) {
                    issue(t, i, s);
                    pending |= 1u << s;
                }
            }
        }
    };
    if (tid == 0 && g.inputs_ready) prologue();
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && !g.inputs_ready) prologue();

    int it = 0;
    bool failed = false;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
        const int s = it % kQuantStages;
        const int i = item_of(t);
        const size_t n = g.n[i];
        const size_t nb = (n + 127) >> 7;
        const bool staged = staged_tile(t, i);
        const bool ok = staged ? mbar_wait(&full[s], (parity >> s) & 1u) : true;
        if (staged && ok) {
            parity ^= 1u << s;
            pending &= ~(1u << s);
        }
        const uint8_t* st = smem + (size_t)s * kQuantStageBytes;
        const uint16_t* x = g.x[i];
        uint8_t* codes = g.codes[i];
        float* scales = g.scales[i];
        const size_t lt = (size_t)(t - g.tile_start[i]);
#pragma unroll
        for (int m = 0; m < kQuantTileBlocks / 32; ++m) {
            const unsigned bl = m * 32 + warp * 4 + sub;          // block inside the tile
            const size_t b = lt * kQuantTileBlocks + bl;           // block inside the item
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
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            const int64_t tn = t + (int64_t)kQuantStages * gridDim.x;     // next tile of stage s
            if (tn < total_tiles) {
                const int in = item_of(tn);
                if (staged_tile(tn, in)) {
                    fence_proxy_async_smem();
                    issue(tn, in, s);
                    pending |= 1u << s;
                }
            }
        }
    }
    if (failed && tid == 0) {
        // report, and let the copies still in flight land before the CTA's
        // shared memory is released
        raise_error(kErrCopyTimeout);
        for (int s = 0; s < kQuantStages; ++s)
            if (pending & (1u << s)) mbar_wait(&full[s], (parity >> s) & 1u);
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
    const unsigned grid = grid_for(tiles, resident);
    return launch(quantize_blockwise_kernel<FMT>, grid, kQuantThreads, kQuantSmem, stream, x, n, codes, scales,
                  inputs_ready);
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
    return launch(quantize_group_kernel<FMT>, grid_for(tiles, resident), kQuantThreads, kQuantSmem, stream, g);
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
    return quantize_entry(x_bf16, n, fmt, codes, scales, 0, stream);
}

extern "C" fp8q_status_t fp8q_quantize_blockwise_ex(const void* x_bf16, size_t n, fp8q_format_t fmt,
                                                    uint8_t* codes, float* scales, unsigned int flags,
                                                    fp8q_stream_t stream) {
    return quantize_entry(x_bf16, n, fmt, codes, scales, flags, stream);
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

extern "C" fp8q_status_t fp8q_quantize_blockwise_group(const fp8q_quant_t* items, int count, fp8q_format_t fmt,
                                                       unsigned int flags, fp8q_stream_t stream) {
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
