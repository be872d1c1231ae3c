// (d) BF16 -> MXFP8 weight prequantization with the 128x4-tiled E8M0 scale
// layout.
//
// "perf: Reduce MXFP8 refit weight-transfer overheads", Summary (eligible
// trainer weights are quantized before the transfer and reuse MXFP8 shuffle
// buffers), self-review (E8M0 zero-scale clamp; 2D and 3D expert tensors)
// and inline review (a K/32 scale dimension of 1 is real).  Block rule from
// the OCP MX v1.0 specification: e = floor(log2 amax) - 8 + 127 for E4M3.
//
// Work split: 128-row x 128-column tiles of the [batch * m, k] row-major view
// of the weights, two consecutive tiles per CTA of 256 threads on a grid that
// covers the group's tiles once; one tile is exactly one 512-byte tile of the
// swizzled scale buffer (128 rows x 4 scale columns).  Thread 0 requests both
// tiles at once, each a single 2D tensor-map copy (cp.async.bulk.tensor, a
// 128 x 128 bf16 box = 32 KB) into its own shared-memory stage armed on its
// mbarrier; rows past the end of a matrix belong to the next matrix or read
// as zeros and are ignored.  Each warp then covers 16 rows, two rows per
// 16-byte shared-memory read (16 lanes x 8 bf16 = 128 columns, no bank
// conflicts); 4 lanes share a 32-element block and reduce its amax with two
// xor-shuffles.  The 512 scale bytes are placed at their swizzled positions
// in shared memory and leave the CTA as one contiguous 512-byte store; codes
// are written row-major.
//
// The exponent needs no floating-point log: for a finite amax >= 0 with
// biased binary32 exponent E, floor(log2 amax) - 8 + 127 = E - 8 when amax
// is normal, and every subnormal or zero amax clamps to 0 -- so
// e = max(E - 8, 0).  The scaling by 2^(127 - e) is exact (a power of two in
// the normal range, 2^-119 .. 2^127).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

// 256 threads (8 warps of 16 rows) per CTA: with 512 the per-tile barrier
// waited on twice as many warps.  Two consecutive tiles per CTA, both
// requested at once; the grid covers the layer once (not persistent), so the
// hardware hands out tiles in order and the tiles in flight stay in one
// narrow address window (3 CTAs per SM by shared memory).  A persistent grid
// of 3-stage CTAs walking the tiles grid-stride took 288.8 us on a whole
// Qwen3-30B-A3B layer against 268.3 us for this form.
constexpr int kMxThreads = 256;
constexpr int kMxRowsPerWarp = 128 / (kMxThreads / 32);
constexpr int kMxTilesPerCta = 2;
constexpr int kMxStageBytes = 128 * 128 * 2;
// stages (1024-byte aligned for the tensor copies), two 512-byte scale
// tiles, the barriers, and slack to align the dynamic shared memory base
constexpr size_t kMxSmem = (size_t)kMxTilesPerCta * kMxStageBytes + 2 * 512 + 8 * kMxTilesPerCta + 1024;

// Up to kMxMaxGroup weight tensors quantized by one launch (a whole layer:
// the expert batches and the attention matrices).  Tensor g owns the global
// tiles [tile_start[g], tile_start[g + 1]).
constexpr int kMxMaxGroup = MXFP8_MAX_GROUP;

struct MxGroup {
    CUtensorMap tmap[kMxMaxGroup];          // [batch * m, k] 16-bit view, 128 x 128 boxes
    int64_t m[kMxMaxGroup];
    int64_t k[kMxMaxGroup];
    int64_t col_tiles[kMxMaxGroup];
    int64_t tiles_per_mat[kMxMaxGroup];
    int64_t tile_start[kMxMaxGroup + 1];
    uint8_t* codes[kMxMaxGroup];
    uint8_t* scales[kMxMaxGroup];
    int count;
    int inputs_ready;                       // the weights may be read before the predecessor grid ends
};

// Which tensor of the group global tile t belongs to (CTA-uniform).
__device__ __forceinline__ int group_of(const MxGroup& g, int64_t t) {
    int gi = 0;
    while (gi + 1 < g.count && t >= g.tile_start[gi + 1]) ++gi;
    return gi;
}

// Where one tile of the group lives: its tensor, matrix, row and column
// tile, and its outputs.  Both of a CTA's tiles are resolved first, before
// anything waits, so the parameter loads overlap the copies in flight
// (264 us against 268 us for the layer when they were resolved after each
// tile's data had landed).
struct MxTileDesc {
    const CUtensorMap* tmap;
    uint8_t* codes;
    uint8_t* scales_tile;
    int64_t m, k, bt, rt, ct;
    int y;       // tensor-map row coordinate
    bool valid;
};

__device__ __forceinline__ MxTileDesc mx_desc(const MxGroup& g, int64_t t, int64_t total_tiles) {
    MxTileDesc d;
    d.valid = t < total_tiles;
    const int gi = group_of(g, d.valid ? t : 0);
    const int64_t local = t - g.tile_start[gi];
    d.m = g.m[gi];
    d.k = g.k[gi];
    d.bt = local / g.tiles_per_mat[gi];
    const int64_t rem = local - d.bt * g.tiles_per_mat[gi];
    d.rt = rem / g.col_tiles[gi];
    d.ct = rem - d.rt * g.col_tiles[gi];
    d.tmap = &g.tmap[gi];
    d.codes = g.codes[gi];
    d.scales_tile = g.scales[gi] + local * 512;
    d.y = (int)(d.bt * d.m + d.rt * 128);
    return d;
}

__global__ void __launch_bounds__(kMxThreads)
mxfp8_quantize_kernel(const __grid_constant__ MxGroup g) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* sbuf = smem + kMxTilesPerCta * kMxStageBytes;            // [2][512]
    uint64_t* full = reinterpret_cast<uint64_t*>(sbuf + 2 * 512);
    const unsigned tid = threadIdx.x;
    const unsigned lane = tid & 31u;
    const unsigned warp = tid >> 5;
    const unsigned c = lane & 15u;                 // 8-column chunk inside the tile
    const unsigned jl = c >> 2;                    // scale column inside the tile
    const int64_t total_tiles = g.tile_start[g.count];
    const int64_t t0 = (int64_t)blockIdx.x * kMxTilesPerCta;
    // both tiles' coordinates, resolved before anything waits
    const MxTileDesc D0 = mx_desc(g, t0, total_tiles);
    const MxTileDesc D1 = mx_desc(g, t0 + 1, total_tiles);

    if (tid == 0) {
        for (int s = 0; s < kMxTilesPerCta; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto request = [&]() {
        if (D0.valid) {
            mbar_arrive_expect_tx(&full[0], kMxStageBytes);
            tma_2d_g2s(smem, D0.tmap, (int)(D0.ct * 128), D0.y, &full[0]);
        }
        if (D1.valid) {
            mbar_arrive_expect_tx(&full[1], kMxStageBytes);
            tma_2d_g2s(smem + kMxStageBytes, D1.tmap, (int)(D1.ct * 128), D1.y, &full[1]);
        }
    };
    // with inputs_ready the caller guarantees that no kernel still running
    // writes the weights: the tiles are requested before the wait
    if (tid == 0 && g.inputs_ready) request();
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && !g.inputs_ready) request();

    int it = 0;
    bool failed = false;
#pragma unroll
    for (; it < kMxTilesPerCta; ++it) {
        const MxTileDesc& D = it == 0 ? D0 : D1;
        if (!D.valid) break;
        const bool ok = mbar_wait(&full[it], 0u);
        const uint8_t* st = smem + (size_t)it * kMxStageBytes;
        uint8_t* sb = sbuf + (it & 1) * 512;
        const int64_t m = D.m, k = D.k;
        const int64_t col = D.ct * 128 + c * 8;
        const bool col_ok = col < k;
#pragma unroll
        for (int i = 0; i < kMxRowsPerWarp / 2; ++i) {
            const int rl = warp * kMxRowsPerWarp + 2 * i + (lane >> 4);    // row inside the tile
            const int64_t row = D.rt * 128 + rl;
            const uint4 v = *reinterpret_cast<const uint4*>(st + rl * 256 + c * 16);
            float f[8];
            unpack8(v, f);
            float a = fabsf(f[0]);
#pragma unroll
            for (int e = 1; e < 8; ++e) a = fmaxf(a, fabsf(f[e]));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
            const int E = (int)(__float_as_uint(a) >> 23);           // a >= 0: no sign bit
            const bool valid = col_ok && row < m;
            const int e8 = (valid && E > 8) ? E - 8 : 0;              // E8M0 byte; padding stays 0
            const float factor = __uint_as_float((uint32_t)(254 - e8) << 23);   // 2^(127 - e8)
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = __fmul_rn(f[e], factor);
            if (valid)
                st_stream(D.codes + ((D.bt * m + row) * k + col),
                          make_uint2(cvt_fp8x4<kE4M3>(q[0], q[1], q[2], q[3]), cvt_fp8x4<kE4M3>(q[4], q[5], q[6], q[7])));
            if ((c & 3u) == 0) sb[(rl & 31) * 16 + (rl >> 5) * 4 + jl] = (uint8_t)e8;
        }
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid < 32) st_stream(D.scales_tile + tid * 16, *reinterpret_cast<const uint4*>(sb + tid * 16));
    }
    if (failed && tid == 0) {
        // report, and let the copies still in flight land before the CTA's
        // shared memory is released
        raise_error(kErrCopyTimeout);
        for (int jj = it; jj < kMxTilesPerCta; ++jj)
            if (t0 + jj < total_tiles) mbar_wait(&full[jj], 0u);
    }
}

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library directly).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace fp8q

namespace fp8q {
unsigned unit_errors_mxfp8(bool clear) { return read_unit_errors(clear); }
}  // namespace fp8q

using namespace fp8q;

extern "C" size_t mxfp8_swizzled_scale_bytes(int64_t batch, int64_t m, int64_t k) {
    if (batch < 0 || m < 0 || k <= 0 || k % MXFP8_BLOCK != 0) return 0;
    const int64_t kb = k / MXFP8_BLOCK;
    return (size_t)batch * (size_t)((m + 127) / 128) * (size_t)((kb + 3) / 4) * 512u;
}

namespace fp8q {

// Argument checks of one tensor of a group; sets *tiles to its tile count.
static fp8q_status_t check_tensor(const mxfp8_tensor_t& t, int64_t* tiles) {
    *tiles = 0;
    if (t.batch < 0 || t.m < 0) return FP8Q_ERR_SIZE;
    if (t.k <= 0 || t.k % MXFP8_BLOCK != 0) return FP8Q_ERR_K;
    if (t.m > 0 && t.batch > 0 && (uint64_t)t.k > FP8Q_MAX_ELEMENTS / (uint64_t)t.m / (uint64_t)t.batch)
        return FP8Q_ERR_SIZE;
    const size_t n = (size_t)t.batch * (size_t)t.m * (size_t)t.k;
    if (n == 0) return FP8Q_OK;
    if (!t.w_bf16 || !t.codes || !t.scales_swizzled) return FP8Q_ERR_NULL;
    if (!aligned16(t.w_bf16) || !aligned16(t.codes) || !aligned16(t.scales_swizzled)) return FP8Q_ERR_ALIGN;
    // tensor-map coordinates are 32-bit signed
    if (t.batch * t.m >= (int64_t)1 << 31 || t.k >= (int64_t)1 << 31) return FP8Q_ERR_SIZE;
    *tiles = t.batch * ((t.m + 127) / 128) * ((t.k / MXFP8_BLOCK + 3) / 4);
    return FP8Q_OK;
}

// The byte ranges a tensor reads (0) and writes (1, 2).
static void tensor_ranges(const mxfp8_tensor_t& t, const void* p[3], size_t sz[3]) {
    const size_t n = (size_t)t.batch * (size_t)t.m * (size_t)t.k;
    p[0] = t.w_bf16;
    sz[0] = 2 * n;
    p[1] = t.codes;
    sz[1] = n;
    p[2] = t.scales_swizzled;
    sz[2] = mxfp8_swizzled_scale_bytes(t.batch, t.m, t.k);
}

static fp8q_status_t launch_group(const mxfp8_tensor_t* tensors, int count, cudaStream_t stream, unsigned flags = 0) {
    if (flags & ~FP8Q_INPUTS_READY) return FP8Q_ERR_FLAGS;
    if (!tensors) return FP8Q_ERR_NULL;
    if (count < 1 || count > kMxMaxGroup) return FP8Q_ERR_SIZE;
    int64_t tiles[kMxMaxGroup];
    for (int i = 0; i < count; ++i) {
        const fp8q_status_t st = check_tensor(tensors[i], &tiles[i]);
        if (st != FP8Q_OK) return st;
    }
    // no output may overlap any input or output of any tensor of the group
    for (int i = 0; i < count; ++i) {
        if (tiles[i] == 0) continue;
        const void* pi[3];
        size_t si[3];
        tensor_ranges(tensors[i], pi, si);
        for (int j = 0; j < count; ++j) {
            if (tiles[j] == 0) continue;
            const void* pj[3];
            size_t sj[3];
            tensor_ranges(tensors[j], pj, sj);
            for (int a = 1; a < 3; ++a)
                for (int b = 0; b < 3; ++b) {
                    if (i == j && a == b) continue;
                    if (overlaps(pi[a], si[a], pj[b], sj[b])) return FP8Q_ERR_ALIAS;
                }
        }
    }
    int64_t all_tiles = 0;
    for (int i = 0; i < count; ++i) all_tiles += tiles[i];
    if (all_tiles == 0) return FP8Q_OK;                 // nothing to do, nothing launched
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cuda_status(cudaErrorNotSupported);
    MxGroup g;
    int used = 0;
    int64_t start = 0;
    for (int i = 0; i < count; ++i) {
        const mxfp8_tensor_t& t = tensors[i];
        if (tiles[i] == 0) continue;
        // the weights as a 2D [batch * m, k] array of 16-bit elements, 128 x 128 boxes
        const cuuint64_t dims[2] = {(cuuint64_t)t.k, (cuuint64_t)(t.batch * t.m)};
        const cuuint64_t strides[1] = {(cuuint64_t)t.k * 2};
        const cuuint32_t box[2] = {128, 128};
        const cuuint32_t estride[2] = {1, 1};
        const CUresult cr = encode(&g.tmap[used], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(t.w_bf16), dims,
                                   strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cuda_status(cudaErrorInvalidValue);
        g.m[used] = t.m;
        g.k[used] = t.k;
        g.col_tiles[used] = (t.k / MXFP8_BLOCK + 3) / 4;
        g.tiles_per_mat[used] = ((t.m + 127) / 128) * g.col_tiles[used];
        g.tile_start[used] = start;
        g.codes[used] = t.codes;
        g.scales[used] = t.scales_swizzled;
        start += tiles[i];
        ++used;
    }
    if (used == 0) return FP8Q_OK;
    g.tile_start[used] = start;
    g.count = used;
    g.inputs_ready = (flags & FP8Q_INPUTS_READY) ? 1 : 0;
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, mxfp8_quantize_kernel, kMxThreads, kMxSmem, kMxSmem, &resident);
    if (st != FP8Q_OK) return st;
    const size_t grid = ((size_t)start + kMxTilesPerCta - 1) / kMxTilesPerCta;
    if (grid > 0x7FFFFFFFu) return FP8Q_ERR_SIZE;
    return launch(mxfp8_quantize_kernel, (unsigned)grid, kMxThreads, kMxSmem, stream, g);
}

}  // namespace fp8q

extern "C" fp8q_status_t mxfp8_quantize_swizzled(const void* w_bf16, int64_t batch, int64_t m, int64_t k,
                                                 uint8_t* codes, uint8_t* scales_swizzled, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("mxfp8_quantize_swizzled");
    const mxfp8_tensor_t t = {w_bf16, batch, m, k, codes, scales_swizzled};
    return launch_group(&t, 1, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8q_status_t mxfp8_quantize_swizzled_group(const mxfp8_tensor_t* tensors, int count,
                                                       fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("mxfp8_quantize_swizzled_group");
    return launch_group(tensors, count, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8q_status_t mxfp8_quantize_swizzled_group_ex(const mxfp8_tensor_t* tensors, int count,
                                                          unsigned int flags, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("mxfp8_quantize_swizzled_group_ex");
    return launch_group(tensors, count, reinterpret_cast<cudaStream_t>(stream), flags);
}
