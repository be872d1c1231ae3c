// (b) Fused k-way dequantize-then-reduce, single-shard dequantize, and the
// naive two-pass order kept as a comparator.
//
// "FP8 Transmission Optimization for VLA Training", section "FP8
// Transmission Optimization and Bottlenecks": the naive order dequantizes
// every shard to HBM and reduces afterwards; the fused kernel reads each
// shard's codes and scales once and keeps the running sum in registers.
//
// Work split: a persistent CTA of 512 threads walks tiles of 4096 elements
// (32 blocks).  Thread 0 keeps up to kRedStages tiles in flight: for each
// tile it issues 2k bulk copies (the k shards' 4096 codes and 32 scales)
// into one shared-memory stage, armed on that stage's mbarrier.  All threads
// wait on the stage's barrier, then each takes 4 consecutive elements in
// each of 2 rounds (a warp covers 128 contiguous elements, one block, per
// round), reads its codes and the block's scale from shared memory and sums
// in rank order 0..k-1:
//   acc = +0;  acc = RN(acc + RN(decode(c_r) * s_r))
// with explicit _rn intrinsics so nothing is fused into an FMA.  Each round
// a warp stores 512 contiguous bytes of fp32 and 256 of bf16.  The ragged
// last tile (n not a multiple of 4096) is read straight from global memory.
#include <mutex>

#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kRedThreads = 512;

// Four codes of a word -> four binary32.  E5M2 codes go straight from the
// word's bytes to two f16 pairs (an E5M2 code is the upper byte of the f16 of
// the same value), without first splitting the word into 16-bit halves:
// with the split, the k = 8 e5m2 reduce took 32.8 us against 30.7 us.
template <int FMT>
__device__ __forceinline__ void red_decode4(uint32_t w, float* f) {
    if (FMT == kE5M2) {
        const uint32_t lo = __byte_perm(w, 0u, 0x1404u), hi = __byte_perm(w, 0u, 0x3424u);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
        decode_fp8x4<FMT>(w, f);
    }
}

constexpr int kRedTile = 4096;
constexpr int kRedStages = 3;

// Shared memory of one stage for k shards: k x (4096 codes + 32 fp32 scales).
__host__ __device__ constexpr uint32_t red_stage_bytes(int k) { return (uint32_t)k * (kRedTile + 4 * (kRedTile / 128)); }
constexpr size_t red_smem_bytes(int k) { return (size_t)kRedStages * red_stage_bytes(k) + 8 * kRedStages; }

struct ShardPtrs {
    const uint8_t* codes[FP8Q_MAX_SHARDS];
    const float* scales[FP8Q_MAX_SHARDS];
};

// 4 results at element e: fp32 as one 16-byte store, bf16 as one 8-byte store.
template <bool OUT_BF16, bool OUT_F32>
__device__ __forceinline__ void store4(const float (&acc)[4], size_t e, uint16_t* out_bf16, float* out_f32) {
    if (OUT_F32)
        st_stream(out_f32 + e, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                          __float_as_uint(acc[3])));
    if (OUT_BF16) st_stream(out_bf16 + e, make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3])));
}

// 16 results at element e0 (the comparator's second pass): fp32 as four
// 16-byte stores, bf16 as two; a ragged end element by element.
template <bool OUT_BF16, bool OUT_F32>
__device__ __forceinline__ void store16(const float (&acc)[16], size_t e0, size_t n, uint16_t* out_bf16,
                                        float* out_f32) {
    const bool full = e0 + 16 <= n;
    if (OUT_F32) {
        if (full) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st_stream(out_f32 + e0 + 4 * q, make_uint4(__float_as_uint(acc[4 * q]), __float_as_uint(acc[4 * q + 1]),
                                                           __float_as_uint(acc[4 * q + 2]),
                                                           __float_as_uint(acc[4 * q + 3])));
        } else {
            st_f32_tail(out_f32 + e0, acc, 16, (long long)n - (long long)e0);
        }
    }
    if (OUT_BF16) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
        if (full) {
            st_stream(out_bf16 + e0, make_uint4(w[0], w[1], w[2], w[3]));
            st_stream(out_bf16 + e0 + 8, make_uint4(w[4], w[5], w[6], w[7]));
        } else {
            st_u16_tail(out_bf16 + e0, w, 8, (long long)n - (long long)e0);
        }
    }
}

// SUM = true: acc starts at +0 and every shard is added (the reduce).
// SUM = false: k == 1 and the dequantized value is written as is (dequantize).
// KMAX >= k bounds the unrolled shard loop (a power of two, so at most half
// of the unrolled iterations are switched off).
template <int FMT, bool OUT_BF16, bool OUT_F32, bool SUM, int KMAX>
__global__ void __launch_bounds__(kRedThreads)
dequant_reduce_kernel(ShardPtrs sh, int k, size_t n, uint16_t* __restrict__ out_bf16, float* __restrict__ out_f32,
                      int inputs_ready) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t stage_bytes = red_stage_bytes(k);
    const uint32_t codes_bytes = (uint32_t)k * kRedTile;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRedStages * stage_bytes);
    const size_t ntiles = (n + kRedTile - 1) / kRedTile;
    const size_t nstaged = n / kRedTile;               // tiles entirely inside the arrays
    const unsigned tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < kRedStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto issue = [&](size_t t, int s) {           // thread 0 only
        uint8_t* st = smem + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        for (int r = 0; r < k; ++r) {
            bulk_g2s(st + r * kRedTile, sh.codes[r] + t * kRedTile, kRedTile, &full[s]);
            bulk_g2s(st + codes_bytes + r * (4 * kRedTile / 128), sh.scales[r] + t * (kRedTile / 128),
                     4 * kRedTile / 128, &full[s]);
        }
    };
    auto prologue = [&]() {                       // thread 0 only: the first tiles
        for (int s = 0; s < kRedStages; ++s) {
            const size_t t = blockIdx.x + (size_t)s * gridDim.x;
            if (t < nstaged) issue(t, s);
        }
    };
    // with inputs_ready the caller guarantees that no kernel still running
    // writes the shards: the first tiles are requested before the wait
    if (tid == 0 && inputs_ready) prologue();
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && !inputs_ready) prologue();

    int it = 0;
    bool failed = false;
    for (size_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = it % kRedStages;
        const bool staged = t < nstaged;
        const bool ok = staged ? mbar_wait(&full[s], (uint32_t)(it / kRedStages) & 1u) : true;
        const uint8_t* st = smem + (size_t)s * stage_bytes;
#pragma unroll 1
        for (int m = 0; m < kRedTile / (4 * kRedThreads); ++m) {
            const uint32_t el = m * (4 * kRedThreads) + 4 * tid;   // element inside the tile
            const size_t e = t * kRedTile + el;               // element inside the arrays
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (staged) {
                uint32_t w[KMAX];
                float sc[KMAX];
#pragma unroll
                for (int r = 0; r < KMAX; ++r) {
                    if (r < k) {
                        w[r] = *reinterpret_cast<const uint32_t*>(st + r * kRedTile + el);
                        sc[r] = *reinterpret_cast<const float*>(st + codes_bytes + r * (4 * kRedTile / 128) +
                                                                (el >> 7) * 4);
                    }
                }
#pragma unroll
                for (int r = 0; r < KMAX; ++r) {
                    if (r < k) {
                        float d[4];
                        red_decode4<FMT>(w[r], d);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float p = __fmul_rn(d[q], sc[r]);
                            acc[q] = SUM ? __fadd_rn(acc[q], p) : p;
                        }
                    }
                }
                store4<OUT_BF16, OUT_F32>(acc, e, out_bf16, out_f32);
            } else if (e < n) {
                // the ragged last tile, element by element from global memory
                for (int r = 0; r < k; ++r) {
                    const float sc = sh.scales[r][e >> 7];
                    for (int q = 0; q < 4; ++q) {
                        if (e + q < n) {
                            const float d = decode_fp8x2<FMT>(sh.codes[r][e + q]).x;
                            const float p = __fmul_rn(d, sc);
                            acc[q] = SUM ? __fadd_rn(acc[q], p) : p;
                        }
                    }
                }
                for (int q = 0; q < 4; ++q) {
                    if (e + q < n) {
                        if (OUT_F32) out_f32[e + q] = acc[q];
                        if (OUT_BF16) out_bf16[e + q] = (uint16_t)(pack_bf16x2(acc[q], 0.0f) & 0xFFFFu);
                    }
                }
            }
        }
        // every thread is done with stage s; refill it with this CTA's tile
        // kRedStages steps ahead
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            const size_t tn = t + (size_t)kRedStages * gridDim.x;
            if (tn < nstaged) {
                fence_proxy_async_smem();
                issue(tn, s);
            }
        }
    }
    if (failed && tid == 0) {
        // report, and let the copies still in flight land before the CTA's
        // shared memory is released
        raise_error(kErrCopyTimeout);
        for (int j = it; j < it + kRedStages; ++j) {
            const size_t tj = blockIdx.x + (size_t)j * gridDim.x;
            if (tj < nstaged) mbar_wait(&full[j % kRedStages], (uint32_t)(j / kRedStages) & 1u);
        }
    }
}

// Second pass of the naive order: k fp32 arrays (`slot` floats apart, a
// multiple of 4 so every slot is 16-byte aligned) summed in rank order from +0.
template <bool OUT_BF16, bool OUT_F32>
__global__ void __launch_bounds__(kRedThreads)
sum_f32_kernel(const float* __restrict__ ws, int k, size_t n, size_t slot, uint16_t* __restrict__ out_bf16,
               float* __restrict__ out_f32) {
    dependency_wait();
    allow_dependents();
    const size_t units = (n + 15) >> 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const size_t e0 = u << 4;
        const bool full = e0 + 16 <= n;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        for (int r = 0; r < k; ++r) {
            const float* p = ws + (size_t)r * slot + e0;
            float v[16];
            if (full) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 t = ld_stream(p + 4 * q);
                    v[4 * q] = __uint_as_float(t.x); v[4 * q + 1] = __uint_as_float(t.y);
                    v[4 * q + 2] = __uint_as_float(t.z); v[4 * q + 3] = __uint_as_float(t.w);
                }
            } else {
                for (int i = 0; i < 16; ++i) v[i] = (e0 + i < n) ? p[i] : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], v[i]);
        }
        store16<OUT_BF16, OUT_F32>(acc, e0, n, out_bf16, out_f32);
    }
}

template <int FMT, bool B, bool F, bool SUM, int KMAX>
static fp8q_status_t launch_reduce_k(const ShardPtrs& sh, int k, size_t n, uint16_t* ob, float* of, cudaStream_t s,
                                     int ready) {
    auto kernel = dequant_reduce_kernel<FMT, B, F, SUM, KMAX>;
    // one cache per shard count: the stage size, and so the occupancy, depends on k
    static KernelCache kc[KMAX + 1];
    const size_t smem = red_smem_bytes(k);
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc[k], kernel, kRedThreads, smem, red_smem_bytes(KMAX), &resident);
    if (st != FP8Q_OK) return st;
    const size_t tiles = (n + kRedTile - 1) / kRedTile;
    const unsigned grid = grid_for(tiles, resident);
    return launch(kernel, grid, kRedThreads, smem, s, sh, k, n, ob, of, ready);
}

template <int FMT, bool B, bool F, bool SUM>
static fp8q_status_t launch_reduce_t(const ShardPtrs& sh, int k, size_t n, uint16_t* ob, float* of, cudaStream_t s,
                                     int ready) {
    if constexpr (!SUM) {
        return launch_reduce_k<FMT, B, F, SUM, 1>(sh, k, n, ob, of, s, ready);
    } else {
        if (k <= 2) return launch_reduce_k<FMT, B, F, SUM, 2>(sh, k, n, ob, of, s, ready);
        if (k <= 4) return launch_reduce_k<FMT, B, F, SUM, 4>(sh, k, n, ob, of, s, ready);
        if (k <= 8) return launch_reduce_k<FMT, B, F, SUM, 8>(sh, k, n, ob, of, s, ready);
        return launch_reduce_k<FMT, B, F, SUM, 16>(sh, k, n, ob, of, s, ready);
    }
}

template <int FMT, bool SUM>
static fp8q_status_t launch_reduce(const ShardPtrs& sh, int k, size_t n, uint16_t* ob, float* of, cudaStream_t s,
                                   int ready = 0) {
    if (ob && of) return launch_reduce_t<FMT, true, true, SUM>(sh, k, n, ob, of, s, ready);
    if (ob) return launch_reduce_t<FMT, true, false, SUM>(sh, k, n, ob, of, s, ready);
    return launch_reduce_t<FMT, false, true, SUM>(sh, k, n, ob, of, s, ready);
}

template <bool B, bool F>
static fp8q_status_t launch_sum_t(const float* ws, int k, size_t n, size_t stride, uint16_t* ob, float* of,
                                  cudaStream_t s) {
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, sum_f32_kernel<B, F>, kRedThreads, 0, 0, &resident);
    if (st != FP8Q_OK) return st;
    const size_t units = (n + 15) / 16;
    const unsigned grid = grid_for((units + kRedThreads - 1) / kRedThreads, resident);
    return launch(sum_f32_kernel<B, F>, grid, kRedThreads, 0, s, ws, k, n, stride, ob, of);
}

// Shared argument checks of the multi-shard entry points.
static fp8q_status_t check_shards(const uint8_t* const* codes, const float* const* scales, int k, size_t n,
                                  fp8q_format_t fmt, const void* out_bf16, const float* out_fp32, ShardPtrs* sh) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (k < 1 || k > FP8Q_MAX_SHARDS) return FP8Q_ERR_K;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!codes || !scales) return FP8Q_ERR_NULL;
    if (!out_bf16 && !out_fp32) return FP8Q_ERR_NULL;
    const size_t nb = fp8q_num_scales(n);
    for (int r = 0; r < FP8Q_MAX_SHARDS; ++r) {
        sh->codes[r] = nullptr;
        sh->scales[r] = nullptr;
    }
    for (int r = 0; r < k; ++r) {
        if (!codes[r] || !scales[r]) return FP8Q_ERR_NULL;
        if (!aligned16(codes[r]) || !aligned16(scales[r])) return FP8Q_ERR_ALIGN;
        if (overlaps(out_bf16, 2 * n, codes[r], n) || overlaps(out_bf16, 2 * n, scales[r], 4 * nb) ||
            overlaps(out_fp32, 4 * n, codes[r], n) || overlaps(out_fp32, 4 * n, scales[r], 4 * nb))
            return FP8Q_ERR_ALIAS;
        sh->codes[r] = codes[r];
        sh->scales[r] = scales[r];
    }
    if ((out_bf16 && !aligned16(out_bf16)) || (out_fp32 && !aligned16(out_fp32))) return FP8Q_ERR_ALIGN;
    if (overlaps(out_bf16, 2 * n, out_fp32, 4 * n)) return FP8Q_ERR_ALIAS;
    return FP8Q_OK;
}

}  // namespace fp8q

namespace fp8q {
unsigned unit_errors_reduce(bool clear) { return read_unit_errors(clear); }
}  // namespace fp8q

using namespace fp8q;

extern "C" size_t fp8q_unfused_stride(size_t n) { return (n + 3) & ~(size_t)3; }

static fp8q_status_t reduce_entry(const uint8_t* const* codes, const float* const* scales, int k, size_t n,
                                  fp8q_format_t fmt, void* out_bf16, float* out_fp32, unsigned flags,
                                  fp8q_stream_t stream) {
    if (flags & ~FP8Q_INPUTS_READY) return FP8Q_ERR_FLAGS;
    ShardPtrs sh;
    fp8q_status_t st = check_shards(codes, scales, k, n, fmt, out_bf16, out_fp32, &sh);
    if (st != FP8Q_OK || n == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t* ob = static_cast<uint16_t*>(out_bf16);
    const int ready = (flags & FP8Q_INPUTS_READY) ? 1 : 0;
    return fmt == FP8Q_E4M3 ? launch_reduce<kE4M3, true>(sh, k, n, ob, out_fp32, s, ready)
                            : launch_reduce<kE5M2, true>(sh, k, n, ob, out_fp32, s, ready);
}

extern "C" fp8q_status_t fp8q_dequant_reduce(const uint8_t* const* codes, const float* const* scales, int k,
                                             size_t n, fp8q_format_t fmt, void* out_bf16, float* out_fp32,
                                             fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_dequant_reduce");
    return reduce_entry(codes, scales, k, n, fmt, out_bf16, out_fp32, 0, stream);
}

extern "C" fp8q_status_t fp8q_dequant_reduce_ex(const uint8_t* const* codes, const float* const* scales, int k,
                                                size_t n, fp8q_format_t fmt, void* out_bf16, float* out_fp32,
                                                unsigned int flags, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_dequant_reduce_ex");
    return reduce_entry(codes, scales, k, n, fmt, out_bf16, out_fp32, flags, stream);
}

extern "C" fp8q_status_t fp8q_dequantize(const uint8_t* codes, const float* scales, size_t n, fp8q_format_t fmt,
                                         void* out_bf16, float* out_fp32, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_dequantize");
    ShardPtrs sh;
    const uint8_t* c[1] = {codes};
    const float* sc[1] = {scales};
    fp8q_status_t st = check_shards(c, sc, 1, n, fmt, out_bf16, out_fp32, &sh);
    if (st != FP8Q_OK || n == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t* ob = static_cast<uint16_t*>(out_bf16);
    return fmt == FP8Q_E4M3 ? launch_reduce<kE4M3, false>(sh, 1, n, ob, out_fp32, s)
                            : launch_reduce<kE5M2, false>(sh, 1, n, ob, out_fp32, s);
}

namespace fp8q {


// ------------------------------------------------ all-gather decode ----
// The end of the simulated ring AllReduce: every rank decodes the same
// gathered codes.  The ranks share one GPU and one copy of the codes, so a
// tile of 4096 codes and its 32 scales is staged once (bulk copies, like the
// reduce with k = 1) and its bf16 values are stored to every rank's output.
// Each of the 512 threads takes 8 consecutive elements (one 16-byte store
// per output; a warp writes 512 contiguous bytes of each output).
// One tile per CTA, on a grid that covers the codes once (not persistent):
// CTAs are dispatched in tile order, so the stores in flight stay in one
// narrow window of each output.  (A persistent grid of 4-stage CTAs walking
// the tiles grid-stride made the 8-rank AllReduce of 256 MiB per rank take
// 1.16 ms against 1.10 ms with this form.)
// MEAN: the decoded value is divided by `divisor` (the rank count) first,
// RN(d / divisor), by markstein_div<2> from y = RN(1/divisor) (exact for
// binary32 dividends with |d| >= 2^-78) and by the IEEE division below that.

constexpr uint32_t kGatherStageBytes = kRedTile + 4 * (kRedTile / 128);
constexpr size_t kGatherSmem = (size_t)kGatherStageBytes + 8;

struct GatherDests {
    uint16_t* out[FP8Q_MAX_HOP_GROUP];
};

template <bool MEAN>
__device__ __forceinline__ float gather_value(float d, float divisor, float y) {
    if (!MEAN) return d;
    return fabsf(d) >= 0x1p-78f ? markstein_div<2>(d, divisor, y) : __fdiv_rn(d, divisor);
}

template <int FMT, bool MEAN>
__global__ void __launch_bounds__(kRedThreads)
gather_decode_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales, size_t n,
                     const __grid_constant__ GatherDests dst, int count, float divisor) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGatherStageBytes);
    const size_t nstaged = n / kRedTile;
    const size_t t = blockIdx.x;
    const unsigned tid = threadIdx.x;
    const float y = MEAN ? __frcp_rn(divisor) : 1.0f;
    const bool staged = t < nstaged;

    if (tid == 0) {
        mbar_init(full, 1);
        fence_barrier_init();
    }
    // the codes are the previous launch's output: no copy before the wait
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0 && staged) {
        mbar_arrive_expect_tx(full, kGatherStageBytes);
        bulk_g2s(smem, codes + t * kRedTile, kRedTile, full);
        bulk_g2s(smem + kRedTile, scales + t * (kRedTile / 128), 4 * kRedTile / 128, full);
    }
    const bool ok = staged ? mbar_wait(full, 0u) : true;
    const uint32_t el = 8 * tid;
    const size_t e = t * kRedTile + el;
    if (staged) {
        const uint2 c8 = *reinterpret_cast<const uint2*>(smem + el);
        const float sc = *reinterpret_cast<const float*>(smem + kRedTile + (el >> 7) * 4);
        float d[8];
        decode_fp8x4<FMT>(c8.x, d);
        decode_fp8x4<FMT>(c8.y, d + 4);
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = pack_bf16x2(gather_value<MEAN>(__fmul_rn(d[2 * q], sc), divisor, y),
                               gather_value<MEAN>(__fmul_rn(d[2 * q + 1], sc), divisor, y));
        const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int o = 0; o < FP8Q_MAX_HOP_GROUP; ++o)
            if (o < count) st_stream(dst.out[o] + e, v);
    } else if (e < n) {
        // the ragged last tile, element by element from global memory
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        for (int q = 0; q < 8; ++q) {
            if (e + q < n) {
                const float dq = decode_fp8x2<FMT>(codes[e + q]).x;
                const float v = gather_value<MEAN>(__fmul_rn(dq, scales[(e + q) >> 7]), divisor, y);
                w[q >> 1] |= (pack_bf16x2(v, 0.0f) & 0xFFFFu) << ((q & 1) * 16);
            }
        }
        for (int o = 0; o < count; ++o) st_u16_tail(dst.out[o] + e, w, 4, (long long)n - (long long)e);
    }
    // a copy that did not land in time: report, and give it one more bounded
    // wait before the CTA's shared memory is released
    if (__syncthreads_or(!ok) && tid == 0) {
        raise_error(kErrCopyTimeout);
        mbar_wait(full, 0u);
    }
}

template <int FMT, bool MEAN>
static fp8q_status_t launch_gather(const uint8_t* codes, const float* scales, size_t n, const GatherDests& dst,
                                   int count, float divisor, cudaStream_t s) {
    auto kernel = gather_decode_kernel<FMT, MEAN>;
    static KernelCache kc;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, kernel, kRedThreads, kGatherSmem, 0, &resident);
    if (st != FP8Q_OK) return st;
    const size_t grid = (n + kRedTile - 1) / kRedTile;
    if (grid > 0x7FFFFFFFu) return FP8Q_ERR_SIZE;
    return launch(kernel, (unsigned)grid, kRedThreads, kGatherSmem, s, codes, scales, n, dst, count, divisor);
}

fp8q_status_t gather_decode_entry(const uint8_t* codes, const float* scales, size_t n, fp8q_format_t fmt,
                                  void* const* outs, int count, int mean_divisor, fp8q_stream_t stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (count < 1 || count > FP8Q_MAX_HOP_GROUP || mean_divisor < 0 || mean_divisor > FP8Q_MAX_HOP_GROUP)
        return FP8Q_ERR_K;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!codes || !scales || !outs) return FP8Q_ERR_NULL;
    if (!aligned16(codes) || !aligned16(scales)) return FP8Q_ERR_ALIGN;
    const size_t nb = fp8q_num_scales(n);
    GatherDests dst = {};
    for (int o = 0; o < count; ++o) {
        if (!outs[o]) return FP8Q_ERR_NULL;
        if (!aligned16(outs[o])) return FP8Q_ERR_ALIGN;
        if (overlaps(outs[o], 2 * n, codes, n) || overlaps(outs[o], 2 * n, scales, 4 * nb)) return FP8Q_ERR_ALIAS;
        for (int q = 0; q < o; ++q)
            if (overlaps(outs[o], 2 * n, outs[q], 2 * n)) return FP8Q_ERR_ALIAS;
        dst.out[o] = static_cast<uint16_t*>(outs[o]);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float div = (float)(mean_divisor > 0 ? mean_divisor : 1);
    if (fmt == FP8Q_E4M3)
        return mean_divisor > 0 ? launch_gather<kE4M3, true>(codes, scales, n, dst, count, div, s)
                                : launch_gather<kE4M3, false>(codes, scales, n, dst, count, div, s);
    return mean_divisor > 0 ? launch_gather<kE5M2, true>(codes, scales, n, dst, count, div, s)
                            : launch_gather<kE5M2, false>(codes, scales, n, dst, count, div, s);
}
}  // namespace fp8q


extern "C" fp8q_status_t fp8q_dequant_reduce_unfused(const uint8_t* const* codes, const float* const* scales,
                                                     int k, size_t n, fp8q_format_t fmt, float* workspace,
                                                     void* out_bf16, float* out_fp32, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_dequant_reduce_unfused");
    ShardPtrs sh;
    fp8q_status_t st = check_shards(codes, scales, k, n, fmt, out_bf16, out_fp32, &sh);
    if (st != FP8Q_OK || n == 0) return st;
    if (!workspace) return FP8Q_ERR_NULL;
    if (!aligned16(workspace)) return FP8Q_ERR_ALIGN;
    const size_t stride = fp8q_unfused_stride(n);      // keeps every shard slot 16-byte aligned
    const size_t wbytes = 4 * (size_t)k * stride;
    if (overlaps(workspace, wbytes, out_bf16, 2 * n) || overlaps(workspace, wbytes, out_fp32, 4 * n))
        return FP8Q_ERR_ALIAS;
    for (int r = 0; r < k; ++r)
        if (overlaps(workspace, wbytes, codes[r], n) || overlaps(workspace, wbytes, scales[r], 4 * fp8q_num_scales(n)))
            return FP8Q_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int r = 0; r < k; ++r) {
        ShardPtrs one;
        one.codes[0] = sh.codes[r];
        one.scales[0] = sh.scales[r];
        st = fmt == FP8Q_E4M3 ? launch_reduce<kE4M3, false>(one, 1, n, nullptr, workspace + (size_t)r * stride, s)
                              : launch_reduce<kE5M2, false>(one, 1, n, nullptr, workspace + (size_t)r * stride, s);
        if (st != FP8Q_OK) return st;
    }
    uint16_t* ob = static_cast<uint16_t*>(out_bf16);
    if (ob && out_fp32) return launch_sum_t<true, true>(workspace, k, n, stride, ob, out_fp32, s);
    if (ob) return launch_sum_t<true, false>(workspace, k, n, stride, ob, out_fp32, s);
    return launch_sum_t<false, true>(workspace, k, n, stride, ob, out_fp32, s);
}

// ------------------------------------------------- no-allocation variant ----
extern "C" fp8q_status_t fp8q_gather_decode(const uint8_t* codes, const float* scales, size_t n, fp8q_format_t fmt,
                                            void* const* outs, int count, unsigned int flags, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_gather_decode");
    if (flags & ~FP8Q_ALLREDUCE_MEAN) return FP8Q_ERR_FLAGS;
    return fp8q::gather_decode_entry(codes, scales, n, fmt, outs, count, (flags & FP8Q_ALLREDUCE_MEAN) ? count : 0,
                                     stream);
}

// fp8q_dequant_reduce_unfused with its workspace in a static device array
// instead of a caller-supplied buffer (for callers that cannot allocate).

namespace fp8q {

static __device__ __align__(256) float g_static_scratch[FP8Q_STATIC_SCRATCH_FLOATS];

static std::mutex g_static_scratch_mu;
static float* g_static_scratch_ptr[kMaxDevices];

// Device address of g_static_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and kept.
static fp8q_status_t static_scratch_address(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_status(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (g_static_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        g_static_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_static_scratch_ptr[dev];
    return FP8Q_OK;
}

}  // namespace fp8q

extern "C" fp8q_status_t fp8q_dequant_reduce_unfused_static(const uint8_t* const* codes, const float* const* scales,
                                                            int k, size_t n, fp8q_format_t fmt, void* out_bf16,
                                                            float* out_fp32, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_dequant_reduce_unfused_static");
    ShardPtrs sh;
    fp8q_status_t st = check_shards(codes, scales, k, n, fmt, out_bf16, out_fp32, &sh);
    if (st != FP8Q_OK || n == 0) return st;
    const size_t slot = fp8q_unfused_stride(n);
    if (slot > FP8Q_STATIC_SCRATCH_FLOATS / (size_t)k) return FP8Q_ERR_SIZE;
    float* ws = nullptr;
    st = static_scratch_address(&ws);
    if (st != FP8Q_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int r = 0; r < k; ++r) {
        ShardPtrs one;
        one.codes[0] = sh.codes[r];
        one.scales[0] = sh.scales[r];
        st = fmt == FP8Q_E4M3 ? launch_reduce<kE4M3, false>(one, 1, n, nullptr, ws + (size_t)r * slot, s)
                              : launch_reduce<kE5M2, false>(one, 1, n, nullptr, ws + (size_t)r * slot, s);
        if (st != FP8Q_OK) return st;
    }
    uint16_t* ob = static_cast<uint16_t*>(out_bf16);
    if (ob && out_fp32) return launch_sum_t<true, true>(ws, k, n, slot, ob, out_fp32, s);
    if (ob) return launch_sum_t<true, false>(ws, k, n, slot, ob, out_fp32, s);
    return launch_sum_t<false, true>(ws, k, n, slot, ob, out_fp32, s);
}
