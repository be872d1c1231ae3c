// (c) One hop of a ring reduction carried on the FP8 wire format.
//
// "FP8 Transmission Optimization for VLA Training", section "FP8
// Transmission Optimization and Bottlenecks" (ring-based collectives on the
// FP8 wire) and "How to Speed Up VLA Training Step by Step", PCIe paragraph
// (ring AllReduce of bf16 gradients).  The receiver of a hop dequantizes the
// incoming chunk, adds its own bf16 partial and requantizes the fp32 sum for
// the next hop, in one pass: the sums stay in registers while the block amax
// is reduced, nothing is re-read from HBM.
//
// Work split: a persistent CTA of 256 threads walks tiles of 32 blocks
// (4096 elements).  Thread 0 keeps up to 3 tiles in flight (2 in short hop
// groups, see launch_hop_group_kernel); a tile
// is three bulk copies into one shared-memory stage (4096 incoming codes,
// their 32 scales, 8 KB of the local bf16 partial) armed on the stage's
// mbarrier.  Once it has landed, 8 lanes own one block: lane j takes
// elements [8j, 8j+8) and [64+8j, 64+8j+8) (conflict-free shared-memory
// reads), the amax is a 3-step xor-shuffle among the 8 lanes, and the
// quotients y / s use the per-block reciprocal with two Markstein
// corrections (exact for binary32 dividends, see block_quotients).  The
// sums stay in registers from the add to the requantization.  The ragged last tile is
// read straight from global memory.
//
// With FP8Q_HOP_LOCAL_READY the local partials of each CTA's first tiles are
// copied before the grid-dependency wait, so that they stream in while the
// previous kernel on the stream drains.
//
// A group of two or more hops (every rank's hop of one step of a simulated
// ring) runs ring_hop_group_kernel: the same tiles and arithmetic, with the
// per-tile bookkeeping hoisted out of the loop.  The kernel is bound by
// instruction issue at large sizes (79% issue-active at 20.2
// thread-instructions per element on a 134M-element hop with scalar
// arithmetic; 71% at 16.6 with the packed arithmetic of hop_block16), so
// per-element and per-tile instructions show directly in its time.
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kHopThreads = 256;
constexpr int kHopTileBlocks = 32;
constexpr int kHopTile = kHopTileBlocks * 128;            // elements
constexpr int kHopCodesBytes = kHopTile;
constexpr int kHopScaleBytes = 4 * kHopTileBlocks;
constexpr int kHopLocalBytes = 2 * kHopTile;
constexpr int kHopStageBytes = kHopCodesBytes + kHopScaleBytes + kHopLocalBytes;

// Up to kHopMaxGroup independent hops in one launch (all ranks' hops of one
// step of a ring simulated on one GPU).  Hop h owns the global tiles
// [tile_start[h], tile_start[h + 1]).
constexpr int kHopMaxGroup = FP8Q_MAX_HOP_GROUP;

struct HopGroup {
    const uint8_t* in_codes[kHopMaxGroup];
    const float* in_scales[kHopMaxGroup];
    const uint16_t* local[kHopMaxGroup];
    uint8_t* out_codes[kHopMaxGroup];
    float* out_scales[kHopMaxGroup];
    uint16_t* out_bf16[kHopMaxGroup];          // may be null per hop
    size_t n[kHopMaxGroup];
    int64_t tile_start[kHopMaxGroup + 1];
    int count;
    int local_ready;       // the local partials may be read before the predecessor grid ends
    float nzero;           // -0.0f
};

// Packed two-lane binary32 arithmetic (PTX f32x2: one instruction for two
// values, each lane rounded exactly as the scalar instruction would round it),
// the widening add of a bf16 and a binary32, and the three-input maximum.
// They take the hop from about 20.5 to 17 thread-instructions per element.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// RN(bf16 + x): the bf16 widened exactly, then one rounded add.
__device__ __forceinline__ float add_bf16_f32(uint16_t h, float x) {
    float r;
    asm("add.rn.f32.bf16 %0, %1, %2;" : "=f"(r) : "h"(h), "f"(x));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// One lane's share of one block: 16 incoming codes (ca, cb) with the block's
// incoming scale s_in and 16 local bf16 values (la, lb) -> the fp32 sums y,
// the block's new scale sc (amax over the 8 lanes of the block) and the 16
// new codes (wa, wb).  REQ_BF16: requantize RNE_bf16(y), the bf16 partial a
// receiver keeps, instead of the fp32 sum y (the alternative reading of the
// hop).  nzero is -0.0f, passed in by the host.
//
// Every value is the one the scalar sequence gives, signed zeros included:
//  * the product RN(d * s_in) is fma(d, s_in, -0): adding -0 to the exact
//    product changes no value and no zero's sign, and as an fma there is no
//    separate multiply left for the compiler to contract into the add (a
//    packed multiply followed by an add was contracted, even with .rn);
//  * y = RN(l + p) with l widened exactly, i.e. RN(p + l);
//  * the quotient steps of markstein_div with -y formed exactly as y * -1
//    and r * -RN(1/s) in place of -r * RN(1/s) (the same product).
template <int FMT, bool REQ_BF16>
__device__ __forceinline__ void hop_block16(const uint2& ca, const uint2& cb, const uint4& la, const uint4& lb,
                                            float s_in, float nzero, uint32_t (&wa)[2], uint32_t (&wb)[2],
                                            float (&y)[16], float& sc) {
    float d[16];
    decode_fp8x4<FMT>(ca.x, d);
    decode_fp8x4<FMT>(ca.y, d + 4);
    decode_fp8x4<FMT>(cb.x, d + 8);
    decode_fp8x4<FMT>(cb.y, d + 12);
    const uint32_t lw[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
    const uint64_t s2 = f2_pack(s_in, s_in), z2 = f2_pack(nzero, nzero);
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float p0, p1;
        f2_unpack(f2_fma(f2_pack(d[2 * i], d[2 * i + 1]), s2, z2), p0, p1);
        y[2 * i] = add_bf16_f32((uint16_t)(lw[i] & 0xFFFFu), p0);
        y[2 * i + 1] = add_bf16_f32((uint16_t)(lw[i] >> 16), p1);
        if (REQ_BF16) {
            y[2 * i] = bf16_lo(pack_bf16x2(y[2 * i], 0.0f));
            y[2 * i + 1] = bf16_lo(pack_bf16x2(y[2 * i + 1], 0.0f));
        }
        a = max3(a, fabsf(y[2 * i]), fabsf(y[2 * i + 1]));
    }
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    sc = block_scale<FMT>(a);
    float q[16];
    if (sc >= 0x1p-58f) {
        // block_quotients<2, 16> in packed form
        const float yr = __frcp_rn(sc);
        const uint64_t yr2 = f2_pack(yr, yr), nyr2 = f2_pack(-yr, -yr), sc2 = f2_pack(sc, sc);
        const uint64_t m1 = f2_pack(-1.0f, -1.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint64_t y2 = f2_pack(y[2 * i], y[2 * i + 1]);
            const uint64_t ny2 = f2_mul(y2, m1);
            uint64_t q2 = f2_mul(y2, yr2);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint64_t r2 = f2_fma(q2, sc2, ny2);
                q2 = f2_fma(r2, nyr2, q2);
            }
            f2_unpack(q2, q[2 * i], q[2 * i + 1]);
        }
    } else {
        block_quotients<2, 16>(y, sc, q);      // s < 2^-58: the IEEE division
    }
    wa[0] = cvt_fp8x4<FMT>(q[0], q[1], q[2], q[3]);
    wa[1] = cvt_fp8x4<FMT>(q[4], q[5], q[6], q[7]);
    wb[0] = cvt_fp8x4<FMT>(q[8], q[9], q[10], q[11]);
    wb[1] = cvt_fp8x4<FMT>(q[12], q[13], q[14], q[15]);
}

// The lane's 16 sums as bf16 (RNE), at elements e0 .. e0+7 and e0+64 .. e0+71.
__device__ __forceinline__ void store_hop_bf16(uint16_t* out_bf16, size_t e0, const float (&y)[16], bool staged,
                                               bool in_range, long long avail) {
    uint32_t ha[4], hb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ha[i] = pack_bf16x2(y[2 * i], y[2 * i + 1]);
        hb[i] = pack_bf16x2(y[8 + 2 * i], y[8 + 2 * i + 1]);
    }
    if (staged) {
        st_stream(out_bf16 + e0, make_uint4(ha[0], ha[1], ha[2], ha[3]));
        st_stream(out_bf16 + e0 + 64, make_uint4(hb[0], hb[1], hb[2], hb[3]));
    } else if (in_range) {
        st_u16_tail(out_bf16 + e0, ha, 4, avail);
        st_u16_tail(out_bf16 + e0 + 64, hb, 4, avail - 64);
    }
}

// NST stages of kHopStageBytes each (2 for short hops, 3 otherwise; see
// launch_hop_kernel).
template <int FMT, bool REQ_BF16, int NST>
__global__ void __launch_bounds__(kHopThreads)
ring_hop_kernel(const __grid_constant__ HopGroup g) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * kHopStageBytes);
    const int64_t total_tiles = g.tile_start[g.count];
    const unsigned tid = threadIdx.x;
    const unsigned lane = tid & 31u, warp = tid >> 5;
    const unsigned j = lane & 7u, sub = lane >> 3;
    const unsigned bl = warp * 4 + sub;                    // block inside the tile

    auto hop_of = [&](int64_t t) {                         // CTA-uniform
        int h = 0;
        while (h + 1 < g.count && t >= g.tile_start[h + 1]) ++h;
        return h;
    };
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    // a tile is staged through shared memory when it lies entirely inside its hop's arrays
    auto staged_tile = [&](int64_t t, int h) { return (size_t)(t - g.tile_start[h] + 1) * kHopTile <= g.n[h]; };
    // arms stage s for a whole tile and copies the tile's local partial
    auto issue_local = [&](int64_t t, int h, int s) {   // thread 0 only
        const size_t lt = (size_t)(t - g.tile_start[h]);
        uint8_t* st = smem + (size_t)s * kHopStageBytes;
        mbar_arrive_expect_tx(&full[s], kHopStageBytes);
        bulk_g2s(st + kHopCodesBytes + kHopScaleBytes, g.local[h] + lt * kHopTile, kHopLocalBytes, &full[s]);
    };
    // the incoming codes and scales of the tile (the rest of the stage's bytes)
    auto issue_incoming = [&](int64_t t, int h, int s) {   // thread 0 only
        const size_t lt = (size_t)(t - g.tile_start[h]);
        uint8_t* st = smem + (size_t)s * kHopStageBytes;
        bulk_g2s(st, g.in_codes[h] + lt * kHopTile, kHopCodesBytes, &full[s]);
        bulk_g2s(st + kHopCodesBytes, g.in_scales[h] + lt * kHopTileBlocks, kHopScaleBytes, &full[s]);
    };
    // A hop's ragged last tile is not staged and can sit between staged tiles,
    // so each stage's barrier parity is tracked explicitly: bit s of `parity`
    // is the phase to wait for on stage s, flipped each time a staged tile of
    // that stage has been consumed.  `pending` (thread 0) marks stages with a
    // copy issued and not yet consumed.
    uint32_t parity = 0;
    uint32_t pending = 0;
    // the first tiles' local partials, before the predecessor grid has ended,
    // when the caller guarantees that it does not write them
    if (tid == 0 && g.local_ready)
        for (int s = 0; s < NST; ++s) {
            const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
            if (t < total_tiles) {
                const int h = hop_of(t);
                if (staged_tile(t, h)) {
                    issue_local(t, h, s);
                    pending |= 1u << s;
                }
            }
        }
    dependency_wait();
    allow_dependents();
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < NST; ++s) {
            const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
            if (t < total_tiles) {
                const int h = hop_of(t);
                if (staged_tile(t, h)) {
                    if (!g.local_ready) issue_local(t, h, s);
                    issue_incoming(t, h, s);
                    pending |= 1u << s;
                }
            }
        }

    int it = 0;
    bool failed = false;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
        const int s = it % NST;
        const int h = hop_of(t);
        const size_t n = g.n[h];
        const bool staged = staged_tile(t, h);
        const bool ok = staged ? mbar_wait(&full[s], (parity >> s) & 1u) : true;
        if (staged && ok) {
            parity ^= 1u << s;
            pending &= ~(1u << s);
        }
        const uint8_t* st = smem + (size_t)s * kHopStageBytes;
        const size_t nb = (n + 127) >> 7;
        const size_t b = (size_t)(t - g.tile_start[h]) * kHopTileBlocks + bl;
        const size_t e0 = (b << 7) + 8 * j;
        const long long avail = (long long)n - (long long)e0;     // valid elements from e0
        uint2 ca, cb;
        uint4 la, lb;
        float s_in;
        if (staged) {
            ca = *reinterpret_cast<const uint2*>(st + bl * 128 + j * 8);
            cb = *reinterpret_cast<const uint2*>(st + bl * 128 + 64 + j * 8);
            s_in = *reinterpret_cast<const float*>(st + kHopCodesBytes + bl * 4);
            const uint8_t* sl = st + kHopCodesBytes + kHopScaleBytes;
            la = *reinterpret_cast<const uint4*>(sl + bl * 256 + j * 16);
            lb = *reinterpret_cast<const uint4*>(sl + bl * 256 + 128 + j * 16);
        } else {
            ca = ld_u8x8_tail(g.in_codes[h] + e0, avail);
            cb = ld_u8x8_tail(g.in_codes[h] + e0 + 64, avail - 64);
            la = ld_bf16x8_tail(g.local[h] + e0, avail);
            lb = ld_bf16x8_tail(g.local[h] + e0 + 64, avail - 64);
            s_in = b < nb ? g.in_scales[h][b] : 0.0f;
        }

        uint32_t wa[2], wb[2];
        float y[16];
        float sc;
        hop_block16<FMT, REQ_BF16>(ca, cb, la, lb, s_in, g.nzero, wa, wb, y, sc);
        uint8_t* out_codes = g.out_codes[h];
        uint16_t* out_bf16 = g.out_bf16[h];
        if (staged) {
            st_stream(out_codes + e0, make_uint2(wa[0], wa[1]));
            st_stream(out_codes + e0 + 64, make_uint2(wb[0], wb[1]));
            if (j == 0) g.out_scales[h][b] = sc;
        } else if (b < nb) {
            st_u8_tail(out_codes + e0, wa, 2, avail);
            st_u8_tail(out_codes + e0 + 64, wb, 2, avail - 64);
            if (j == 0) g.out_scales[h][b] = sc;
        }
        if (out_bf16 != nullptr) store_hop_bf16(out_bf16, e0, y, staged, b < nb, avail);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid == 0) {
            const int64_t tn = t + (int64_t)NST * gridDim.x;     // next tile of stage s
            if (tn < total_tiles) {
                const int hn = hop_of(tn);
                if (staged_tile(tn, hn)) {
                    fence_proxy_async_smem();
                    issue_local(tn, hn, s);
                    issue_incoming(tn, hn, s);
                    pending |= 1u << s;
                }
            }
        }
    }
    if (failed && tid == 0) {
        // report, and let the copies still in flight land before the CTA's
        // shared memory is released
        raise_error(kErrCopyTimeout);
        for (int s = 0; s < NST; ++s)
            if (pending & (1u << s)) mbar_wait(&full[s], (parity >> s) & 1u);
    }
}

// The same hop for a group of two or more hops (all ranks' hops of one step
// of a simulated ring), with the per-tile bookkeeping hoisted: the hop index
// is carried from tile to tile (tiles only move forward), the staged-tile
// bound of each hop is precomputed on the host, and the stage index is a
// counter.  With several hops the single-hop kernel's per-tile search over
// the hop table costs about 14% more instructions, in a kernel that is bound
// by instruction issue at large sizes (8 hops of 16.8M elements: 108.5 us
// there, 94.9 us here; the 8-rank AllReduce of 256 MiB per rank 1.07 ->
// 1.03 ms, with each thread's shared-memory offsets fixed and the outputs
// addressed from the tile's base).  For one hop the carried index made the chain slower, so single
// hops keep ring_hop_kernel.
struct HopGroupMulti {
    const uint8_t* in_codes[kHopMaxGroup];
    const float* in_scales[kHopMaxGroup];
    const uint16_t* local[kHopMaxGroup];
    uint8_t* out_codes[kHopMaxGroup];
    float* out_scales[kHopMaxGroup];
    uint16_t* out_bf16[kHopMaxGroup];          // may be null per hop
    size_t n[kHopMaxGroup];
    int64_t tile_start[kHopMaxGroup + 1];
    int64_t staged_end[kHopMaxGroup];          // global tiles below this one are staged (per hop)
    int count;
    int local_ready;
    float nzero;
};

template <int FMT, bool REQ_BF16, int NST>
__global__ void __launch_bounds__(kHopThreads)
ring_hop_group_kernel(const __grid_constant__ HopGroupMulti g) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * kHopStageBytes);
    const int64_t total_tiles = g.tile_start[g.count];
    const unsigned tid = threadIdx.x;
    const unsigned lane = tid & 31u, warp = tid >> 5;
    const unsigned j = lane & 7u, sub = lane >> 3;
    const unsigned bl = warp * 4 + sub;                    // block inside the tile
    // this thread's fixed offsets: element (and code byte) inside the tile,
    // and the shared-memory bytes of its scale and local partial in a stage
    const unsigned e = bl * 128 + j * 8;
    const unsigned off_scale = kHopCodesBytes + bl * 4;
    const unsigned off_local = kHopCodesBytes + kHopScaleBytes + bl * 256 + j * 16;
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    auto hop_from = [&](int h, int64_t t) {                // CTA-uniform; t never decreases
        while (h + 1 < g.count && t >= g.tile_start[h + 1]) ++h;
        return h;
    };
    auto issue_local = [&](int64_t t, int h, int s) {   // thread 0 only
        const size_t lt = (size_t)(t - g.tile_start[h]);
        uint8_t* st = smem + (size_t)s * kHopStageBytes;
        mbar_arrive_expect_tx(&full[s], kHopStageBytes);
        bulk_g2s(st + kHopCodesBytes + kHopScaleBytes, g.local[h] + lt * kHopTile, kHopLocalBytes, &full[s]);
    };
    auto issue_incoming = [&](int64_t t, int h, int s) {   // thread 0 only
        const size_t lt = (size_t)(t - g.tile_start[h]);
        uint8_t* st = smem + (size_t)s * kHopStageBytes;
        bulk_g2s(st, g.in_codes[h] + lt * kHopTile, kHopCodesBytes, &full[s]);
        bulk_g2s(st + kHopCodesBytes, g.in_scales[h] + lt * kHopTileBlocks, kHopScaleBytes, &full[s]);
    };
    // parity / pending as in ring_hop_kernel
    uint32_t parity = 0, pending = 0;
    if (tid == 0 && g.local_ready) {
        int h = 0;
        for (int s = 0; s < NST; ++s) {
            const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
            if (t >= total_tiles) break;
            h = hop_from(h, t);
            if (t < g.staged_end[h]) {
                issue_local(t, h, s);
                pending |= 1u << s;
            }
        }
    }
    dependency_wait();
    allow_dependents();
    __syncthreads();
    int hp = 0;                                   // thread 0: hop of the next tile to request
    int64_t tp = blockIdx.x;                      // thread 0: the next tile to request
    if (tid == 0) {
        for (int s = 0; s < NST; ++s, tp += gridDim.x) {
            if (tp >= total_tiles) break;
            hp = hop_from(hp, tp);
            if (tp < g.staged_end[hp]) {
                if (!g.local_ready) issue_local(tp, hp, s);
                issue_incoming(tp, hp, s);
                pending |= 1u << s;
            }
        }
    }
    int s = 0;
    uint32_t stage_off = 0;
    int h = 0;
    bool failed = false;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        h = hop_from(h, t);
        const bool staged = t < g.staged_end[h];
        const bool ok = staged ? mbar_wait(&full[s], (parity >> s) & 1u) : true;
        if (staged && ok) {
            parity ^= 1u << s;
            pending &= ~(1u << s);
        }
        // the tile's first element, and the hop's outputs from there
        const size_t tile_e = (size_t)(t - g.tile_start[h]) * kHopTile;
        uint8_t* out_codes = g.out_codes[h] + tile_e;
        float* out_scales = g.out_scales[h] + tile_e / 128;
        uint16_t* out_bf16 = g.out_bf16[h];
        const uint8_t* st = smem + stage_off;
        uint2 ca, cb;
        uint4 la, lb;
        float s_in;
        long long avail = 0;
        bool in_range = true;
        if (staged) {
            ca = *reinterpret_cast<const uint2*>(st + e);
            cb = *reinterpret_cast<const uint2*>(st + e + 64);
            s_in = *reinterpret_cast<const float*>(st + off_scale);
            la = *reinterpret_cast<const uint4*>(st + off_local);
            lb = *reinterpret_cast<const uint4*>(st + off_local + 128);
        } else {
            // the hop's ragged last tile, from global memory
            const size_t n = g.n[h];
            const size_t e0 = tile_e + e;
            avail = (long long)n - (long long)e0;
            in_range = (e0 >> 7) < ((n + 127) >> 7);
            ca = ld_u8x8_tail(g.in_codes[h] + e0, avail);
            cb = ld_u8x8_tail(g.in_codes[h] + e0 + 64, avail - 64);
            la = ld_bf16x8_tail(g.local[h] + e0, avail);
            lb = ld_bf16x8_tail(g.local[h] + e0 + 64, avail - 64);
            s_in = in_range ? g.in_scales[h][e0 >> 7] : 0.0f;
        }
        uint32_t wa[2], wb[2];
        float y[16];
        float sc;
        hop_block16<FMT, REQ_BF16>(ca, cb, la, lb, s_in, g.nzero, wa, wb, y, sc);
        if (staged) {
            st_stream(out_codes + e, make_uint2(wa[0], wa[1]));
            st_stream(out_codes + e + 64, make_uint2(wb[0], wb[1]));
            if (j == 0) out_scales[bl] = sc;
        } else if (in_range) {
            st_u8_tail(out_codes + e, wa, 2, avail);
            st_u8_tail(out_codes + e + 64, wb, 2, avail - 64);
            if (j == 0) out_scales[bl] = sc;
        }
        if (out_bf16 != nullptr) store_hop_bf16(out_bf16 + tile_e, e, y, staged, in_range, avail);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid == 0 && tp < total_tiles) {           // the tile NST ahead, into stage s
            hp = hop_from(hp, tp);
            if (tp < g.staged_end[hp]) {
                fence_proxy_async_smem();
                issue_local(tp, hp, s);
                issue_incoming(tp, hp, s);
                pending |= 1u << s;
            }
        }
        tp += gridDim.x;
        if (s + 1 == NST) {
            s = 0;
            stage_off = 0;
        } else {
            ++s;
            stage_off += kHopStageBytes;
        }
    }
    if (failed && tid == 0) {
        raise_error(kErrCopyTimeout);
        for (int q = 0; q < NST; ++q)
            if (pending & (1u << q)) mbar_wait(&full[q], (parity >> q) & 1u);
    }
}

// Host checks of one hop (as documented for fp8q_ring_hop).
static fp8q_status_t check_hop(const fp8q_hop_t& hp) {
    if (hp.n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (hp.n == 0) return FP8Q_OK;
    if (!hp.in_codes || !hp.in_scales || !hp.local_bf16 || !hp.out_codes || !hp.out_scales) return FP8Q_ERR_NULL;
    if (!aligned16(hp.in_codes) || !aligned16(hp.in_scales) || !aligned16(hp.local_bf16) ||
        !aligned16(hp.out_codes) || !aligned16(hp.out_scales) || (hp.out_bf16 && !aligned16(hp.out_bf16)))
        return FP8Q_ERR_ALIGN;
    return FP8Q_OK;
}

// Byte ranges of a hop: reads 0..2, writes 3..5.
static void hop_ranges(const fp8q_hop_t& hp, const void* p[6], size_t sz[6]) {
    const size_t n = hp.n, nb = fp8q_num_scales(n);
    p[0] = hp.in_codes;  sz[0] = n;
    p[1] = hp.in_scales; sz[1] = 4 * nb;
    p[2] = hp.local_bf16; sz[2] = 2 * n;
    p[3] = hp.out_codes; sz[3] = n;
    p[4] = hp.out_scales; sz[4] = 4 * nb;
    p[5] = hp.out_bf16;  sz[5] = hp.out_bf16 ? 2 * n : 0;
}

template <int FMT, bool REQ, int NST>
static fp8q_status_t launch_hop_group_kernel_n(const HopGroupMulti& g, size_t tiles, cudaStream_t stream) {
    static KernelCache kc;
    constexpr size_t smem = (size_t)NST * kHopStageBytes + 8 * NST;
    int resident = 0;
    const fp8q_status_t st =
        prepare_kernel(kc, ring_hop_group_kernel<FMT, REQ, NST>, kHopThreads, smem, smem, &resident);
    if (st != FP8Q_OK) return st;
    return launch(ring_hop_group_kernel<FMT, REQ, NST>, grid_for(tiles, resident), kHopThreads, smem, stream, g);
}

// A short group (under 8 tiles per CTA of a full grid) runs 2 stages, a long
// one 3: the 8-rank AllReduce of the 8 x 13.1M bucket, whose hop groups are
// 3,200 tiles each, takes 119.0 us with 2 stages and 120.0 with 3.
template <int FMT, bool REQ>
static fp8q_status_t launch_hop_group_kernel(const HopGroupMulti& g, size_t tiles, cudaStream_t stream) {
    if (tiles < (size_t)8 * 4 * (size_t)sm_count()) return launch_hop_group_kernel_n<FMT, REQ, 2>(g, tiles, stream);
    return launch_hop_group_kernel_n<FMT, REQ, 3>(g, tiles, stream);
}

template <int FMT, bool REQ, int NST>
static fp8q_status_t launch_hop_kernel_n(const HopGroup& g, size_t tiles, cudaStream_t stream) {
    static KernelCache kc;
    constexpr size_t smem = (size_t)NST * kHopStageBytes + 8 * NST;
    int resident = 0;
    const fp8q_status_t st = prepare_kernel(kc, ring_hop_kernel<FMT, REQ, NST>, kHopThreads, smem, smem, &resident);
    if (st != FP8Q_OK) return st;
    return launch(ring_hop_kernel<FMT, REQ, NST>, grid_for(tiles, resident), kHopThreads, smem, stream, g);
}

// Single hops run 3 stages at every size.  With scalar arithmetic a short hop
// (under 8 tiles per CTA of a full grid, e.g. the 13.1M-element shard: 3,200
// tiles over 608 CTAs) was faster with 2 (the 7-hop chain at 13.1M: 75.0
// against 77.0 us); with the packed arithmetic of hop_block16 the third stage
// pays there too (the chain 75.7 -> 73.3 us, and 2 stages lose 5 us at
// 64 MiB per hop).
template <int FMT, bool REQ>
static fp8q_status_t launch_hop_kernel(const HopGroup& g, size_t tiles, cudaStream_t stream) {
    return launch_hop_kernel_n<FMT, REQ, 3>(g, tiles, stream);
}

static fp8q_status_t launch_hops(const fp8q_hop_t* hops, int count, fp8q_format_t fmt, cudaStream_t stream,
                                 bool requant_bf16 = false, unsigned flags = 0) {
    if (flags & ~FP8Q_HOP_LOCAL_READY) return FP8Q_ERR_FLAGS;
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (!hops) return FP8Q_ERR_NULL;
    if (count < 1 || count > kHopMaxGroup) return FP8Q_ERR_SIZE;
    for (int i = 0; i < count; ++i) {
        const fp8q_status_t st = check_hop(hops[i]);
        if (st != FP8Q_OK) return st;
    }
    // no output may overlap another output or any input of the group; the one
    // exception is a hop's bf16 output written in place over its own local partial
    for (int i = 0; i < count; ++i) {
        if (hops[i].n == 0) continue;
        const void* pi[6];
        size_t si[6];
        hop_ranges(hops[i], pi, si);
        for (int j = 0; j < count; ++j) {
            if (hops[j].n == 0) continue;
            const void* pj[6];
            size_t sj[6];
            hop_ranges(hops[j], pj, sj);
            for (int a = 3; a < 6; ++a)
                for (int b = 0; b < 6; ++b) {
                    if (i == j && a == b) continue;
                    if (i == j && a == 5 && b == 2 && pi[5] == pj[2]) continue;
                    if (overlaps(pi[a], si[a], pj[b], sj[b])) return FP8Q_ERR_ALIAS;
                }
        }
    }
    int nonempty = 0;
    for (int i = 0; i < count; ++i) nonempty += hops[i].n != 0;
    if (nonempty == 0) return FP8Q_OK;
    if (nonempty >= 2) {
        HopGroupMulti g;
        int used = 0;
        int64_t start = 0;
        for (int i = 0; i < count; ++i) {
            const fp8q_hop_t& hp = hops[i];
            if (hp.n == 0) continue;
            g.in_codes[used] = hp.in_codes;
            g.in_scales[used] = hp.in_scales;
            g.local[used] = static_cast<const uint16_t*>(hp.local_bf16);
            g.out_codes[used] = hp.out_codes;
            g.out_scales[used] = hp.out_scales;
            g.out_bf16[used] = static_cast<uint16_t*>(hp.out_bf16);
            g.n[used] = hp.n;
            g.tile_start[used] = start;
            g.staged_end[used] = start + (int64_t)(hp.n / kHopTile);
            start += (int64_t)((hp.n + kHopTile - 1) / kHopTile);
            ++used;
        }
        g.tile_start[used] = start;
        g.count = used;
        g.local_ready = (flags & FP8Q_HOP_LOCAL_READY) ? 1 : 0;
        g.nzero = -0.0f;
        const size_t tiles = (size_t)start;
        if (fmt == FP8Q_E4M3)
            return requant_bf16 ? launch_hop_group_kernel<kE4M3, true>(g, tiles, stream)
                                : launch_hop_group_kernel<kE4M3, false>(g, tiles, stream);
        return requant_bf16 ? launch_hop_group_kernel<kE5M2, true>(g, tiles, stream)
                            : launch_hop_group_kernel<kE5M2, false>(g, tiles, stream);
    }
    HopGroup g;
    int used = 0;
    int64_t start = 0;
    for (int i = 0; i < count; ++i) {
        const fp8q_hop_t& hp = hops[i];
        if (hp.n == 0) continue;
        g.in_codes[used] = hp.in_codes;
        g.in_scales[used] = hp.in_scales;
        g.local[used] = static_cast<const uint16_t*>(hp.local_bf16);
        g.out_codes[used] = hp.out_codes;
        g.out_scales[used] = hp.out_scales;
        g.out_bf16[used] = static_cast<uint16_t*>(hp.out_bf16);
        g.n[used] = hp.n;
        g.tile_start[used] = start;
        start += (int64_t)((hp.n + kHopTile - 1) / kHopTile);
        ++used;
    }
    if (used == 0) return FP8Q_OK;
    g.tile_start[used] = start;
    g.count = used;
    g.local_ready = (flags & FP8Q_HOP_LOCAL_READY) ? 1 : 0;
        g.nzero = -0.0f;
    const size_t tiles = (size_t)start;
    if (fmt == FP8Q_E4M3)
        return requant_bf16 ? launch_hop_kernel<kE4M3, true>(g, tiles, stream)
                            : launch_hop_kernel<kE4M3, false>(g, tiles, stream);
    return requant_bf16 ? launch_hop_kernel<kE5M2, true>(g, tiles, stream)
                        : launch_hop_kernel<kE5M2, false>(g, tiles, stream);
}

}  // namespace fp8q

namespace fp8q {
unsigned unit_errors_ring_hop(bool clear) { return read_unit_errors(clear); }
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status_t fp8q_ring_hop(const uint8_t* in_codes, const float* in_scales, const void* local_bf16,
                                       size_t n, fp8q_format_t fmt, uint8_t* out_codes, float* out_scales,
                                       void* out_bf16, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_ring_hop");
    const fp8q_hop_t hp = {in_codes, in_scales, local_bf16, n, out_codes, out_scales, out_bf16};
    return launch_hops(&hp, 1, fmt, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8q_status_t fp8q_ring_hop_group(const fp8q_hop_t* hops, int count, fp8q_format_t fmt,
                                             fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_ring_hop_group");
    return launch_hops(hops, count, fmt, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8q_status_t fp8q_ring_hop_group_ex(const fp8q_hop_t* hops, int count, fp8q_format_t fmt,
                                                unsigned int flags, fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_ring_hop_group_ex");
    return launch_hops(hops, count, fmt, reinterpret_cast<cudaStream_t>(stream), false, flags);
}

extern "C" fp8q_status_t fp8q_ring_hop_bf16_requant(const uint8_t* in_codes, const float* in_scales,
                                                    const void* local_bf16, size_t n, fp8q_format_t fmt,
                                                    uint8_t* out_codes, float* out_scales, void* out_bf16,
                                                    fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_ring_hop_bf16_requant");
    const fp8q_hop_t hp = {in_codes, in_scales, local_bf16, n, out_codes, out_scales, out_bf16};
    return launch_hops(&hp, 1, fmt, reinterpret_cast<cudaStream_t>(stream), true);
}
