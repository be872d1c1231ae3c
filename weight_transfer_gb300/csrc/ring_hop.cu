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
// Work split: 8 lanes own one 128-element block; lane j holds elements
// [8j, 8j+8) and [64+8j, 64+8j+8) (two 16-byte loads of the local partial,
// two 8-byte loads of codes), so every load instruction of a warp reads whole
// 128-byte (bf16) or 64-byte (codes) half-blocks.  The amax is a 3-step
// xor-shuffle among the 8 lanes; a warp covers 4 blocks per step.  The
// quotients y / s use the per-block reciprocal with two Markstein
// corrections (exact for binary32 dividends, see block_quotients).
#include "fp8q_device.cuh"
#include "fp8q_host.cuh"

namespace fp8q {

constexpr int kHopThreads = 256;

template <int FMT, bool OUT_BF16>
__global__ void __launch_bounds__(kHopThreads)
ring_hop_kernel(const uint8_t* __restrict__ in_codes, const float* __restrict__ in_scales,
                const uint16_t* local, size_t n, uint8_t* __restrict__ out_codes,
                float* __restrict__ out_scales, uint16_t* out_bf16) {
    const size_t nb = (n + 127) >> 7;
    const size_t nfull = n >> 7;
    const unsigned lane = threadIdx.x & 31u;
    const unsigned j = lane & 7u;
    const unsigned sub = lane >> 3;
    const size_t warp = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t base = warp; 4 * base < nb; base += nwarps) {    // warp-uniform bound
        const size_t b = 4 * base + sub;
        const size_t e0 = (b << 7) + 8 * j;
        const long long avail = (long long)n - (long long)e0;      // valid elements from e0
        uint2 ca = make_uint2(0u, 0u), cb = ca;
        uint4 la = make_uint4(0u, 0u, 0u, 0u), lb = la;
        float s_in = 0.0f;
        if (b < nfull) {
            ca = ld_stream8(in_codes + e0);
            cb = ld_stream8(in_codes + e0 + 64);
            la = ld_once(local + e0);
            lb = ld_once(local + e0 + 64);
        } else if (b < nb) {
            ca = ld_u8x8_tail(in_codes + e0, avail);
            cb = ld_u8x8_tail(in_codes + e0 + 64, avail - 64);
            la = ld_bf16x8_tail(local + e0, avail);
            lb = ld_bf16x8_tail(local + e0 + 64, avail - 64);
        }
        if (b < nb) s_in = ld_stream_f32(in_scales + b);

        float d[16], lf[16], y[16];
        decode_fp8x4<FMT>(ca.x, d);
        decode_fp8x4<FMT>(ca.y, d + 4);
        decode_fp8x4<FMT>(cb.x, d + 8);
        decode_fp8x4<FMT>(cb.y, d + 12);
        unpack8(la, *reinterpret_cast<float(*)[8]>(lf));
        unpack8(lb, *reinterpret_cast<float(*)[8]>(lf + 8));
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            y[i] = __fadd_rn(__fmul_rn(d[i], s_in), lf[i]);
            a = fmaxf(a, fabsf(y[i]));
        }
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        const float s = block_scale<FMT>(a);
        float q[16];
        block_quotients<2, 16>(y, s, q);
        uint32_t wa[2] = {cvt_fp8x4<FMT>(q[0], q[1], q[2], q[3]), cvt_fp8x4<FMT>(q[4], q[5], q[6], q[7])};
        uint32_t wb[2] = {cvt_fp8x4<FMT>(q[8], q[9], q[10], q[11]), cvt_fp8x4<FMT>(q[12], q[13], q[14], q[15])};
        if (b < nfull) {
            st_stream(out_codes + e0, make_uint2(wa[0], wa[1]));
            st_stream(out_codes + e0 + 64, make_uint2(wb[0], wb[1]));
        } else if (b < nb) {
            st_u8_tail(out_codes + e0, wa, 2, avail);
            st_u8_tail(out_codes + e0 + 64, wb, 2, avail - 64);
        }
        if (b < nb && j == 0) out_scales[b] = s;
        if (OUT_BF16) {
            uint32_t ha[4], hb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ha[i] = pack_bf16x2(y[2 * i], y[2 * i + 1]);
                hb[i] = pack_bf16x2(y[8 + 2 * i], y[8 + 2 * i + 1]);
            }
            if (b < nfull) {
                st_stream(out_bf16 + e0, make_uint4(ha[0], ha[1], ha[2], ha[3]));
                st_stream(out_bf16 + e0 + 64, make_uint4(hb[0], hb[1], hb[2], hb[3]));
            } else if (b < nb) {
                st_u16_tail(out_bf16 + e0, ha, 4, avail);
                st_u16_tail(out_bf16 + e0 + 64, hb, 4, avail - 64);
            }
        }
    }
}

template <int FMT, bool B>
static fp8q_status_t launch_hop_t(const uint8_t* ic, const float* is, const uint16_t* loc, size_t n, uint8_t* oc,
                                  float* os, uint16_t* ob, cudaStream_t s) {
    static int resident = resident_blocks(ring_hop_kernel<FMT, B>, kHopThreads);
    const size_t blocks_per_cta = (kHopThreads / 32) * 4;
    const unsigned grid = grid_for(((n + 127) / 128 + blocks_per_cta - 1) / blocks_per_cta, resident);
    ring_hop_kernel<FMT, B><<<grid, kHopThreads, 0, s>>>(ic, is, loc, n, oc, os, ob);
    return launch_status();
}

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status_t fp8q_ring_hop(const uint8_t* in_codes, const float* in_scales, const void* local_bf16,
                                       size_t n, fp8q_format_t fmt, uint8_t* out_codes, float* out_scales,
                                       void* out_bf16, fp8q_stream_t stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) return FP8Q_OK;
    if (!in_codes || !in_scales || !local_bf16 || !out_codes || !out_scales) return FP8Q_ERR_NULL;
    if (!aligned16(in_codes) || !aligned16(in_scales) || !aligned16(local_bf16) || !aligned16(out_codes) ||
        !aligned16(out_scales) || (out_bf16 && !aligned16(out_bf16)))
        return FP8Q_ERR_ALIGN;
    const size_t nb = fp8q_num_scales(n);
    const void* ins[3] = {in_codes, in_scales, local_bf16};
    const size_t in_sz[3] = {n, 4 * nb, 2 * n};
    void* outs[3] = {out_codes, out_scales, out_bf16};
    const size_t out_sz[3] = {n, 4 * nb, 2 * n};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 3; ++i) {
            if (o == 2 && i == 2 && outs[2] == ins[2]) continue;   // in-place update of the local partial
            if (overlaps(outs[o], out_sz[o], ins[i], in_sz[i])) return FP8Q_ERR_ALIAS;
        }
        for (int p = o + 1; p < 3; ++p)
            if (overlaps(outs[o], out_sz[o], outs[p], out_sz[p])) return FP8Q_ERR_ALIAS;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t* loc = static_cast<const uint16_t*>(local_bf16);
    uint16_t* ob = static_cast<uint16_t*>(out_bf16);
    if (fmt == FP8Q_E4M3)
        return ob ? launch_hop_t<kE4M3, true>(in_codes, in_scales, loc, n, out_codes, out_scales, ob, s)
                  : launch_hop_t<kE4M3, false>(in_codes, in_scales, loc, n, out_codes, out_scales, ob, s);
    return ob ? launch_hop_t<kE5M2, true>(in_codes, in_scales, loc, n, out_codes, out_scales, ob, s)
              : launch_hop_t<kE5M2, false>(in_codes, in_scales, loc, n, out_codes, out_scales, ob, s);
}
