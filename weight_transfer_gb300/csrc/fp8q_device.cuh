// Device-side building blocks of the fp8q kernels (sm_103a).
//
// Everything here is exact or correctly rounded binary32 arithmetic; the
// library is compiled without fast-math and with -fmad=false, and every
// rounding step that the codec's definition fixes is spelled with an
// explicit *_rn intrinsic so the compiler can neither fuse nor reorder it.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp8q {

constexpr int kE4M3 = 0;
constexpr int kE5M2 = 1;

// Largest finite magnitude of each OFP8 format (E4M3: 1.75 * 2^8,
// E5M2: 1.75 * 2^15); the blockwise scale is amax divided by it.
// `inverse` is RN(1 / value): 1.75 has the binary32 reciprocal
// 0x1.24924ap-1 (1/1.75 = 0.571428..., rounded to nearest).
template <int FMT> struct FmtMax;
template <> struct FmtMax<kE4M3> {
    static constexpr float value = 448.0f;
    static constexpr float inverse = 0x1.24924ap-9f;
};
template <> struct FmtMax<kE5M2> {
    static constexpr float value = 57344.0f;
    static constexpr float inverse = 0x1.24924ap-16f;
};

// ---------------------------------------------------------------- bf16 ----
// A bf16 is the upper half of a binary32, so widening is a shift.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Two binary32 -> packed bf16x2 with round-to-nearest-even (cvt.rn.bf16x2.f32:
// the first operand lands in the upper half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ----------------------------------------------------------------- FP8 ----
// Two binary32 -> two FP8 codes, round-to-nearest-even, saturating to the
// largest finite magnitude (the .satfinite form of the native conversion).
// Returns a 16-bit pair with `lo` in bits 0..7 and `hi` in bits 8..15.
template <int FMT> __device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t cvt_fp8x2<kE4M3>(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
template <> __device__ __forceinline__ uint32_t cvt_fp8x2<kE5M2>(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four binary32 -> four codes in one 32-bit word (byte i = element i).
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x4(float a, float b, float c, float d) {
    return __byte_perm(cvt_fp8x2<FMT>(a, b), cvt_fp8x2<FMT>(c, d), 0x5410u);
}

// Two codes (bytes 0 and 1 of `two`) -> two binary32.  Both formats embed
// exactly in f16, so the decode is exact.
template <int FMT> __device__ __forceinline__ float2 decode_fp8x2(uint32_t two);
template <> __device__ __forceinline__ float2 decode_fp8x2<kE4M3>(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}
template <> __device__ __forceinline__ float2 decode_fp8x2<kE5M2>(uint32_t two) {
    // an E5M2 code is the upper byte of the f16 with the same value
    uint32_t h2 = __byte_perm(two, 0u, 0x1404u);
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

// Four codes of a 32-bit word -> four binary32.
template <int FMT>
__device__ __forceinline__ void decode_fp8x4(uint32_t w, float* f) {
    float2 a = decode_fp8x2<FMT>(w & 0xFFFFu);
    float2 b = decode_fp8x2<FMT>(w >> 16);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// -------------------------------------------- programmatic dependent launch ----
// Every kernel of the library is launched so that it may be dispatched while
// the previous kernel on its stream is still finishing.  A kernel calls
// dependency_wait() before its first global-memory access: the wait returns
// once the preceding grid has completed and its writes are visible (at once
// when the launch had no such overlap).  allow_dependents() right after it
// lets the next launch's blocks take SM slots as this grid's blocks retire;
// they only fit as this grid drains, so the overlap covers launch, block
// dispatch and the shared-memory prologue, never data.
__device__ __forceinline__ void dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------- memory access ----
// Streaming 16-byte load through the read-only path without L1 allocation:
// every byte is read once.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Same, through the coherent path: for data that the kernel may also write
// (the in-place ring hop updates the local partial it reads).
__device__ __forceinline__ uint4 ld_once(const void* p) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ float ld_stream_f32(const float* p) {
    float r;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(r) : "l"(p));
    return r;
}

// Streaming (evict-first) stores: outputs are written once and not re-read.
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream(void* p, const uint2& v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Guarded loads / stores for the one ragged unit at the end of an array.
// `avail` = number of valid elements from the unit's start (may be <= 0).
__device__ __forceinline__ uint4 ld_bf16x8_tail(const uint16_t* p, long long avail) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int i = 0; i < 8; ++i)
        if (i < avail) w[i >> 1] |= (uint32_t)p[i] << ((i & 1) * 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 ld_u8x16_tail(const uint8_t* p, long long avail) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int i = 0; i < 16; ++i)
        if (i < avail) w[i >> 2] |= (uint32_t)p[i] << ((i & 3) * 8);
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint2 ld_u8x8_tail(const uint8_t* p, long long avail) {
    uint32_t w[2] = {0u, 0u};
    for (int i = 0; i < 8; ++i)
        if (i < avail) w[i >> 2] |= (uint32_t)p[i] << ((i & 3) * 8);
    return make_uint2(w[0], w[1]);
}
__device__ __forceinline__ void st_u8_tail(uint8_t* p, const uint32_t* w, int nwords, long long avail) {
    for (int i = 0; i < nwords * 4; ++i)
        if (i < avail) p[i] = (uint8_t)(w[i >> 2] >> ((i & 3) * 8));
}
__device__ __forceinline__ void st_u16_tail(uint16_t* p, const uint32_t* w, int nwords, long long avail) {
    for (int i = 0; i < nwords * 2; ++i)
        if (i < avail) p[i] = (uint16_t)(w[i >> 1] >> ((i & 1) * 16));
}
__device__ __forceinline__ void st_f32_tail(float* p, const float* f, int count, long long avail) {
    for (int i = 0; i < count; ++i)
        if (i < avail) p[i] = f[i];
}

// ------------------------------------------- bulk copies (TMA) to smem ----
// The kernels stage their input tiles in shared memory with cp.async.bulk
// (1D) or cp.async.bulk.tensor (2D tensor map).  Completion is tracked by
// one mbarrier per stage ("transaction bytes"): the issuing thread arms the
// barrier with the byte count, the copy engine counts the bytes down, and
// the readers wait on the barrier's phase parity.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes freshly initialised barriers visible to the copy engine.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this CTA's earlier shared-memory accesses before later bulk copies
// into the same bytes (generic proxy -> async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wall-clock bound of every wait on a copy: a copy that has not landed after
// this long will never land, and the kernel reports it instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Waits until phase `parity` of the barrier has completed; false if that did
// not happen within `limit_ns` (kWaitLimitNs for every kernel of the library;
// the bounded-wait self-test passes a shorter limit).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i)
            if (mbar_test(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// 1D bulk copy global -> shared; both addresses 16-byte aligned, bytes a
// multiple of 16.  Completes `bytes` transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(smem_dst)),
                 "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// 2D tiled bulk copy of the box at (x, y) of a tensor map; x * element size
// must be a multiple of 16 bytes, out-of-range elements read as zero.
__device__ __forceinline__ void tma_2d_g2s(void* smem_dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Device-side error bits (see fp8q_device_errors).  Each translation unit
// has its own word; the host ORs them together.
constexpr unsigned kErrCopyTimeout = 1u;

static __device__ unsigned int g_unit_errors;

__device__ __forceinline__ void raise_error(unsigned bits) { atomicOr(&g_unit_errors, bits); }

// Host side: this unit's error bits (the caller has synchronized the device).
static inline unsigned read_unit_errors(bool clear) {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_unit_errors, sizeof v) != cudaSuccess) return ~0u;
    if (clear && v) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_unit_errors, &z, sizeof z);
    }
    return v;
}

// --------------------------------------------------------------- scale ----
// RN(x / d) by Markstein's correction step from y = RN(1/d):
//     q0 = RN(x*y);  r = RN(q0*d - x) (fma);  q = RN(q0 - r*y) (fma)
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990; "IA-64 and Elementary
// Functions", 2000).  The residual is formed negated, q0*d - x instead of
// x - q0*d: both roundings are sign-symmetric so the result is the same for
// every x != 0, and x = -0 then yields -0 (the plain form gives +0).
//
//  * One step is exact for bf16 dividends: it equals RN(x/d) for all 2^30
//    pairs of a bf16 significand and a binary32 significand at unit scale
//    (exhaustive check in tests/fastdiv/check.c).
//  * Two steps are exact for binary32 dividends: one step leaves q within
//    half an ulp plus a 2^-46-relative term of x/d, i.e. faithful, and
//    Markstein's theorem (y = RN(1/d), q faithful => the next step gives
//    RN(x/d)) covers the second.
//
// Every operation commutes with power-of-two scaling of x and d while all
// intermediates stay normal binary32, which extends the unit-scale result to
// all exponents for which x, d, y, q0 and a non-zero r are normal.  r is a
// non-zero multiple of 2^(e_x - 47) (x has a 24-bit significand, q0*d a
// 48-bit one), so |x| >= 2^-78 keeps it normal.
template <int STEPS>
__device__ __forceinline__ float markstein_div(float x, float d, float y) {
    float q = __fmul_rn(x, y);
#pragma unroll
    for (int c = 0; c < STEPS; ++c) {
        const float r = __fmaf_rn(q, d, -x);
        q = __fmaf_rn(-r, y, q);
    }
    return q;
}

// The block scale s = RN(amax / Fmax), Fmax = 1.75 * 2^8 (e4m3) or
// 1.75 * 2^15 (e5m2), by one Markstein step from the constant RN(1 / Fmax).
// amax is a bf16 value in the quantizers and a full binary32 value in the
// ring hop (the amax of its fp32 sums).  With the divisor fixed, one step is
// exact for every binary32 dividend: tests/fastdiv/check.c ("scale") checks
// all 2^23 significands in ten binades from 2^-78 to 2^127 for both maxima,
// and the sequence commutes with the power-of-two scaling of amax between
// them (see markstein_div).  amax < 2^-78 takes the IEEE division.
template <int FMT>
__device__ __forceinline__ float block_scale(float amax) {
    constexpr float F = FmtMax<FMT>::value;
    return amax >= 0x1p-78f ? markstein_div<1>(amax, F, FmtMax<FMT>::inverse) : __fdiv_rn(amax, F);
}

// RN(x_i / s) for all elements of one block, without a per-element division:
// y = RN(1/s) once (rcp.rn, correctly rounded), then markstein_div with
// STEPS = 1 for bf16 dividends and STEPS = 2 for binary32 dividends.
//
// For every element whose code can be non-zero (|x/s| >= 2^-20) the
// conditions of markstein_div hold as soon as s >= 2^-58 (then |x| >= 2^-78).
// Elements with |x/s| < 2^-20 round to a signed-zero code either way (the
// result stays far below the smallest FP8 subnormal, 2^-16, and keeps the
// sign of x).  Blocks with s < 2^-58 (amax < 448 * 2^-58 for e4m3) use the
// IEEE division; s == 0 only for an all-zero block, whose signed zeros pass
// through unchanged.
template <int STEPS, int N>
__device__ __forceinline__ void block_quotients(const float* x, float s, float* q) {
    if (s >= 0x1p-58f) {
        const float y = __frcp_rn(s);
#pragma unroll
        for (int i = 0; i < N; ++i) q[i] = markstein_div<STEPS>(x[i], s, y);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) q[i] = s == 0.0f ? x[i] : __fdiv_rn(x[i], s);
    }
}

}  // namespace fp8q
