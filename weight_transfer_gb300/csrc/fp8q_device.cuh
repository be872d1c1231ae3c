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
template <int FMT> struct FmtMax;
template <> struct FmtMax<kE4M3> { static constexpr float value = 448.0f; };
template <> struct FmtMax<kE5M2> { static constexpr float value = 57344.0f; };

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
    return cvt_fp8x2<FMT>(a, b) | (cvt_fp8x2<FMT>(c, d) << 16);
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

// --------------------------------------------------------------- scale ----
// The block scale s = RN(amax / Fmax): a true IEEE binary32 division (the
// compiler's correctly rounded div.rn.f32), once per block.
template <int FMT>
__device__ __forceinline__ float block_scale(float amax) {
    return __fdiv_rn(amax, FmtMax<FMT>::value);
}

// q = x / s for a block scale s; s == 0 only for an all-zero block, whose
// elements are signed zeros and are passed through unchanged.
__device__ __forceinline__ float scaled_quotient(float x, float s) {
    return s == 0.0f ? x : __fdiv_rn(x, s);
}

__device__ __forceinline__ float with_sign_of(float mag, float sgn) {
    return __uint_as_float((__float_as_uint(mag) & 0x7FFFFFFFu) | (__float_as_uint(sgn) & 0x80000000u));
}

// RN(x_i / s) for all elements of one block, without a per-element division.
//
// With y = RN(1/s) computed once (rcp.rn, correctly rounded), each quotient
// is q0 = RN(x*y) followed by CORRECTIONS Markstein steps
//     r = RN(x - q*s)  (fma),   q = RN(q + r*y)  (fma)
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990; "IA-64 and Elementary
// Functions", 2000).  The sign is taken from x so that x = -0 stays -0.
//
//  * CORRECTIONS = 1 is used for bf16 dividends.  It equals RN(x/s) for all
//    2^30 pairs of a bf16 significand and a binary32 significand at unit
//    scale (exhaustive check in tests/fastdiv/check.c).
//  * CORRECTIONS = 2 is used for binary32 dividends.  One step leaves q
//    within half an ulp plus a 2^-46-relative term of x/s, i.e. faithful;
//    Markstein's theorem (y = RN(1/s), q faithful => RN(q + r*y) = RN(x/s))
//    makes the second step exact.
//
// Every operation commutes with power-of-two scaling of x and s while all
// intermediates are normal binary32.  That holds for every element whose
// code can be non-zero (|x/s| >= 2^-20) as soon as s >= 2^-58: then
// |x| >= 2^-78 and the residual r, a non-zero multiple of 2^(e_x - 47), is
// at least 2^-125.  Elements with |x/s| < 2^-20 round to a signed-zero code
// either way (the result stays far below the smallest FP8 subnormal, 2^-16).
// Blocks with s < 2^-58 (amax < 448 * 2^-58 for e4m3) take the IEEE
// division instead.
template <int CORRECTIONS, int N>
__device__ __forceinline__ void block_quotients(const float* x, float s, float* q) {
    if (s >= 0x1p-58f) {
        const float y = __frcp_rn(s);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float t = __fmul_rn(x[i], y);
#pragma unroll
            for (int c = 0; c < CORRECTIONS; ++c) {
                const float r = __fmaf_rn(-t, s, x[i]);
                t = __fmaf_rn(r, y, t);
            }
            q[i] = with_sign_of(t, x[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) q[i] = scaled_quotient(x[i], s);
    }
}

}  // namespace fp8q
