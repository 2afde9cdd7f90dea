// ep_fp8.cuh -- the e4m3 codec shared by the low-latency send and the FP8
// normal-mode rows: per 128 channels, scale = amax / 448 (IEEE fp32 division),
// code = cvt.rn.satfinite.e4m3 of x / scale (the IEEE fp32 quotient); a zero
// scale keeps only the sign of x.
#pragma once
#include <cuda_fp8.h>

#include "ep_internal.cuh"

namespace ep {

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    // low byte <- a, high byte <- b
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Sixteen consecutive bf16 channels (two 16-byte vectors) to floats.
__device__ __forceinline__ void bf16x16_to_f32(const int4& p0, const int4& p1, float* v) {
    const uint32_t uu[8] = {(uint32_t)p0.x, (uint32_t)p0.y, (uint32_t)p0.z, (uint32_t)p0.w,
                            (uint32_t)p1.x, (uint32_t)p1.y, (uint32_t)p1.z, (uint32_t)p1.w};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        v[2 * u] = __uint_as_float(uu[u] << 16);
        v[2 * u + 1] = __uint_as_float(uu[u] & 0xffff0000u);
    }
}

// x / scale as the IEEE (round-to-nearest) fp32 quotient, from y = RN(1/scale)
// computed once per block: q0 = RN(x*y), the exact residual r = q0*scale - x
// by one fma, then q = RN(q0 - r*y).  This is Markstein's correction step
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990): with y correctly rounded and
// q0 within an ulp of the quotient, q is the correctly rounded quotient as
// long as nothing underflows.  Over every pair of a bf16 x and a bf16 block
// maximum with |x| <= amax and scale >= 2^-100, the e4m3 code of q equals the
// code of the IEEE quotient (checked exhaustively); q can differ from it only
// below 2^-10, where both codes are +-0 with x's sign.  The residual's sign
// convention keeps that sign for x = -0.
__device__ __forceinline__ float div_by_scale(float x, float scale, float y) {
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(q0, scale, -x);
    return __fmaf_rn(-r, y, q0);
}

// Scales below this (block maxima under ~3.5e-28) and non-finite ones divide
// each element with __fdiv_rn instead.
constexpr float kRcpScaleMin = 0x1p-100f;
constexpr float kRcpScaleMax = 3.0e38f;

// Quantises the 16 channels a lane holds; the 8 lanes of an aligned lane group
// hold one 128-channel block and share its scale.  Every lane of the warp must
// call it (shuffles); lanes without data pass zeros.
__device__ __forceinline__ int4 quantize16(const float* v, float* scale_out) {
    float amax = 0.0f;
#pragma unroll
    for (int u = 0; u < 16; ++u) amax = fmaxf(amax, fabsf(v[u]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.0f);
    uint32_t w4[4];
    if (scale == 0.0f) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t c = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) c |= ((__float_as_uint(v[4 * u + b]) >> 31) ? 0x80u : 0u) << (8 * b);
            w4[u] = c;
        }
    } else if (scale >= kRcpScaleMin && scale <= kRcpScaleMax) {
        const float y = __frcp_rn(scale);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t lo = e4m3x2(div_by_scale(v[4 * u], scale, y), div_by_scale(v[4 * u + 1], scale, y));
            const uint32_t hi = e4m3x2(div_by_scale(v[4 * u + 2], scale, y), div_by_scale(v[4 * u + 3], scale, y));
            w4[u] = (lo & 0xffffu) | (hi << 16);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t lo = e4m3x2(__fdiv_rn(v[4 * u], scale), __fdiv_rn(v[4 * u + 1], scale));
            const uint32_t hi = e4m3x2(__fdiv_rn(v[4 * u + 2], scale), __fdiv_rn(v[4 * u + 3], scale));
            w4[u] = (lo & 0xffffu) | (hi << 16);
        }
    }
    *scale_out = scale;
    return make_int4((int)w4[0], (int)w4[1], (int)w4[2], (int)w4[3]);
}

}  // namespace ep
