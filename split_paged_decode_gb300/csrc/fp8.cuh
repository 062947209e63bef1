// fp8.cuh -- OCP FP8 E4M3 conversions for the fp8-cache kernels (sm_103a).
//
// A bf16 or fp32 quantity x that meets an E4M3 cache in a kind::f8f6f4 MMA is
// carried as two E4M3 operands whose sum is 16 x up to the rounding of the
// second (about 2^-8 of |x|, as bf16 gives), so that one fp32 accumulator
// receives 16 x: Q as h = e4m3(x) and l = e4m3(16 (x - h)), used as 16 h and
// l (the caller keeps |x| <= 28 so that 16 h <= 448, the largest E4M3
// value); P <= 16 as h = e4m3(16 P) and l = e4m3(16 P - h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace fad {

// Nearest E4M3 value of x (round to nearest even, saturating at +-448).
__device__ __forceinline__ float e4m3_round(float x)
{
    const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
}

// x -> (16 h, l) as floats that are exact E4M3 values; |x| <= 28.
__device__ __forceinline__ void e4m3_split(float x, float& hi16, float& lo)
{
    const float h = e4m3_round(x);
    hi16 = 16.f * h;
    lo = 16.f * (x - h);
}

// Two values x0, x1 (|x| <= 448 - 16) -> the E4M3 codes of h_i = e4m3(x_i)
// and of l_i = e4m3(x_i - h_i), packed two per word (x0's in the low byte):
// h + l carries x to about 2^-8 of |x|. Three packed conversions for the pair.
__device__ __forceinline__ void e4m3_split2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
    const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
    hi = (uint32_t)h;
    lo = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
}

// Two floats -> two E4M3 codes packed in the low 16 bits (a in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// The power of two sigma with amax * sigma <= limit (largest such; 1 for
// amax == 0 or not finite).
__device__ __forceinline__ float e4m3_split_scale(float amax, float limit)
{
    if (!(amax > 0.f) || !(amax < INFINITY)) return 1.f;
    float sig = exp2f(floorf(log2f(limit / amax)));
    while (amax * sig > limit) sig *= 0.5f;
    while (amax * sig * 2.f <= limit) sig *= 2.f;
    return sig;
}

}  // namespace fad
