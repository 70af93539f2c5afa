// E4M3 quantisation helpers shared by the kernels that write FP8 codes: the scale of a row
// or column (RN(amax / 448), 1 for a zero amax), the correctly rounded quotient x / scale
// without a division (Markstein's FMA correction with the correctly rounded reciprocal; see
// fp8.cu), and the conversion of eight bf16 values to eight codes, round to nearest even,
// saturating at 448.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// scale = RN(amax / 448) (1 for a zero amax) and its correctly rounded reciprocal.
struct Fp8Scale {
    float s, rs;
    __device__ __forceinline__ explicit Fp8Scale(float amax) {
        s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        rs = __frcp_rn(s);
    }
    __device__ __forceinline__ static Fp8Scale of(float scale) {  // a scale formed before
        Fp8Scale f(0.f);
        f.s = scale;
        f.rs = __frcp_rn(scale);
        return f;
    }
    __device__ __forceinline__ float quot(float x) const {  // RN(x / s)
        const float q0 = __fmul_rn(x, rs);
        const float e = __fmaf_rn(-q0, s, x);
        return __fmaf_rn(e, rs, q0);
    }
};

__device__ __forceinline__ float amax8(const uint4 v, float m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
    return m;
}

// Eight bf16 values -> eight E4M3 codes.
__device__ __forceinline__ uint2 codes8(const uint4 v, const Fp8Scale& sc) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t p0 = __nv_cvt_float2_to_fp8x2(
            make_float2(sc.quot(bf16_lo(w[2 * h])), sc.quot(bf16_hi(w[2 * h]))), __NV_SATFINITE,
            __NV_E4M3);
        const __nv_fp8x2_storage_t p1 = __nv_cvt_float2_to_fp8x2(
            make_float2(sc.quot(bf16_lo(w[2 * h + 1])), sc.quot(bf16_hi(w[2 * h + 1]))),
            __NV_SATFINITE, __NV_E4M3);
        packed[h] = (uint32_t)p0 | ((uint32_t)p1 << 16);
    }
    return make_uint2(packed[0], packed[1]);
}


// Eight floats (already bf16 values) -> eight codes.
__device__ __forceinline__ uint2 codes8f(const float (&v)[8], const Fp8Scale& sc) {
    uint32_t packed[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t p0 = __nv_cvt_float2_to_fp8x2(
            make_float2(sc.quot(v[4 * h]), sc.quot(v[4 * h + 1])), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t p1 = __nv_cvt_float2_to_fp8x2(
            make_float2(sc.quot(v[4 * h + 2]), sc.quot(v[4 * h + 3])), __NV_SATFINITE, __NV_E4M3);
        packed[h] = (uint32_t)p0 | ((uint32_t)p1 << 16);
    }
    return make_uint2(packed[0], packed[1]);
}

}  // namespace moe
