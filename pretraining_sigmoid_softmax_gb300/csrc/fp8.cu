// Rowwise FP8 (E4M3) quantisation of GEMM operands ("The whole stack, in the open" (Apex-3):
// the benchmark and training run with --precision fp8_rowwise): per row, scale = amax / 448
// and code = E4M3(x / scale), round to nearest even, saturating. Both quotients are the
// correctly rounded fp32 quotients (IEEE division), so the codes are reproducible bit for
// bit. Per element the quotient is formed without a division: with rs = RN(1 / scale) (the
// correctly rounded reciprocal), q0 = RN(x rs), e = x - scale q0 (exact in one FMA) and
// q = RN(q0 + e rs) is RN(x / scale) - Markstein's theorem for FMA division with a correctly
// rounded reciprocal, valid while nothing under- or overflows; |x / scale| <= 448 here, and
// quotients small enough to underflow quantise to zero whichever way they round.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "sizes.h"

namespace moe {
namespace {

constexpr int kQWarps = 8;

__global__ void __launch_bounds__(kQWarps * 32) quantize_rows_fp8_kernel(
    const __nv_bfloat16* __restrict__ X, const int64_t* __restrict__ limit, int64_t rows, int cols,
    uint8_t* __restrict__ Q, float* __restrict__ S) {
    const int lane = threadIdx.x % 32;
    const int64_t nwarps = (int64_t)gridDim.x * kQWarps;
    int64_t n = rows;
    if (limit) n = min(n, *limit);
    const int nvec = cols / 8;
    for (int64_t r = (int64_t)blockIdx.x * kQWarps + threadIdx.x / 32; r < n; r += nwarps) {
        const uint4* src = reinterpret_cast<const uint4*>(X + r * cols);
        float m = 0.f;
        for (int c = lane; c < nvec; c += 32) {
            const uint4 v = src[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float s = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
        const float rs = __frcp_rn(s);
        auto quot = [s, rs](float x) {  // RN(x / s)
            const float q0 = __fmul_rn(x, rs);
            const float e = __fmaf_rn(-q0, s, x);
            return __fmaf_rn(e, rs, q0);
        };
        uint2* dst = reinterpret_cast<uint2*>(Q + r * cols);
        for (int c = lane; c < nvec; c += 32) {
            const uint4 v = src[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t packed[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const __nv_fp8x2_storage_t p0 = __nv_cvt_float2_to_fp8x2(
                    make_float2(quot(bf16_lo(w[2 * h])), quot(bf16_hi(w[2 * h]))),
                    __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t p1 = __nv_cvt_float2_to_fp8x2(
                    make_float2(quot(bf16_lo(w[2 * h + 1])), quot(bf16_hi(w[2 * h + 1]))),
                    __NV_SATFINITE, __NV_E4M3);
                packed[h] = (uint32_t)p0 | ((uint32_t)p1 << 16);
            }
            dst[c] = make_uint2(packed[0], packed[1]);
        }
        if (lane == 0) S[r] = s;
    }
}

}  // namespace

int launch_quantize_rows_fp8(const __nv_bfloat16* X, const int64_t* limit, int64_t rows, int cols,
                             uint8_t* Q, float* S, cudaStream_t st) {
    int64_t blocks = cdiv(rows, kQWarps);
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_rows_fp8_kernel<<<(unsigned)blocks, kQWarps * 32, 0, st>>>(X, limit, rows, cols, Q, S);
    return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" int moe_quantize_rows_fp8(const moe_bf16* X, const int64_t* rows_limit, int64_t rows,
                                     int cols, uint8_t* Q, float* scale, moe_stream_t stream) {
    if (!X || !Q || !scale) return MOE_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(X) || !aligned16(Q)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    return launch_quantize_rows_fp8(reinterpret_cast<const __nv_bfloat16*>(X), rows_limit, rows,
                                    cols, Q, scale, (cudaStream_t)stream);
}
