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

// Rowwise codes are a function of the row alone, so the codes of a token's k expert-major
// rows are its own codes: quantise the T token rows once and copy codes and scale to the
// rows (one warp per token, 16-byte vectors), instead of quantising the k-fold larger
// permuted bf16 rows.
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) gather_fp8_kernel(
    const uint8_t* __restrict__ xq, const float* __restrict__ sx,
    const int32_t* __restrict__ slot_to_row, int64_t T, int d, int k, uint8_t* __restrict__ Xq,
    float* __restrict__ sX) {
    const int lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * kGatherWarps + threadIdx.x / 32;
    if (t >= T) return;
    int32_t my_row = -1;
    if (lane < k) my_row = slot_to_row[t * k + lane];
    if (my_row >= 0) sX[my_row] = sx[t];
    const uint4* src = reinterpret_cast<const uint4*>(xq + t * d);
    const int nvec = d / 16;
    for (int c0 = 0; c0 < nvec; c0 += 32) {  // warp-uniform trip count
        const int c = c0 + lane;
        const bool in = c < nvec;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (in) v = src[c];
        for (int i = 0; i < k; ++i) {
            const int32_t row = __shfl_sync(0xffffffffu, my_row, i);
            if (in && row >= 0) reinterpret_cast<uint4*>(Xq + (int64_t)row * d)[c] = v;
        }
    }
}

// Padding rows of each segment (the trailing rows with perm_token < 0; at most
// MOE_ROW_ALIGN - 1 per expert) get what quantising a zero row gives: zero codes, scale 1.
constexpr int kPadSplitFp8 = 16;

__global__ void __launch_bounds__(256) pad_rows_fp8_kernel(const int64_t* __restrict__ row_offsets,
                                                           const int32_t* __restrict__ perm_token,
                                                           int d, uint8_t* __restrict__ Xq,
                                                           float* __restrict__ sX) {
    const int e = blockIdx.x;
    const int64_t hi = row_offsets[e + 1];
    int64_t lo = row_offsets[e];
    if (hi - lo > MOE_ROW_ALIGN - 1) lo = hi - (MOE_ROW_ALIGN - 1);
    const int vec_per_row = d / 16;
    for (int64_t i = (int64_t)blockIdx.y * blockDim.x + threadIdx.x; i < (hi - lo) * vec_per_row;
         i += (int64_t)gridDim.y * blockDim.x) {
        const int64_t r = lo + i / vec_per_row;
        const int c = (int)(i % vec_per_row);
        if (perm_token[r] < 0) {
            reinterpret_cast<uint4*>(Xq + r * d)[c] = make_uint4(0, 0, 0, 0);
            if (c == 0) sX[r] = 1.0f;
        }
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

extern "C" int moe_permute_fp8(const uint8_t* xq, const float* sx, const int32_t* slot_to_row,
                               const int32_t* perm_token, const int64_t* row_offsets, int64_t T,
                               int d, int E, int k, uint8_t* Xq, float* sX, moe_stream_t stream) {
    if (!xq || !sx || !slot_to_row || !perm_token || !row_offsets || !Xq || !sX)
        return MOE_ERR_INVALID_ARG;
    if (T <= 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(xq) || !aligned16(Xq)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    gather_fp8_kernel<<<(unsigned)cdiv(T, kGatherWarps), kGatherWarps * 32, 0, st>>>(
        xq, sx, slot_to_row, T, d, k, Xq, sX);
    pad_rows_fp8_kernel<<<dim3(E, kPadSplitFp8), 256, 0, st>>>(row_offsets, perm_token, d, Xq, sX);
    return launch_status();
}
