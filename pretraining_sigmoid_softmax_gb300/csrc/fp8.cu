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
#include "fp8.cuh"
#include "sizes.h"

namespace moe {
namespace {

constexpr int kQWarps = 8;

// One warp per row. With X1, the row is the concatenation [X0 row | X1 row] (each `cols`
// wide) under one scale, and its codes fill 2 cols bytes of Q.
__global__ void __launch_bounds__(kQWarps * 32) quantize_rows_fp8_kernel(
    const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ X1,
    const int64_t* __restrict__ limit, int64_t rows, int cols, uint8_t* __restrict__ Q,
    float* __restrict__ S) {
    const int lane = threadIdx.x % 32;
    const int64_t nwarps = (int64_t)gridDim.x * kQWarps;
    int64_t n = rows;
    if (limit) n = min(n, *limit);
    const int nvec = cols / 8;
    const int64_t qcols = X1 ? 2 * (int64_t)cols : cols;
    for (int64_t r = (int64_t)blockIdx.x * kQWarps + threadIdx.x / 32; r < n; r += nwarps) {
        const uint4* src = reinterpret_cast<const uint4*>(X + r * cols);
        const uint4* src1 = X1 ? reinterpret_cast<const uint4*>(X1 + r * cols) : nullptr;
        float m = 0.f;
        for (int c = lane; c < nvec; c += 32) {
            m = amax8(src[c], m);
            if (src1) m = amax8(src1[c], m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const Fp8Scale sc(m);
        uint2* dst = reinterpret_cast<uint2*>(Q + r * qcols);
        for (int c = lane; c < nvec; c += 32) {
            dst[c] = codes8(src[c], sc);
            if (src1) dst[nvec + c] = codes8(src1[c], sc);
        }
        if (lane == 0) S[r] = sc.s;
    }
}

// ------------------------------------------------ columnwise scales, transposed codes
// X is E matrices of K x N bf16 (row-major), or, with X1, the K = 2 K0 stack of X0 over X1
// (both E x K0 x N). Column n of matrix e gets scale RN(amax / 448) over its K values, and
// its codes are written transposed, Qt[e][n][0..K), so that a GEMM contracting over K
// reads them K-major.
constexpr int kColThreads = 256;

// Column amax: thread = 8 adjacent columns (16-byte loads), block = kAmaxThreads threads x
// kAmaxRows rows, so that even one small matrix fills the GPU. Block maxima meet by an
// integer atomic max on the bits of non-negative floats, which order as the floats do (a
// maximum does not depend on the order of its arguments). `bits` starts at zero.
constexpr int kAmaxThreads = 128;
constexpr int kAmaxRows = 128;

__global__ void __launch_bounds__(kAmaxThreads) col_amax_kernel(
    const __nv_bfloat16* __restrict__ X0, const __nv_bfloat16* __restrict__ X1, int K0, int N,
    unsigned int* __restrict__ bits) {
    const int e = blockIdx.y;
    const int K = X1 ? 2 * K0 : K0;
    const int c = (blockIdx.x * kAmaxThreads + threadIdx.x) * 8;
    if (c >= N) return;
    const int r0 = blockIdx.z * kAmaxRows;
    const int r1 = min(K, r0 + kAmaxRows);
    auto row = [&](int r) {
        return reinterpret_cast<const uint4*>(
            (r < K0 ? X0 + ((int64_t)e * K0 + r) * N : X1 + ((int64_t)e * K0 + (r - K0)) * N) + c);
    };
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0.f;
    auto fold = [&](const uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            m[2 * q] = fmaxf(m[2 * q], fabsf(bf16_lo(w[q])));
            m[2 * q + 1] = fmaxf(m[2 * q + 1], fabsf(bf16_hi(w[q])));
        }
    };
    int r = r0;
    for (; r + 4 <= r1; r += 4) {  // four rows in flight
        const uint4 v0 = *row(r), v1 = *row(r + 1), v2 = *row(r + 2), v3 = *row(r + 3);
        fold(v0);
        fold(v1);
        fold(v2);
        fold(v3);
    }
    for (; r < r1; ++r) fold(*row(r));
#pragma unroll
    for (int j = 0; j < 8; ++j) atomicMax(bits + (int64_t)e * N + c + j, __float_as_uint(m[j]));
}

// amax (as bits) -> scale, in place.
__global__ void col_scale_kernel(float* __restrict__ S, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) S[i] = Fp8Scale(S[i]).s;
}

// Tiles of 128 K-rows x 64 columns: read as 128 bf16 row pieces of 128 bytes, written as 64
// code rows of 128 bytes (whole lines).
constexpr int kColTileK = 128;
constexpr int kColTileN = 64;

__global__ void __launch_bounds__(kColThreads) col_quantize_kernel(
    const __nv_bfloat16* __restrict__ X0, const __nv_bfloat16* __restrict__ X1, int K0, int N,
    const float* __restrict__ S, uint8_t* __restrict__ Qt) {
    __shared__ float tile[kColTileK][kColTileN + 1];
    const int e = blockIdx.z;
    const int n0 = blockIdx.x * kColTileN;
    const int k0 = blockIdx.y * kColTileK;  // over K = K0 or 2 K0
    const int K = X1 ? 2 * K0 : K0;
    const int tid = threadIdx.x;
    // load: 128 rows x 64 bf16 (8 vectors of 8 per row); 1024 vectors, four per thread
    for (int i = tid; i < kColTileK * (kColTileN / 8); i += kColThreads) {
        const int r = i / (kColTileN / 8), c8 = i % (kColTileN / 8);
        const int k = k0 + r;
        const __nv_bfloat16* src = (k < K0 ? X0 + (int64_t)e * K0 * N + (int64_t)k * N
                                           : X1 + (int64_t)e * K0 * N + (int64_t)(k - K0) * N) +
                                   n0 + 8 * c8;
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            tile[r][8 * c8 + 2 * q] = bf16_lo(w[q]);
            tile[r][8 * c8 + 2 * q + 1] = bf16_hi(w[q]);
        }
    }
    __syncthreads();
    // store: code row n (128 K values) in eight 16-byte pieces; 512 pieces, two per thread
    for (int i = tid; i < kColTileN * 8; i += kColThreads) {
        const int nl = i / 8, piece = i % 8;
        const Fp8Scale cs = Fp8Scale::of(S[(int64_t)e * N + n0 + nl]);
        uint32_t out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t word = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int kk = 16 * piece + 4 * q + 2 * h;
                const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(
                    make_float2(cs.quot(tile[kk][nl]), cs.quot(tile[kk + 1][nl])), __NV_SATFINITE,
                    __NV_E4M3);
                word |= (uint32_t)p << (16 * h);
            }
            out[q] = word;
        }
        uint8_t* dst = Qt + ((int64_t)e * N + n0 + nl) * K + k0 + 16 * piece;
        *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
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
                             uint8_t* Q, float* S, cudaStream_t st, const __nv_bfloat16* X1) {
    int64_t blocks = cdiv(rows, kQWarps);
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_rows_fp8_kernel<<<(unsigned)blocks, kQWarps * 32, 0, st>>>(X, X1, limit, rows, cols,
                                                                       Q, S);
    return launch_status();
}

int launch_pad_rows_fp8(const int64_t* row_offsets, const int32_t* perm_token, int d, int E,
                        uint8_t* Xq, float* sX, cudaStream_t st) {
    pad_rows_fp8_kernel<<<dim3(E, kPadSplitFp8), 256, 0, st>>>(row_offsets, perm_token, d, Xq, sX);
    return launch_status();
}

int launch_quantize_cols_fp8(const __nv_bfloat16* X0, const __nv_bfloat16* X1, int E, int K0,
                             int N, uint8_t* Qt, float* S, cudaStream_t st) {
    const int K = X1 ? 2 * K0 : K0;
    if (cudaMemsetAsync(S, 0, sizeof(float) * (size_t)E * N, st) != cudaSuccess) return MOE_ERR_LAUNCH;
    col_amax_kernel<<<dim3((unsigned)cdiv(N, 8 * kAmaxThreads), (unsigned)E,
                           (unsigned)cdiv(K, kAmaxRows)),
                      kAmaxThreads, 0, st>>>(X0, X1, K0, N, reinterpret_cast<unsigned int*>(S));
    col_scale_kernel<<<(unsigned)cdiv((int64_t)E * N, 256), 256, 0, st>>>(S, (int64_t)E * N);
    col_quantize_kernel<<<dim3((unsigned)(N / kColTileN), (unsigned)(K / kColTileK), (unsigned)E),
                          kColThreads, 0, st>>>(X0, X1, K0, N, S, Qt);
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
                                    cols, Q, scale, (cudaStream_t)stream, nullptr);
}

extern "C" int moe_quantize_rows2_fp8(const moe_bf16* X0, const moe_bf16* X1,
                                      const int64_t* rows_limit, int64_t rows, int cols,
                                      uint8_t* Q, float* scale, moe_stream_t stream) {
    if (!X0 || !X1 || !Q || !scale) return MOE_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(X0) || !aligned16(X1) || !aligned16(Q)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    return launch_quantize_rows_fp8(reinterpret_cast<const __nv_bfloat16*>(X0), rows_limit, rows,
                                    cols, Q, scale, (cudaStream_t)stream,
                                    reinterpret_cast<const __nv_bfloat16*>(X1));
}

extern "C" int moe_quantize_cols_fp8(const moe_bf16* X0, const moe_bf16* X1, int E, int K0, int N,
                                     uint8_t* Qt, float* scale, moe_stream_t stream) {
    if (!X0 || !Qt || !scale) return MOE_ERR_INVALID_ARG;
    if (E <= 0 || K0 <= 0 || N <= 0) return MOE_ERR_INVALID_ARG;
    if (K0 % 128 != 0 || N % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(X0) || (X1 && !aligned16(X1)) || !aligned16(Qt)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    return launch_quantize_cols_fp8(reinterpret_cast<const __nv_bfloat16*>(X0),
                                    reinterpret_cast<const __nv_bfloat16*>(X1), E, K0, N, Qt,
                                    scale, (cudaStream_t)stream);
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
