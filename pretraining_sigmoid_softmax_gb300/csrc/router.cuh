// Pieces shared by the router kernels (SIMT and tensor-core).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

namespace moe {

// Ordering used for the choice: larger value first, lower expert index on equal values.
__device__ __forceinline__ bool route_better(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

__device__ __forceinline__ float route_sigmoid(float l) { return 1.0f / (1.0f + expf(-l)); }

// The sigmoid inside the selection value sigmoid(l) + b, which only orders experts: the
// exponential and reciprocal by the hardware approximations (__expf, __fdividef) instead of
// the correctly rounded expf and division. Over all l its absolute error stays within a few
// 1e-7 (the relative error of __expf grows with |l|, but sigmoid's slope e^-|l| shrinks
// faster), so it can reorder only experts whose values lie that close; the scores and gates
// of the chosen experts use route_sigmoid. For l < -88, __expf(-l) is +inf and the value 0.
__device__ __forceinline__ float route_select_sigmoid(float l) {
    return __fdividef(1.0f, 1.0f + __expf(-l));
}

// Order-preserving integer key of a selection value: for non-NaN a and b, a > b exactly when
// route_key(a) > route_key(b) as signed integers, and a == b exactly when the keys are equal
// (-0 is folded into +0 first, as the float order has them equal). Positive floats keep their
// bits; for negative ones the magnitude bits are flipped, so a larger magnitude sorts lower.
// No non-NaN value has the key INT_MIN, which marks an empty slot.
__device__ __forceinline__ int route_key(float v) {
    const int b = __float_as_int(v + 0.0f);
    return b ^ ((b >> 31) & 0x7fffffff);
}

// The K best experts among those pushed so far, best first, in the choice's order. Experts
// must be pushed in increasing index order: a later expert then displaces an earlier one only
// with a strictly larger value, so equal values keep the lower index ahead, and an empty slot
// (key INT_MIN) loses to every expert. A push compares the new key with all K slots at once
// and shifts the slots below its place down by one (an insertion network: branch-free, a
// fixed number of compares and selects). Each slot also carries the expert's logit.
template <int K>
struct RouteTopK {
    int key[K];
    int e[K];
    float l[K];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            key[j] = INT_MIN;
            e[j] = 0;
            l[j] = 0.f;
        }
    }
    __device__ __forceinline__ void push(int ck, int ce, float cl) {
        bool b[K];
#pragma unroll
        for (int j = 0; j < K; ++j) b[j] = ck > key[j];  // true from the new expert's place down
#pragma unroll
        for (int j = K - 1; j > 0; --j) {
            key[j] = b[j] ? (b[j - 1] ? key[j - 1] : ck) : key[j];
            e[j] = b[j] ? (b[j - 1] ? e[j - 1] : ce) : e[j];
            l[j] = b[j] ? (b[j - 1] ? l[j - 1] : cl) : l[j];
        }
        key[0] = b[0] ? ck : key[0];
        e[0] = b[0] ? ce : e[0];
        l[0] = b[0] ? cl : l[0];
    }
};

// Three bf16 pieces of an fp32 value: p0 = bf16(v), p1 = bf16(v - p0), p2 = bf16(v - p0 - p1).
// Both differences are exact in fp32 (Sterbenz: each piece is within a factor 2 of what it
// rounds), and each rounding keeps 8 more significant bits, so |v - (p0 + p1 + p2)| is at
// most 2^-24 |v|: the pieces hold v to fp32's own unit roundoff.
__device__ __forceinline__ void split3_bf16(float v, __nv_bfloat16& p0, __nv_bfloat16& p1,
                                            __nv_bfloat16& p2) {
    p0 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(p0);
    p1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(p1);
    p2 = __float2bfloat16_rn(r2);
}

// Tensor-core router forward (E <= 128; route_tc.cu). w3 is scratch for the three bf16
// pieces of W_r ([3][route_tc_epad(E)][d]); z_part receives 4 partial sums of lse^2 per
// 128-token tile (softmax mode), *nz is set to their count.
int launch_route_logits_tc(const __nv_bfloat16* x, const float* W_r, const float* b, int64_t T,
                           int d, int E, int k, int mode, float* logits, int32_t* topk_idx,
                           float* topk_gate, float* topk_score, float* lse, double* z_part,
                           int64_t* nz, __nv_bfloat16* w3, cudaStream_t st);

// Tensor-core W_r-gradient partial sums (E <= 128; route_tc.cu): part[s][e][j] over the
// tokens of split s, from the three bf16 pieces of the logit gradient (piece p a [T, np]
// matrix at dl3 + p * pstride, each 16-byte aligned). *nsplit is set to the number of splits
// written.
int launch_route_dwr_tc(const __nv_bfloat16* x, const __nv_bfloat16* dl3, int64_t pstride,
                        int64_t T, int d, int E, float* part, int64_t* nsplit, cudaStream_t st);

// Router input-gradient term dx_r = dlogits W_r on the tensor cores (E <= 128; route_tc.cu).
// Scratch: dl2, the first two bf16 pieces of dlogits ([T, np] each, pstride elements apart,
// 16-byte aligned), and w3, the three pieces of W_r ([3][np][d]). dx_r [T, d] fp32.
int launch_router_dx_tc(const float* dlogits, const float* W_r, int64_t T, int d, int E,
                        __nv_bfloat16* dl2, int64_t pstride, __nv_bfloat16* w3, float* dx_r,
                        cudaStream_t st);

}  // namespace moe
