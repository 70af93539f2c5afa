// Pieces shared by the router kernels (SIMT and tensor-core).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace moe {

// Ordering used for the choice: larger value first, lower expert index on equal values.
__device__ __forceinline__ bool route_better(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

__device__ __forceinline__ float route_sigmoid(float l) { return 1.0f / (1.0f + expf(-l)); }

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
