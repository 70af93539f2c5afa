// Router forward (logits, top-k choice, gates, z-loss) and router backward (logit
// gradient, W_r gradient).
//
// Router: "The whole stack, in the open" (Apex-3), "What's inside", row "Fine-grained
// MoE": a sigmoid router picks the top experts and a per-expert bias balances the load
// with no loss term. KempnerForge README, "Features": softmax top-k router and router
// z-loss. Handbook summary, section 2.5: router logits in fp32.
//
// The logits are an fp32 SIMT contraction over d (the router has E <= 256 outputs per
// token, too narrow for a tensor-core tile to pay, and fp32 is the stated router dtype).
// Every output is one thread's sequential sum over d, so results are bitwise repeatable.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "sizes.h"

namespace moe {
namespace {

constexpr int kTM = kRouteTokensPerCta;  // tokens per CTA (64)
constexpr int kKC = 32;                  // d-chunk per smem stage
constexpr int kThreads = 256;

// Ordering used for the choice: larger value first, lower expert index on equal values.
__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

__device__ __forceinline__ float sigmoid_f(float l) { return 1.0f / (1.0f + expf(-l)); }

// EJ = experts per thread column (E padded to 16 * EJ).
template <int EJ>
__global__ void __launch_bounds__(kThreads) route_fwd_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ W_r,
    const float* __restrict__ bias, int64_t T, int d, int E, int k, int mode,
    float* __restrict__ logits, int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
    float* __restrict__ topk_score, float* __restrict__ lse_out, double* __restrict__ z_part) {
    constexpr int EP = 16 * EJ;  // padded expert count of this instantiation
    // dynamic smem: the staging tiles (xs, wsm) and later the logit tile (lg) share space
    extern __shared__ __align__(16) unsigned char route_smem[];
    float(*xs)[kTM] = reinterpret_cast<float(*)[kTM]>(route_smem);
    float(*wsm)[EP] = reinterpret_cast<float(*)[EP]>(route_smem + sizeof(float) * kKC * kTM);
    float(*lg)[EP + 1] = reinterpret_cast<float(*)[EP + 1]>(route_smem);
    __shared__ double zw[kThreads / 32];

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int64_t t0 = (int64_t)blockIdx.x * kTM;

    float acc[4][EJ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += kKC) {
        // x chunk: 64 tokens x 32 columns of bf16, 8 columns (16 bytes) per thread
        {
            const int tok = tid / 4, part = tid % 4;
            const int64_t t = t0 + tok;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t < T) v = *reinterpret_cast<const uint4*>(x + t * d + k0 + part * 8);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                xs[part * 8 + 2 * q][tok] = bf16_lo(w[q]);
                xs[part * 8 + 2 * q + 1][tok] = bf16_hi(w[q]);
            }
        }
        // W_r chunk: EP experts x 32 columns of fp32
        for (int i = tid; i < EP * (kKC / 4); i += kThreads) {
            const int e = i / (kKC / 4), part = i % (kKC / 4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < E) v = *reinterpret_cast<const float4*>(W_r + (int64_t)e * d + k0 + part * 4);
            wsm[part * 4 + 0][e] = v.x;
            wsm[part * 4 + 1][e] = v.y;
            wsm[part * 4 + 2][e] = v.z;
            wsm[part * 4 + 3][e] = v.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kKC; ++kk) {
            const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
            float wv[EJ];
#pragma unroll
            for (int j = 0; j < EJ; ++j) wv[j] = wsm[kk][tx * EJ + j];
#pragma unroll
            for (int j = 0; j < EJ; ++j) {
                acc[0][j] = fmaf(xv.x, wv[j], acc[0][j]);
                acc[1][j] = fmaf(xv.y, wv[j], acc[1][j]);
                acc[2][j] = fmaf(xv.z, wv[j], acc[2][j]);
                acc[3][j] = fmaf(xv.w, wv[j], acc[3][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) lg[ty * 4 + i][tx * EJ + j] = acc[i][j];
    __syncthreads();

    if (logits) {
        for (int i = tid; i < kTM * E; i += kThreads) {
            const int r = i / E, e = i % E;
            if (t0 + r < T) logits[(t0 + r) * E + e] = lg[r][e];
        }
    }

    // top-k: one warp per token, lane holds experts lane + 32 j
    const int warp = tid / 32, lane = tid % 32;
    constexpr int VJ = (EP + 31) / 32;
    double zsum = 0.0;
    for (int r = warp; r < kTM; r += kThreads / 32) {
        const int64_t t = t0 + r;
        if (t >= T) break;
        float val[VJ];
#pragma unroll
        for (int j = 0; j < VJ; ++j) {
            const int e = lane + 32 * j;
            float v = -INFINITY;
            if (e < E) {
                const float l = lg[r][e];
                v = (mode == MOE_MODE_SIGMOID) ? sigmoid_f(l) + bias[e] : l;
                if (v != v) v = -INFINITY;  // a NaN never wins
            }
            val[j] = v;
        }
        // softmax statistics over all experts
        float mx = -INFINITY, sum = 0.f, lse = 0.f;
        if (mode == MOE_MODE_SOFTMAX) {
#pragma unroll
            for (int j = 0; j < VJ; ++j)
                if (lane + 32 * j < E) mx = fmaxf(mx, lg[r][lane + 32 * j]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
            for (int j = 0; j < VJ; ++j)
                if (lane + 32 * j < E) sum += expf(lg[r][lane + 32 * j] - mx);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            lse = mx + logf(sum);
        }
        int my_e = -1;
        float my_s = 0.f;
        float ssum = 0.f;
        uint32_t taken = 0;  // bit j: expert lane + 32 j already chosen
        for (int i = 0; i < k; ++i) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < VJ; ++j) {
                const int e = lane + 32 * j;
                if (e < E && !((taken >> j) & 1u) && better(val[j], e, bv, be)) {
                    bv = val[j];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (better(ov, oe, bv, be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            const float l = lg[r][be];
            const float s = (mode == MOE_MODE_SIGMOID) ? sigmoid_f(l) : expf(l - mx) / sum;
            ssum += s;
            if (lane == i) {
                my_e = be;
                my_s = s;
            }
        }
        if (lane < k) {
            topk_idx[t * k + lane] = my_e;
            topk_score[t * k + lane] = my_s;
            topk_gate[t * k + lane] = (mode == MOE_MODE_SIGMOID) ? my_s / ssum : my_s;
        }
        if (mode == MOE_MODE_SOFTMAX) {
            if (lane == 0) lse_out[t] = lse;
            zsum += (double)lse * (double)lse;
        }
    }
    if (mode == MOE_MODE_SOFTMAX) {
        if (lane == 0) zw[warp] = zsum;
        __syncthreads();
        if (tid == 0) {
            double s = 0.0;
            for (int w = 0; w < kThreads / 32; ++w) s += zw[w];
            z_part[blockIdx.x] = s;
        }
    }
}

__global__ void z_finalize_kernel(const double* __restrict__ z_part, int64_t nblocks, int64_t T,
                                  float z_coef, float* __restrict__ z_loss) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        double s = 0.0;
        for (int64_t i = 0; i < nblocks; ++i) s += z_part[i];
        z_loss[0] = (float)((double)z_coef * s / (double)T);
    }
}

// ---------------------------------------------------------------------------- backward

// One warp per token: dense row of the logit gradient.
__global__ void __launch_bounds__(256) route_bwd_dlogits_kernel(
    const float* __restrict__ dg, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_gate, const float* __restrict__ topk_score,
    const float* __restrict__ logits, const float* __restrict__ lse, int64_t T, int E, int k,
    int mode, float z_scale, float* __restrict__ dlogits) {
    const int lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (t >= T) return;
    // slot values held by lanes < k
    int my_e = -1;
    float my_g = 0.f, my_s = 0.f, my_dg = 0.f;
    if (lane < k) {
        my_e = topk_idx[t * k + lane];
        my_g = topk_gate[t * k + lane];
        my_s = topk_score[t * k + lane];
        my_dg = dg[t * k + lane];
    }
    // fixed-order sums over the slots (slot 0 first)
    float S = 0.f, gdg = 0.f;
    for (int i = 0; i < k; ++i) {
        S += __shfl_sync(0xffffffffu, my_s, i);
        gdg += __shfl_sync(0xffffffffu, my_g * my_dg, i);
    }
    if (mode == MOE_MODE_SIGMOID) {
        const float ds = (my_dg - gdg) / S;
        const float v = ds * my_s * (1.f - my_s);
        for (int e0 = 0; e0 < E; e0 += 32) {  // warp-uniform trip count
            const int e = e0 + lane;
            float out = 0.f;
            for (int i = 0; i < k; ++i) {
                const int ei = __shfl_sync(0xffffffffu, my_e, i);
                const float vi = __shfl_sync(0xffffffffu, v, i);
                if (ei == e) out = vi;
            }
            if (e < E) dlogits[t * E + e] = out;
        }
    } else {
        const float l_se = lse[t];
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            float sel = 0.f;
            for (int i = 0; i < k; ++i) {
                const int ei = __shfl_sync(0xffffffffu, my_e, i);
                const float di = __shfl_sync(0xffffffffu, my_dg, i);
                if (ei == e) sel = di;
            }
            if (e < E) {
                const float p = expf(logits[t * E + e] - l_se);
                dlogits[t * E + e] = p * (sel - gdg) + z_scale * l_se * p;
            }
        }
    }
}

// dW_r partial sums: part[s][e][j] = sum over tokens of split s of dlogits[t][e] * x[t][j].
// CTA tile: 64 experts x 128 columns; 256 threads, each 8 experts x 4 columns.
constexpr int kBwTE = 64, kBwTJ = 128, kBwTK = 32;

__global__ void __launch_bounds__(256) route_bwd_dwr_kernel(
    const float* __restrict__ dlogits, const __nv_bfloat16* __restrict__ x, int64_t T, int d,
    int E, float* __restrict__ part) {
    __shared__ __align__(16) float xs[kBwTK][kBwTJ];
    __shared__ __align__(16) float ds[kBwTK][kBwTE];
    const int tid = threadIdx.x;
    const int tx = tid % 32, ty = tid / 32;
    const int j0 = blockIdx.x * kBwTJ;
    const int e0 = blockIdx.y * kBwTE;
    const int64_t tbeg = (int64_t)blockIdx.z * kRouteBwdTokensPerSplit;
    const int64_t tend = min(T, tbeg + kRouteBwdTokensPerSplit);
    float acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
    for (int64_t tc = tbeg; tc < tend; tc += kBwTK) {
        // x chunk: 32 tokens x 128 columns bf16 = 32 x 16 uint4
        for (int i = tid; i < kBwTK * (kBwTJ / 8); i += 256) {
            const int r = i / (kBwTJ / 8), c = i % (kBwTJ / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tc + r < tend) v = *reinterpret_cast<const uint4*>(x + (tc + r) * d + j0 + c * 8);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                xs[r][c * 8 + 2 * q] = bf16_lo(w[q]);
                xs[r][c * 8 + 2 * q + 1] = bf16_hi(w[q]);
            }
        }
        for (int i = tid; i < kBwTK * kBwTE; i += 256) {
            const int r = i / kBwTE, e = i % kBwTE;
            float v = 0.f;
            if (tc + r < tend && e0 + e < E) v = dlogits[(tc + r) * E + e0 + e];
            ds[r][e] = v;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < kBwTK; ++r) {
            const float4 xv = *reinterpret_cast<const float4*>(&xs[r][tx * 4]);
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const float dv = ds[r][ty * 8 + a];
                acc[a][0] = fmaf(dv, xv.x, acc[a][0]);
                acc[a][1] = fmaf(dv, xv.y, acc[a][1]);
                acc[a][2] = fmaf(dv, xv.z, acc[a][2]);
                acc[a][3] = fmaf(dv, xv.w, acc[a][3]);
            }
        }
        __syncthreads();
    }
    float* out = part + (size_t)blockIdx.z * E * d;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int e = e0 + ty * 8 + a;
        if (e < E)
            *reinterpret_cast<float4*>(out + (size_t)e * d + j0 + tx * 4) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
}

__global__ void route_bwd_reduce_kernel(const float* __restrict__ part, int64_t nsplit,
                                        int64_t n, float* __restrict__ dW_r) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float s = 0.f;
    for (int64_t p = 0; p < nsplit; ++p) s += part[p * n + i];
    dW_r[i] = s;
}

template <int EJ>
int launch_route_fwd(const moe_bf16* x, const float* W_r, const float* b, int64_t T, int d,
                     int E, int k, int mode, float* logits, int32_t* idx, float* gate,
                     float* score, float* lse, double* zp, cudaStream_t st) {
    const int64_t nb = route_blocks(T);
    constexpr int EP = 16 * EJ;
    const size_t stage = sizeof(float) * kKC * (kTM + EP);
    const size_t tile = sizeof(float) * kTM * (EP + 1);
    const size_t smem = stage > tile ? stage : tile;
    if (cudaFuncSetAttribute(route_fwd_kernel<EJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    route_fwd_kernel<EJ><<<(unsigned)nb, kThreads, smem, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(x), W_r, b, T, d, E, k, mode, logits, idx, gate,
        score, lse, zp);
    return launch_status();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route(const moe_bf16* x, const float* W_r, const float* b, int64_t T, int d,
                         int E, int k, int mode, float z_coef, float* logits,
                         int32_t* topk_idx, float* topk_gate, float* topk_score, float* lse,
                         float* z_loss, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!x || !W_r || !topk_idx || !topk_gate || !topk_score) return MOE_ERR_INVALID_ARG;
    if (T <= 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_MODE_SIGMOID && mode != MOE_MODE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_MODE_SIGMOID && !b) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_MODE_SOFTMAX && (!logits || !lse || !z_loss)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(W_r)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    WsCarver wc(ws, ws_bytes);
    double* zp = wc.take<double>(route_blocks(T));
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    int rc;
    if (E <= 16) rc = launch_route_fwd<1>(x, W_r, b, T, d, E, k, mode, logits, topk_idx, topk_gate, topk_score, lse, zp, st);
    else if (E <= 32) rc = launch_route_fwd<2>(x, W_r, b, T, d, E, k, mode, logits, topk_idx, topk_gate, topk_score, lse, zp, st);
    else if (E <= 64) rc = launch_route_fwd<4>(x, W_r, b, T, d, E, k, mode, logits, topk_idx, topk_gate, topk_score, lse, zp, st);
    else if (E <= 128) rc = launch_route_fwd<8>(x, W_r, b, T, d, E, k, mode, logits, topk_idx, topk_gate, topk_score, lse, zp, st);
    else rc = launch_route_fwd<16>(x, W_r, b, T, d, E, k, mode, logits, topk_idx, topk_gate, topk_score, lse, zp, st);
    if (rc != MOE_OK) return rc;
    if (mode == MOE_MODE_SOFTMAX) {
        z_finalize_kernel<<<1, 32, 0, st>>>(zp, route_blocks(T), T, z_coef, z_loss);
        rc = launch_status();
    }
    return rc;
}

extern "C" int moe_route_bwd(const float* dg, const moe_bf16* x, const int32_t* topk_idx,
                             const float* topk_gate, const float* topk_score,
                             const float* logits, const float* lse, int64_t T, int d, int E,
                             int k, int mode, float z_coef, float* dlogits, float* dW_r,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!dg || !x || !topk_idx || !topk_gate || !topk_score || !dlogits || !dW_r)
        return MOE_ERR_INVALID_ARG;
    if (T <= 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_MODE_SIGMOID && mode != MOE_MODE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_MODE_SOFTMAX && (!logits || !lse)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(dW_r)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    WsCarver wc(ws, ws_bytes);
    const int64_t nsplit = route_bwd_splits(T);
    float* part = wc.take<float>((size_t)nsplit * E * d);
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const float z_scale = 2.0f * z_coef / (float)T;
    route_bwd_dlogits_kernel<<<(unsigned)cdiv(T, 8), 256, 0, st>>>(
        dg, topk_idx, topk_gate, topk_score, logits, lse, T, E, k, mode, z_scale, dlogits);
    if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    dim3 grid(d / kBwTJ, (unsigned)cdiv(E, kBwTE), (unsigned)nsplit);
    route_bwd_dwr_kernel<<<grid, 256, 0, st>>>(dlogits, reinterpret_cast<const __nv_bfloat16*>(x),
                                               T, d, E, part);
    if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    const int64_t n = (int64_t)E * d;
    route_bwd_reduce_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(part, nsplit, n, dW_r);
    return launch_status();
}
