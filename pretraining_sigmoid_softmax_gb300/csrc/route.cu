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

constexpr int kKC = 32;                  // d-chunk per smem stage
constexpr int kThreads = 256;

// Ordering used for the choice: larger value first, lower expert index on equal values.
__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

__device__ __forceinline__ float sigmoid_f(float l) { return 1.0f / (1.0f + expf(-l)); }

// Logit tile of TM tokens x EP (padded) experts per CTA, 256 threads; each thread owns
// TTOK tokens x EJ experts and sums over d sequentially (fixed order). The next 32-wide
// d-chunk is prefetched into registers while the current one is multiplied from shared
// memory.
template <int EP, int TM, int TTOK, int EJ>
__global__ void __launch_bounds__(kThreads) route_fwd_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ W_r,
    const float* __restrict__ bias, int64_t T, int d, int E, int k, int mode,
    float* __restrict__ logits, int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
    float* __restrict__ topk_score, float* __restrict__ lse_out, double* __restrict__ z_part) {
    constexpr int TXN = EP / EJ;  // thread columns
    static_assert((TM / TTOK) * TXN == kThreads, "thread tiling");
    static_assert(TTOK % 4 == 0 && (EJ % 4 == 0 || EJ == 2), "vector widths");
    constexpr int XV = TM * (kKC / 8);  // uint4 (8 bf16) per x chunk
    constexpr int WV = EP * (kKC / 4);  // float4 per W chunk
    constexpr int XL = (XV + kThreads - 1) / kThreads;
    constexpr int WL = (WV + kThreads - 1) / kThreads;
    // dynamic smem: the staging tiles (xs, wsm) and later the logit tile (lg) share space
    extern __shared__ __align__(16) unsigned char route_smem[];
    float(*xs)[TM] = reinterpret_cast<float(*)[TM]>(route_smem);
    float(*wsm)[EP] = reinterpret_cast<float(*)[EP]>(route_smem + sizeof(float) * kKC * TM);
    float(*lg)[EP + 1] = reinterpret_cast<float(*)[EP + 1]>(route_smem);
    __shared__ double zw[kThreads / 32];

    const int tid = threadIdx.x;
    const int ty = tid / TXN, tx = tid % TXN;
    const int64_t t0 = (int64_t)blockIdx.x * TM;

    float acc[TTOK][EJ];
#pragma unroll
    for (int i = 0; i < TTOK; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) acc[i][j] = 0.f;

    uint4 xr[XL];
    float4 wr[WL];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int q = 0; q < XL; ++q) {
            const int i = tid + q * kThreads;
            const int tok = i / (kKC / 8), part = i % (kKC / 8);
            xr[q] = make_uint4(0, 0, 0, 0);
            if (i < XV && t0 + tok < T)
                xr[q] = __ldg(reinterpret_cast<const uint4*>(x + (t0 + tok) * d + k0 + part * 8));
        }
#pragma unroll
        for (int q = 0; q < WL; ++q) {
            const int i = tid + q * kThreads;
            const int e = i / (kKC / 4), part = i % (kKC / 4);
            wr[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < WV && e < E)
                wr[q] = __ldg(reinterpret_cast<const float4*>(W_r + (int64_t)e * d + k0 + part * 4));
        }
    };
    fetch(0);
    for (int k0 = 0; k0 < d; k0 += kKC) {
        __syncthreads();  // the previous chunk's readers are done
#pragma unroll
        for (int q = 0; q < XL; ++q) {
            const int i = tid + q * kThreads;
            if (i < XV) {
                const int tok = i / (kKC / 8), part = i % (kKC / 8);
                const uint32_t w[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    xs[part * 8 + 2 * h][tok] = bf16_lo(w[h]);
                    xs[part * 8 + 2 * h + 1][tok] = bf16_hi(w[h]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < WL; ++q) {
            const int i = tid + q * kThreads;
            if (i < WV) {
                const int e = i / (kKC / 4), part = i % (kKC / 4);
                wsm[part * 4 + 0][e] = wr[q].x;
                wsm[part * 4 + 1][e] = wr[q].y;
                wsm[part * 4 + 2][e] = wr[q].z;
                wsm[part * 4 + 3][e] = wr[q].w;
            }
        }
        __syncthreads();
        if (k0 + kKC < d) fetch(k0 + kKC);  // in flight while this chunk is multiplied
#pragma unroll 4
        for (int kk = 0; kk < kKC; ++kk) {
            float xv[TTOK], wv[EJ];
#pragma unroll
            for (int i = 0; i < TTOK; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(&xs[kk][ty * TTOK + i]);
                xv[i] = v.x;
                xv[i + 1] = v.y;
                xv[i + 2] = v.z;
                xv[i + 3] = v.w;
            }
            if constexpr (EJ == 2) {
                const float2 v = *reinterpret_cast<const float2*>(&wsm[kk][tx * EJ]);
                wv[0] = v.x;
                wv[1] = v.y;
            } else {
#pragma unroll
                for (int j = 0; j < EJ; j += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(&wsm[kk][tx * EJ + j]);
                    wv[j] = v.x;
                    wv[j + 1] = v.y;
                    wv[j + 2] = v.z;
                    wv[j + 3] = v.w;
                }
            }
#pragma unroll
            for (int i = 0; i < TTOK; ++i)
#pragma unroll
                for (int j = 0; j < EJ; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
    }
    __syncthreads();  // staging tiles are dead; reuse the space for the logit tile
#pragma unroll
    for (int i = 0; i < TTOK; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) lg[ty * TTOK + i][tx * EJ + j] = acc[i][j];
    __syncthreads();

    if (logits) {
        for (int i = tid; i < TM * E; i += kThreads) {
            const int r = i / E, e = i % E;
            if (t0 + r < T) logits[(t0 + r) * E + e] = lg[r][e];
        }
    }

    // top-k: one warp per token, lane holds experts lane + 32 j
    const int warp = tid / 32, lane = tid % 32;
    constexpr int VJ = (EP + 31) / 32;
    double zsum = 0.0;
    for (int r = warp; r < TM; r += kThreads / 32) {
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
// CTA tile: 64 experts x 128 columns; 256 threads, each 8 experts x 4 columns, summing over
// the split's tokens in order. The next 32-token chunk is prefetched into registers.
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
    // per chunk: x 32 x 128 bf16 = 512 uint4, dlogits 32 x 64 fp32 = 2048 floats
    uint4 xr[2];
    float dr[8];
    auto fetch = [&](int64_t tc) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = tid + q * 256;
            const int r = i / (kBwTJ / 8), c = i % (kBwTJ / 8);
            xr[q] = make_uint4(0, 0, 0, 0);
            if (tc + r < tend) xr[q] = __ldg(reinterpret_cast<const uint4*>(x + (tc + r) * d + j0 + c * 8));
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = tid + q * 256;
            const int r = i / kBwTE, e = i % kBwTE;
            dr[q] = 0.f;
            if (tc + r < tend && e0 + e < E) dr[q] = __ldg(dlogits + (tc + r) * E + e0 + e);
        }
    };
    fetch(tbeg);
    for (int64_t tc = tbeg; tc < tend; tc += kBwTK) {
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = tid + q * 256;
            const int r = i / (kBwTJ / 8), c = i % (kBwTJ / 8);
            const uint32_t w[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                xs[r][c * 8 + 2 * h] = bf16_lo(w[h]);
                xs[r][c * 8 + 2 * h + 1] = bf16_hi(w[h]);
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = tid + q * 256;
            ds[i / kBwTE][i % kBwTE] = dr[q];
        }
        __syncthreads();
        if (tc + kBwTK < tend) fetch(tc + kBwTK);
#pragma unroll 4
        for (int r = 0; r < kBwTK; ++r) {
            const float4 xv = *reinterpret_cast<const float4*>(&xs[r][tx * 4]);
            const float4 d0 = *reinterpret_cast<const float4*>(&ds[r][ty * 8]);
            const float4 d1 = *reinterpret_cast<const float4*>(&ds[r][ty * 8 + 4]);
            const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                acc[a][0] = fmaf(dv[a], xv.x, acc[a][0]);
                acc[a][1] = fmaf(dv[a], xv.y, acc[a][1]);
                acc[a][2] = fmaf(dv[a], xv.z, acc[a][2]);
                acc[a][3] = fmaf(dv[a], xv.w, acc[a][3]);
            }
        }
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

template <int EP, int TM, int TTOK, int EJ>
int launch_route_fwd(const moe_bf16* x, const float* W_r, const float* b, int64_t T, int d,
                     int E, int k, int mode, float* logits, int32_t* idx, float* gate,
                     float* score, float* lse, double* zp, int64_t* nblocks, cudaStream_t st) {
    const int64_t nb = cdiv(T, TM);
    *nblocks = nb;
    const size_t stage = sizeof(float) * kKC * (TM + EP);
    const size_t tile = sizeof(float) * TM * (EP + 1);
    const size_t smem = stage > tile ? stage : tile;
    auto kern = route_fwd_kernel<EP, TM, TTOK, EJ>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    kern<<<(unsigned)nb, kThreads, smem, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), W_r, b,
                                               T, d, E, k, mode, logits, idx, gate, score, lse,
                                               zp);
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
    int64_t nb = 0;
#define MOE_ROUTE_ARGS x, W_r, b, T, d, E, k, mode, logits, topk_idx, topk_gate, topk_score, lse, zp, &nb, st
    if (E <= 16) rc = launch_route_fwd<16, 128, 4, 2>(MOE_ROUTE_ARGS);
    else if (E <= 32) rc = launch_route_fwd<32, 128, 4, 4>(MOE_ROUTE_ARGS);
    else if (E <= 64) rc = launch_route_fwd<64, 128, 8, 4>(MOE_ROUTE_ARGS);
    else if (E <= 128) rc = launch_route_fwd<128, 128, 8, 8>(MOE_ROUTE_ARGS);
    else rc = launch_route_fwd<256, 64, 8, 8>(MOE_ROUTE_ARGS);
#undef MOE_ROUTE_ARGS
    if (rc != MOE_OK) return rc;
    if (mode == MOE_MODE_SOFTMAX) {
        z_finalize_kernel<<<1, 32, 0, st>>>(zp, nb, T, z_coef, z_loss);
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
