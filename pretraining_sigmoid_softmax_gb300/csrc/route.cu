// Router forward (logits, top-k choice, gates, z-loss) and router backward (logit
// gradient, W_r gradient).
//
// Router: "The whole stack, in the open" (Apex-3), "What's inside", row "Fine-grained
// MoE": a sigmoid router picks the top experts and a per-expert bias balances the load
// with no loss term. KempnerForge README, "Features": softmax top-k router and router
// z-loss. Handbook summary, section 2.5: router logits in fp32.
//
// Routers of up to 128 experts run their two contractions (logits, W_r gradient) on the
// tensor cores (route_tc.cu). Wider routers use the fp32 SIMT kernels here: every output is
// one thread's sequential sum, so results are bitwise repeatable on either path.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "router.cuh"
#include "sizes.h"

namespace moe {
namespace {

constexpr int kKC = 32;                  // d-chunk per smem stage
constexpr int kThreads = 256;

__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
    return route_better(v1, e1, v2, e2);
}

__device__ __forceinline__ float sigmoid_f(float l) { return route_sigmoid(l); }

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
                v = (mode == MOE_MODE_SIGMOID) ? route_select_sigmoid(l) + bias[e] : l;
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

// One CTA of 256 threads: thread i sums partials i, i + 256, ... in order, then a fixed
// tree over the threads (the same association on every run).
__global__ void __launch_bounds__(256) z_finalize_kernel(const double* __restrict__ z_part,
                                                         int64_t nblocks, int64_t T, float z_coef,
                                                         float* __restrict__ z_loss) {
    __shared__ double red[256];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < nblocks; i += 256) s += z_part[i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) z_loss[0] = (float)((double)z_coef * red[0] / (double)T);
}

// ---------------------------------------------------------------------------- backward

// One warp per token: dense row of the logit gradient.
__global__ void __launch_bounds__(256) route_bwd_dlogits_kernel(
    const float* __restrict__ dg, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_gate, const float* __restrict__ topk_score,
    const float* __restrict__ logits, const float* __restrict__ lse,
    const float* __restrict__ extra, int64_t T, int E, int k, int mode, float z_scale,
    float* __restrict__ dlogits, __nv_bfloat16* __restrict__ dl3, int np, int64_t pstride,
    const int32_t* __restrict__ slot_to_row, float* __restrict__ dl_rows) {
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
    // with dl3, the row is also written as three bf16 pieces, piece p at dl3 + p * pstride as
    // a [T, np] matrix (zero past E)
    const int ecount = dl3 ? np : E;
    const float ds = (my_dg - gdg) / S;
    const float vs = ds * my_s * (1.f - my_s);
    if (dl_rows && lane < k) {  // sigmoid mode, no extra term: the slot's own logit gradient
        const int32_t r = slot_to_row[t * k + lane];
        if (r >= 0) dl_rows[r] = vs;
    }
    const float l_se = mode == MOE_MODE_SIGMOID ? 0.f : lse[t];
    for (int e0 = 0; e0 < ecount; e0 += 32) {  // warp-uniform trip count
        const int e = e0 + lane;
        float out = 0.f;
        if (mode == MOE_MODE_SIGMOID) {
            for (int i = 0; i < k; ++i) {
                const int ei = __shfl_sync(0xffffffffu, my_e, i);
                const float vi = __shfl_sync(0xffffffffu, vs, i);
                if (ei == e) out = vi;
            }
        } else {
            float sel = 0.f;
            for (int i = 0; i < k; ++i) {
                const int ei = __shfl_sync(0xffffffffu, my_e, i);
                const float di = __shfl_sync(0xffffffffu, my_dg, i);
                if (ei == e) sel = di;
            }
            if (e < E) {
                const float p = expf(logits[t * E + e] - l_se);
                out = p * (sel - gdg) + z_scale * l_se * p;
            }
        }
        if (e < E) {
            if (extra) out += extra[t * E + e];
            dlogits[t * E + e] = out;
        }
        if (dl3) {
            __nv_bfloat16 p0, p1, p2;
            split3_bf16(e < E ? out : 0.f, p0, p1, p2);
            const int64_t i = t * np + e;
            dl3[i] = p0;
            dl3[pstride + i] = p1;
            dl3[2 * pstride + i] = p2;
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

// ------------------------------------------------------------------ balancing losses
// Per-token probabilities pi over all experts: softmax of the logits, or the sigmoid
// scores normalised to sum 1. Per (sequence, chunk of kAuxChunk tokens): column sums of pi
// and chosen-expert counts, one thread per expert summing its tokens in order.
constexpr int kAuxChunk = 256;

__global__ void __launch_bounds__(kThreads) aux_partial_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ topk_idx, int64_t seq_len,
    int E, int k, int mode, float* __restrict__ Ppart, int32_t* __restrict__ Cpart) {
    __shared__ float nrm_a[kAuxChunk];  // softmax: max; sigmoid: sum of scores
    __shared__ float nrm_b[kAuxChunk];  // softmax: sum of exp(l - max)
    const int64_t s = blockIdx.x, c = blockIdx.y;
    const int64_t t0 = s * seq_len + c * kAuxChunk;
    const int64_t n = min((int64_t)kAuxChunk, seq_len - c * kAuxChunk);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int r = warp; r < n; r += kThreads / 32) {
        const float* lg = logits + (t0 + r) * E;
        float a = (mode == MOE_MODE_SOFTMAX) ? -INFINITY : 0.f, b = 0.f;
        if (mode == MOE_MODE_SOFTMAX) {
            for (int e = lane; e < E; e += 32) a = fmaxf(a, lg[e]);
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            for (int e = lane; e < E; e += 32) b += expf(lg[e] - a);
            for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
        } else {
            for (int e = lane; e < E; e += 32) a += sigmoid_f(lg[e]);
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        }
        if (lane == 0) {
            nrm_a[r] = a;
            nrm_b[r] = b;
        }
    }
    __syncthreads();
    const int e = threadIdx.x;
    if (e >= E) return;
    float P = 0.f;
    int32_t cnt = 0;
    for (int r = 0; r < n; ++r) {
        const float l = logits[(t0 + r) * E + e];
        P += (mode == MOE_MODE_SOFTMAX) ? expf(l - nrm_a[r]) / nrm_b[r] : sigmoid_f(l) / nrm_a[r];
        const int32_t* id = topk_idx + (t0 + r) * k;
        for (int i = 0; i < k; ++i) cnt += (id[i] == e);
    }
    const int64_t slot = (s * gridDim.y + c) * E + e;
    Ppart[slot] = P;
    Cpart[slot] = cnt;
}

// One CTA: f and P per expert and per sequence, the two losses, and the f values the
// backward needs (aux_f[e] = f_e, aux_f[E + s E + e] = f[s,e]).
__global__ void __launch_bounds__(kThreads) aux_final_kernel(
    const float* __restrict__ Ppart, const int32_t* __restrict__ Cpart, int64_t B, int64_t C,
    int64_t seq_len, int E, int k, float switch_coef, float seq_coef, float* __restrict__ aux_f,
    float* __restrict__ aux_loss) {
    __shared__ double sw[kThreads], sq[kThreads];
    const int e = threadIdx.x;
    double sw_e = 0.0, sq_e = 0.0;
    if (e < E) {
        const double T = (double)B * (double)seq_len;
        double Psum = 0.0, csum = 0.0;
        for (int64_t s = 0; s < B; ++s) {
            double Ps = 0.0, cs = 0.0;
            for (int64_t c = 0; c < C; ++c) {
                Ps += Ppart[(s * C + c) * E + e];
                cs += Cpart[(s * C + c) * E + e];
            }
            const double fs = (double)E * cs / ((double)k * (double)seq_len);
            aux_f[E + s * E + e] = (float)fs;
            sq_e += fs * (Ps / (double)seq_len);
            Psum += Ps;
            csum += cs;
        }
        const double f = csum / (T * (double)k);
        aux_f[e] = (float)f;
        sw_e = f * (Psum / T);
    }
    sw[e] = sw_e;
    sq[e] = sq_e;
    __syncthreads();
    if (e == 0) {
        double a = 0.0, b = 0.0;
        for (int j = 0; j < E; ++j) {
            a += sw[j];
            b += sq[j];
        }
        aux_loss[0] = (float)((double)switch_coef * (double)E * a);
        aux_loss[1] = (float)((double)seq_coef * b / (double)B);
    }
}

// Gradient of the two losses with respect to the logits, one warp per token:
// g_e = switch_coef E f_e / T + seq_coef f[s,e] / (B L); softmax: pi (g - <g, pi>);
// sigmoid: (g - <g, pi>) / S * s (1 - s).
__global__ void __launch_bounds__(256) aux_bwd_kernel(
    const float* __restrict__ logits, const float* __restrict__ aux_f, int64_t T, int E,
    int64_t seq_len, int mode, float switch_coef, float seq_coef, float* __restrict__ dl) {
    const int lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (t >= T) return;  // whole warp
    const int64_t B = T / seq_len, s = t / seq_len;
    const float* lg = logits + t * E;
    float a = (mode == MOE_MODE_SOFTMAX) ? -INFINITY : 0.f, b = 0.f;
    if (mode == MOE_MODE_SOFTMAX) {
        for (int e = lane; e < E; e += 32) a = fmaxf(a, lg[e]);
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        for (int e = lane; e < E; e += 32) b += expf(lg[e] - a);
        for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
    } else {
        for (int e = lane; e < E; e += 32) a += sigmoid_f(lg[e]);
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    }
    const float c_sw = switch_coef * (float)E / (float)T;
    const float c_sq = seq_coef / ((float)B * (float)seq_len);
    float gpi = 0.f;
    for (int e = lane; e < E; e += 32) {
        const float l = lg[e];
        const float pi = (mode == MOE_MODE_SOFTMAX) ? expf(l - a) / b : sigmoid_f(l) / a;
        gpi += (c_sw * aux_f[e] + c_sq * aux_f[E + s * E + e]) * pi;
    }
    for (int o = 16; o > 0; o >>= 1) gpi += __shfl_xor_sync(0xffffffffu, gpi, o);
    for (int e = lane; e < E; e += 32) {
        const float l = lg[e];
        const float g = c_sw * aux_f[e] + c_sq * aux_f[E + s * E + e];
        float v;
        if (mode == MOE_MODE_SOFTMAX) {
            v = expf(l - a) / b * (g - gpi);
        } else {
            const float sg = sigmoid_f(l);
            v = (g - gpi) / a * sg * (1.f - sg);
        }
        dl[t * E + e] = v;
    }
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
    const int epad = route_tc_epad(E);
    int64_t nzp = route_blocks(T);
    if (4 * route_tc_tiles(T) > nzp) nzp = 4 * route_tc_tiles(T);
    double* zp = wc.take<double>(nzp);
    __nv_bfloat16* w3 = epad ? wc.take<__nv_bfloat16>((size_t)3 * epad * d) : nullptr;
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    int rc;
    int64_t nb = 0;
    if (epad) {
        rc = launch_route_logits_tc(reinterpret_cast<const __nv_bfloat16*>(x), W_r, b, T, d, E, k,
                                    mode, logits, topk_idx, topk_gate, topk_score, lse, zp, &nb,
                                    w3, st);
    } else {
        rc = launch_route_fwd<256, 64, 8, 8>(x, W_r, b, T, d, E, k, mode, logits, topk_idx,
                                             topk_gate, topk_score, lse, zp, &nb, st);
    }
    if (rc != MOE_OK) return rc;
    if (mode == MOE_MODE_SOFTMAX) {
        z_finalize_kernel<<<1, 256, 0, st>>>(zp, nb, T, z_coef, z_loss);
        rc = launch_status();
    }
    return rc;
}

extern "C" int moe_route_bwd(const float* dg, const moe_bf16* x, const int32_t* topk_idx,
                             const float* topk_gate, const float* topk_score,
                             const float* logits, const float* lse, const float* dlogits_extra,
                             int64_t T, int d, int E, int k, int mode, float z_coef,
                             float* dlogits, float* dW_r, const int32_t* slot_to_row,
                             float* dl_rows, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!dg || !x || !topk_idx || !topk_gate || !topk_score || !dlogits || !dW_r)
        return MOE_ERR_INVALID_ARG;
    if ((slot_to_row == nullptr) != (dl_rows == nullptr)) return MOE_ERR_INVALID_ARG;
    if (dl_rows && (mode != MOE_MODE_SIGMOID || dlogits_extra)) return MOE_ERR_INVALID_ARG;
    if (T <= 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_MODE_SIGMOID && mode != MOE_MODE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_MODE_SOFTMAX && (!logits || !lse)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(dW_r)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    WsCarver wc(ws, ws_bytes);
    const int np = route_tc_np(E);
    int64_t nsplit = route_bwd_splits(T);
    if (np && route_tc_splits_max(T) > nsplit) nsplit = route_tc_splits_max(T);
    float* part = wc.take<float>((size_t)nsplit * E * d);
    __nv_bfloat16* dl3 = nullptr;
    // three pieces, each [T, np], each starting on a 256-byte boundary (pstride elements apart)
    const int64_t pstride = (T * np + 127) / 128 * 128;
    if (np) dl3 = wc.take<__nv_bfloat16>((size_t)3 * pstride);
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const float z_scale = 2.0f * z_coef / (float)T;
    route_bwd_dlogits_kernel<<<(unsigned)cdiv(T, 8), 256, 0, st>>>(
        dg, topk_idx, topk_gate, topk_score, logits, lse, dlogits_extra, T, E, k, mode, z_scale,
        dlogits, dl3, np, pstride, slot_to_row, dl_rows);
    if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    if (np) {
        int rc = launch_route_dwr_tc(reinterpret_cast<const __nv_bfloat16*>(x), dl3, pstride, T,
                                     d, E, part, &nsplit, st);
        if (rc != MOE_OK) return rc;
    } else {
        dim3 grid(d / kBwTJ, (unsigned)cdiv(E, kBwTE), (unsigned)nsplit);
        route_bwd_dwr_kernel<<<grid, 256, 0, st>>>(
            dlogits, reinterpret_cast<const __nv_bfloat16*>(x), T, d, E, part);
        if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    }
    const int64_t n = (int64_t)E * d;
    route_bwd_reduce_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(part, nsplit, n, dW_r);
    return launch_status();
}

extern "C" int moe_router_dx(const float* dlogits, const float* W_r, int64_t T, int d, int E,
                             float* dx_r, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!dlogits || !W_r || !dx_r) return MOE_ERR_INVALID_ARG;
    if (T <= 0 || d <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    const int np = route_tc_np(E);
    if (!np || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(dx_r) || !aligned16(W_r)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    WsCarver wc(ws, ws_bytes);
    const int64_t pstride = (T * np + 127) / 128 * 128;
    __nv_bfloat16* dl2 = wc.take<__nv_bfloat16>((size_t)2 * pstride);
    __nv_bfloat16* w3 = wc.take<__nv_bfloat16>((size_t)3 * np * d);
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    return launch_router_dx_tc(dlogits, W_r, T, d, E, dl2, pstride, w3, dx_r, (cudaStream_t)stream);
}

extern "C" int moe_aux_loss(const float* logits, const int32_t* topk_idx, int64_t T, int E, int k,
                            int mode, int64_t seq_len, float switch_coef, float seq_coef,
                            float* aux_loss, float* aux_f, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
    if (!logits || !topk_idx || !aux_loss || !aux_f) return MOE_ERR_INVALID_ARG;
    if (T <= 0 || E <= 0 || k <= 0 || seq_len <= 0 || T % seq_len != 0) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_MODE_SIGMOID && mode != MOE_MODE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32) return MOE_ERR_UNSUPPORTED;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    const int64_t B = T / seq_len, C = cdiv(seq_len, kAuxChunk);
    WsCarver wc(ws, ws_bytes);
    float* Ppart = wc.take<float>((size_t)B * C * E);
    int32_t* Cpart = wc.take<int32_t>((size_t)B * C * E);
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    aux_partial_kernel<<<dim3((unsigned)B, (unsigned)C), kThreads, 0, st>>>(
        logits, topk_idx, seq_len, E, k, mode, Ppart, Cpart);
    aux_final_kernel<<<1, kThreads, 0, st>>>(Ppart, Cpart, B, C, seq_len, E, k, switch_coef,
                                              seq_coef, aux_f, aux_loss);
    return launch_status();
}

extern "C" int moe_aux_loss_bwd(const float* logits, const float* aux_f, int64_t T, int E, int mode,
                                int64_t seq_len, float switch_coef, float seq_coef,
                                float* dlogits_aux, moe_stream_t stream) {
    if (!logits || !aux_f || !dlogits_aux) return MOE_ERR_INVALID_ARG;
    if (T <= 0 || E <= 0 || seq_len <= 0 || T % seq_len != 0) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_MODE_SIGMOID && mode != MOE_MODE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    aux_bwd_kernel<<<(unsigned)cdiv(T, 8), 256, 0, (cudaStream_t)stream>>>(
        logits, aux_f, T, E, seq_len, mode, switch_coef, seq_coef, dlogits_aux);
    return launch_status();
}
