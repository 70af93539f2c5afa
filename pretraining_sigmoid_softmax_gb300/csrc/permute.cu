// Token dispatch (histogram, scan, stable expert-major permutation, 16-byte row copies),
// the gate-weighted combine, their backward passes and the aux-loss-free bias update.
//
// Dispatch and combine: handbook summary ("How to train a large-scale Mixture-of-Experts
// model from scratch"), section 2.5: tokens must be sent to the chosen experts and each
// expert's output returned. Bias update: "The whole stack, in the open" (Apex-3), "What's
// inside", row "Fine-grained MoE": a per-expert bias balances the load without a loss term.
//
// These steps move bytes: every row copy is a warp-wide run of 16-byte vectors so each
// memory instruction touches whole 512-byte spans. Counting uses integer atomics in shared
// memory only (order-independent); every floating-point sum has a fixed order.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "fp8.cuh"
#include "sizes.h"

namespace moe {
namespace {

constexpr int kHistThreads = kHistTokensPerCta;     // one token per thread
constexpr int kScatterThreads = kHistTokensPerCta;  // one token per thread
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kScanThreads = 1024;                  // one warp per expert at a time
constexpr int kWarpsPerCta = 8;                     // warp-per-token kernels

// Expert of slot (t, i), or -1 when the index is out of range or repeats an earlier slot
// of the same token (both are input errors; the slot is dropped).
__device__ __forceinline__ int valid_expert(const int32_t* __restrict__ idx, int64_t t, int k,
                                            int i, int E) {
    const int e = idx[t * k + i];
    if (e < 0 || e >= E) return -1;
    for (int j = 0; j < i; ++j)
        if (idx[t * k + j] == e) return -1;
    return e;
}

// Per chunk of kHistTokensPerCta tokens, the number of slots of each expert, stored expert
// major: block_counts[e * nblocks + chunk].
__global__ void __launch_bounds__(kHistThreads) hist_kernel(const int32_t* __restrict__ idx,
                                                            int64_t T, int E, int k,
                                                            int32_t* __restrict__ block_counts,
                                                            int* status) {
    __shared__ int cnt[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += kHistThreads) cnt[e] = 0;
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * kHistTokensPerCta + threadIdx.x;
    if (t < T) {
        for (int i = 0; i < k; ++i) {
            const int e = valid_expert(idx, t, k, i, E);
            if (e >= 0) atomicAdd(&cnt[e], 1);
            else record_error(status, MOE_ERR_BAD_INDEX, 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kHistThreads)
        block_counts[(int64_t)e * gridDim.x + blockIdx.x] = cnt[e];
}

// One CTA: per expert, the running sums over the chunks (block bases), then the counts, the
// unpadded offsets and the 128-row padded segment offsets. Warp w takes experts w, w + 32,
// ...; for an expert its lanes own consecutive runs of chunks: each sums its run, an
// exclusive warp scan of those sums gives each run's base, and a second pass writes the
// chunk bases. Integer sums: the result does not depend on the grouping.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(
    const int32_t* __restrict__ block_counts, int64_t nblocks, int E,
    int32_t* __restrict__ block_base, int32_t* __restrict__ counts, int64_t* __restrict__ offsets,
    int64_t* __restrict__ row_offsets) {
    __shared__ int32_t c_sh[kMaxExperts];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t per = (nblocks + 31) / 32;
    const int64_t b_lo = lane * per < nblocks ? lane * per : nblocks;
    const int64_t b_hi = b_lo + per < nblocks ? b_lo + per : nblocks;
    for (int e = warp; e < E; e += kScanThreads / 32) {
        const int32_t* src = block_counts + (int64_t)e * nblocks;
        int32_t* dst = block_base + (int64_t)e * nblocks;
        int32_t sum = 0;
        int64_t b = b_lo;
        for (; b + 4 <= b_hi; b += 4) sum += (src[b] + src[b + 1]) + (src[b + 2] + src[b + 3]);
        for (; b < b_hi; ++b) sum += src[b];
        int32_t incl = sum;  // inclusive scan of the lanes' run sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int32_t run = incl - sum;
        for (b = b_lo; b < b_hi; ++b) {
            const int32_t v = src[b];
            dst[b] = run;
            run += v;
        }
        if (lane == 31) c_sh[e] = incl;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kScanThreads) counts[e] = c_sh[e];
    if (threadIdx.x == 0) {
        int64_t o = 0, ro = 0;
        for (int j = 0; j < E; ++j) {
            offsets[j] = o;
            row_offsets[j] = ro;
            o += c_sh[j];
            ro += (c_sh[j] + MOE_ROW_ALIGN - 1) / MOE_ROW_ALIGN * MOE_ROW_ALIGN;
        }
        offsets[E] = o;
        row_offsets[E] = ro;
    }
}

// The padding kernels run kPadSplit CTAs per expert (grid E x kPadSplit), each taking a
// strided share of the expert's padding rows.
constexpr int kPadSplit = 16;

// Padding rows of expert e's segment, share `split` of kPadSplit: perm_token = -1, a zero row
// of buf and (optionally) a zero row gate.
__device__ __forceinline__ void pad_rows_share(const int64_t* __restrict__ row_offsets,
                                               const int32_t* __restrict__ counts, int d,
                                               int32_t* __restrict__ perm_token,
                                               __nv_bfloat16* __restrict__ buf,
                                               float* __restrict__ row_gate, int e, int split) {
    const int64_t lo = row_offsets[e] + counts[e], hi = row_offsets[e + 1];
    const int vec_per_row = d / 8;
    for (int64_t i = (int64_t)split * blockDim.x + threadIdx.x; i < (hi - lo) * vec_per_row;
         i += (int64_t)kPadSplit * blockDim.x) {
        const int64_t r = lo + i / vec_per_row;
        const int c = (int)(i % vec_per_row);
        reinterpret_cast<uint4*>(buf + r * d)[c] = make_uint4(0, 0, 0, 0);
        if (c == 0) {
            if (perm_token) perm_token[r] = -1;
            if (row_gate) row_gate[r] = 0.f;
        }
    }
}

// Zero the padding rows of expert e's segment, found as the trailing rows with perm_token < 0
// (share `split` of kPadSplit).
__device__ __forceinline__ void zero_pad_rows_share(const int64_t* __restrict__ row_offsets,
                                                    const int32_t* __restrict__ perm_token, int d,
                                                    __nv_bfloat16* __restrict__ buf, int e,
                                                    int split) {
    const int64_t hi = row_offsets[e + 1];
    int64_t lo = row_offsets[e];
    if (hi - lo > MOE_ROW_ALIGN - 1) lo = hi - (MOE_ROW_ALIGN - 1);
    const int vec_per_row = d / 8;
    for (int64_t i = (int64_t)split * blockDim.x + threadIdx.x; i < (hi - lo) * vec_per_row;
         i += (int64_t)kPadSplit * blockDim.x) {
        const int64_t r = lo + i / vec_per_row;
        if (perm_token[r] < 0)
            reinterpret_cast<uint4*>(buf + r * d)[i % vec_per_row] = make_uint4(0, 0, 0, 0);
    }
}

// Stable ranks: within a chunk of kHistTokensPerCta tokens, warp w owns tokens [32 w, 32 w +
// 32). Row of (t, i) = row_offsets[e] + chunk base of e + warp base of e + rank within warp.
// Blocks past the nblocks chunks pad the segments instead (kPadSplit per expert: perm_token
// -1, zero rows of X_perm and of the row gates). With row_gate, each slot's gate is copied to
// its row as well (the gate folded into the expert).
__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(
    const int32_t* __restrict__ idx, int64_t T, int E, int k, int64_t nblocks,
    const int32_t* __restrict__ block_base, const int64_t* __restrict__ row_offsets,
    const int32_t* __restrict__ counts, int d, int32_t* __restrict__ perm_token,
    int32_t* __restrict__ slot_to_row, __nv_bfloat16* __restrict__ X_perm,
    const float* __restrict__ gate, float* __restrict__ row_gate) {
    if (blockIdx.x >= nblocks) {  // block-uniform: no barrier below is reached
        const int p = (int)(blockIdx.x - nblocks);
        pad_rows_share(row_offsets, counts, d, perm_token, X_perm, row_gate, p / kPadSplit,
                       p % kPadSplit);
        return;
    }
    __shared__ int32_t wcnt[kScatterWarps][kMaxExperts];
    __shared__ uint32_t wmask[kScatterWarps][kMaxExperts];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < kScatterWarps * kMaxExperts; i += kScatterThreads) {
        (&wcnt[0][0])[i] = 0;
        (&wmask[0][0])[i] = 0u;
    }
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * kHistTokensPerCta + tid;
    const bool live = t < T;
    if (live)
        for (int i = 0; i < k; ++i) {
            const int e = valid_expert(idx, t, k, i, E);
            if (e >= 0) {
                atomicAdd(&wcnt[warp][e], 1);
                atomicOr(&wmask[warp][e], 1u << lane);
            }
        }
    __syncthreads();
    for (int e = tid; e < E; e += kScatterThreads) {  // exclusive scan over warps, per expert
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < kScatterWarps; ++w) {
            const int32_t c = wcnt[w][e];
            wcnt[w][e] = run;
            run += c;
        }
    }
    __syncthreads();
    if (!live) return;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int i = 0; i < k; ++i) {
        const int e = valid_expert(idx, t, k, i, E);
        int32_t row = -1;
        if (e >= 0) {
            const int rank = __popc(wmask[warp][e] & lt_mask);
            row = (int32_t)(row_offsets[e] + block_base[(int64_t)e * nblocks + blockIdx.x] +
                            wcnt[warp][e] + rank);
            perm_token[row] = (int32_t)t;
            if (row_gate) row_gate[row] = gate[t * k + i];
        }
        slot_to_row[t * k + i] = row;
    }
}

// Copy x[t] to the k rows of token t: one warp per token, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_kernel(const __nv_bfloat16* __restrict__ x,
                                                     const int32_t* __restrict__ slot_to_row,
                                                     int64_t T, int d, int k,
                                                     __nv_bfloat16* __restrict__ X_perm) {
    const int lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + threadIdx.x / 32;
    if (t >= T) return;
    int32_t my_row = -1;
    if (lane < k) my_row = slot_to_row[t * k + lane];
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    const int nvec = d / 8;
    for (int c0 = 0; c0 < nvec; c0 += 32) {  // warp-uniform trip count
        const int c = c0 + lane;
        const bool in = c < nvec;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (in) v = src[c];
        for (int i = 0; i < k; ++i) {
            const int32_t row = __shfl_sync(0xffffffffu, my_row, i);
            if (in && row >= 0) reinterpret_cast<uint4*>(X_perm + (int64_t)row * d)[c] = v;
        }
    }
}

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4 v, float g) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[2 * q] = fmaf(g, bf16_lo(w[q]), acc[2 * q]);
        acc[2 * q + 1] = fmaf(g, bf16_hi(w[q]), acc[2 * q + 1]);
    }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(w[q]);
        acc[2 * q + 1] += bf16_hi(w[q]);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                      pack_bf16x2(a[6], a[7]));
}

// out[t] = sum_i g[t,i] * Y_perm[row(t,i)] (+ Y_shared[t]); fp32, slot order, shared last.
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ Y_perm,
                                                      const float* __restrict__ gate,
                                                      const int32_t* __restrict__ slot_to_row,
                                                      const __nv_bfloat16* __restrict__ Y_sh,
                                                      int64_t T, int d, int k,
                                                      __nv_bfloat16* __restrict__ out) {
    const int lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + threadIdx.x / 32;
    if (t >= T) return;
    int32_t my_row = -1;
    float my_g = 0.f;
    if (lane < k) {
        my_row = slot_to_row[t * k + lane];
        my_g = gate ? gate[t * k + lane] : 1.0f;  // no gates: rows already carry them
    }
    const int nvec = d / 8;
    for (int c0 = 0; c0 < nvec; c0 += 32) {  // warp-uniform trip count
        const int c = c0 + lane;
        const bool in = c < nvec;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < k; ++i) {
            const int32_t row = __shfl_sync(0xffffffffu, my_row, i);
            const float g = __shfl_sync(0xffffffffu, my_g, i);
            if (in && row >= 0)
                acc_bf16x8(acc, reinterpret_cast<const uint4*>(Y_perm + (int64_t)row * d)[c], g);
        }
        if (!in) continue;
        if (Y_sh) add_bf16x8(acc, reinterpret_cast<const uint4*>(Y_sh + t * d)[c]);
        reinterpret_cast<uint4*>(out + t * d)[c] = pack8(acc);
    }
}

// dY_perm[row(t,i)] = bf16(g[t,i] * dY[t]); dg[t,i] = <dY[t], Y_perm[row(t,i)]>. Without
// gates the rows are plain copies of dY[t]; without Y_perm no dg is formed.
// CODES: also the E4M3 codes and scale of every written row, equal to what
// moe_quantize_rows_fp8 of dY_perm gives: each row is bf16(g dY[t]), a monotone function of
// dY[t] for g >= 0, so its amax is bf16(g amax|dY[t]|), known before the row is written.
template <int KMAX, bool CODES = false>
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const __nv_bfloat16* __restrict__ dY, const __nv_bfloat16* __restrict__ Y_perm,
    const float* __restrict__ gate, const int32_t* __restrict__ slot_to_row, int64_t T, int d,
    int k, __nv_bfloat16* __restrict__ dY_perm, float* __restrict__ dg, int64_t tok_blocks,
    const int64_t* __restrict__ row_offsets, const int32_t* __restrict__ perm_token,
    uint8_t* __restrict__ dYq = nullptr, float* __restrict__ sdY = nullptr) {
    if (blockIdx.x >= tok_blocks) {  // the segments' padding rows of dY_perm, kPadSplit per expert
        const int p = (int)(blockIdx.x - tok_blocks);
        zero_pad_rows_share(row_offsets, perm_token, d, dY_perm, p / kPadSplit, p % kPadSplit);
        return;
    }
    const int lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + threadIdx.x / 32;
    if (t >= T) return;
    int32_t my_row = -1;
    float my_g = 0.f;
    if (lane < k) {
        my_row = slot_to_row[t * k + lane];
        my_g = gate ? gate[t * k + lane] : 1.0f;
    }
    float sc_s[CODES ? KMAX : 1], sc_rs[CODES ? KMAX : 1];  // each slot row's scale
    if constexpr (CODES) {
        float m = 0.f;
        for (int c = lane; c < d / 8; c += 32) m = amax8(reinterpret_cast<const uint4*>(dY + t * d)[c], m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const Fp8Scale sc(__bfloat162float(__float2bfloat16_rn(my_g * m)));
        if (lane < k && my_row >= 0) sdY[my_row] = sc.s;
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            sc_s[i] = __shfl_sync(0xffffffffu, sc.s, i);
            sc_rs[i] = __shfl_sync(0xffffffffu, sc.rs, i);
        }
    }
    float dot[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) dot[i] = 0.f;
    const int nvec = d / 8;
    for (int c0 = 0; c0 < nvec; c0 += 32) {  // warp-uniform trip count
        const int c = c0 + lane;
        const bool in = c < nvec;
        uint4 dv = make_uint4(0, 0, 0, 0);
        if (in) dv = reinterpret_cast<const uint4*>(dY + t * d)[c];
        const uint32_t w[4] = {dv.x, dv.y, dv.z, dv.w};
        float dyf[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            dyf[2 * q] = bf16_lo(w[q]);
            dyf[2 * q + 1] = bf16_hi(w[q]);
        }
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            if (i < k) {
                const int32_t row = __shfl_sync(0xffffffffu, my_row, i);
                const float g = __shfl_sync(0xffffffffu, my_g, i);
                if (in && row >= 0) {
                    if (Y_perm) {
                        const uint4 yv = reinterpret_cast<const uint4*>(Y_perm + (int64_t)row * d)[c];
                        const uint32_t y[4] = {yv.x, yv.y, yv.z, yv.w};
                        float s = dot[i];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            s = fmaf(dyf[2 * q], bf16_lo(y[q]), s);
                            s = fmaf(dyf[2 * q + 1], bf16_hi(y[q]), s);
                        }
                        dot[i] = s;
                    }
                    float o[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) o[q] = g * dyf[q];
                    reinterpret_cast<uint4*>(dY_perm + (int64_t)row * d)[c] = pack8(o);
                    if constexpr (CODES) {  // the codes of the bf16 values just stored
                        Fp8Scale sc = Fp8Scale::of(sc_s[i]);
                        sc.rs = sc_rs[i];
#pragma unroll
                        for (int q = 0; q < 8; ++q) o[q] = __bfloat162float(__float2bfloat16_rn(o[q]));
                        reinterpret_cast<uint2*>(dYq + (int64_t)row * d)[c] = codes8f(o, sc);
                    }
                }
            }
        }
    }
    if (!dg) return;
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
        if (i < k) {
            float s = dot[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) dg[t * k + i] = s;
        }
    }
}

// row_gate[slot_to_row[s]] = gate[s] for every slot s (rows were zeroed first).
__global__ void row_gates_kernel(const float* __restrict__ gate, const int32_t* __restrict__ slot_to_row,
                                 int64_t n, int64_t rows, float* __restrict__ row_gate) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int32_t r = slot_to_row[i];
    if (r >= 0 && r < rows) row_gate[r] = gate[i];
}

// dg[s] = sum_j part[slot_to_row[s], j], j = 0 .. nparts-1 in order.
__global__ void gate_grad_kernel(const float* __restrict__ part, int nparts,
                                 const int32_t* __restrict__ slot_to_row, int64_t n,
                                 float* __restrict__ dg) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int32_t r = slot_to_row[i];
    float s = 0.f;
    if (r >= 0) {
        const float* p = part + (int64_t)r * nparts;
        for (int j = 0; j < nparts; ++j) s += p[j];
    }
    dg[i] = s;
}

// dx[t] = sum_i dX_perm[slot_to_row[t,i]] + dx_shared[t] + sum_e dlogits[t,e] W_r[e].
// One warp per token. The token's nonzero router terms (k in sigmoid mode, E in softmax
// mode) are listed once, in expert order, in the warp's shared-memory slice; the row loop
// then touches only those rows of W_r.
template <int KMAX, bool DXR>
__global__ void __launch_bounds__(256) permute_bwd_kernel(
    const __nv_bfloat16* __restrict__ dX_perm, const int32_t* __restrict__ slot_to_row,
    const __nv_bfloat16* __restrict__ dx_sh, const float* __restrict__ dlogits,
    const float* __restrict__ W_r, const float* __restrict__ dx_r, int64_t T, int d, int E,
    int k, __nv_bfloat16* __restrict__ dx) {
    __shared__ int s_e[kWarpsPerCta][kMaxExperts];
    __shared__ float s_g[kWarpsPerCta][kMaxExperts];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    if (t >= T) return;  // whole warp
    int32_t my_row = -1;
    if (lane < k) my_row = slot_to_row[t * k + lane];
    int32_t rows[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) rows[i] = __shfl_sync(0xffffffffu, my_row, i);
    int n = 0;
    if (dlogits) {
        for (int e0 = 0; e0 < E; e0 += 32) {  // warp-uniform trip count
            const int e = e0 + lane;
            const float g = e < E ? dlogits[t * E + e] : 0.f;
            const unsigned m = __ballot_sync(0xffffffffu, g != 0.f);
            if (g != 0.f) {
                const int pos = n + __popc(m & ((1u << lane) - 1u));
                s_e[warp][pos] = e;
                s_g[warp][pos] = g;
            }
            n += __popc(m);
        }
        __syncwarp();
    }
    const int nvec = d / 8;
    for (int c = lane; c < nvec; c += 32) {  // no warp collectives inside
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            if (i < k && rows[i] >= 0)
                add_bf16x8(acc, reinterpret_cast<const uint4*>(dX_perm + (int64_t)rows[i] * d)[c]);
        }
        if (dx_sh) add_bf16x8(acc, reinterpret_cast<const uint4*>(dx_sh + t * d)[c]);
        if constexpr (DXR) {  // the router's term, formed beforehand (moe_router_dx)
            const float4* r = reinterpret_cast<const float4*>(dx_r + t * d + c * 8);
            const float4 a = r[0], b = r[1];
            acc[0] += a.x;
            acc[1] += a.y;
            acc[2] += a.z;
            acc[3] += a.w;
            acc[4] += b.x;
            acc[5] += b.y;
            acc[6] += b.z;
            acc[7] += b.w;
        }
        for (int j = 0; j < n; ++j) {
            const float g = s_g[warp][j];
            const float4* w = reinterpret_cast<const float4*>(W_r + (int64_t)s_e[warp][j] * d + c * 8);
            const float4 a = __ldg(w), b = __ldg(w + 1);
            acc[0] = fmaf(g, a.x, acc[0]);
            acc[1] = fmaf(g, a.y, acc[1]);
            acc[2] = fmaf(g, a.z, acc[2]);
            acc[3] = fmaf(g, a.w, acc[3]);
            acc[4] = fmaf(g, b.x, acc[4]);
            acc[5] = fmaf(g, b.y, acc[5]);
            acc[6] = fmaf(g, b.z, acc[6]);
            acc[7] = fmaf(g, b.w, acc[7]);
        }
        reinterpret_cast<uint4*>(dx + t * d)[c] = pack8(acc);
    }
}

__global__ void bias_update_kernel(const int32_t* __restrict__ counts, int E, int64_t T, int k,
                                   float gamma, float* __restrict__ b) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    // sign(T*k/E - c) == sign(T*k - E*c), exact in integers
    const int64_t diff = T * (int64_t)k - (int64_t)E * counts[e];
    const float sgn = diff > 0 ? 1.f : (diff < 0 ? -1.f : 0.f);
    b[e] = b[e] + gamma * sgn;
}

// Proportional variant: b[e] += gamma * (T*k - E*c) / (T*k). The ratio is formed in fp64
// from exact integers and rounded once to fp32; the product and the sum are single fp32
// roundings (no fused multiply-add).
__global__ void bias_update_proportional_kernel(const int32_t* __restrict__ counts, int E,
                                                int64_t T, int k, float gamma,
                                                float* __restrict__ b) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const double n = (double)T * (double)k;
    const float r = (float)((n - (double)E * (double)counts[e]) / n);
    b[e] = __fadd_rn(b[e], __fmul_rn(gamma, r));
}

inline unsigned warp_grid(int64_t T) { return (unsigned)cdiv(T, kWarpsPerCta); }

template <bool DXR>
void launch_permute_bwd(unsigned grid, cudaStream_t st, const __nv_bfloat16* a,
                        const int32_t* slot_to_row, const __nv_bfloat16* sh, const float* dlogits,
                        const float* W_r, const float* dx_router, int64_t T, int d, int E, int k,
                        __nv_bfloat16* o) {
    if (k <= 2) permute_bwd_kernel<2, DXR><<<grid, 256, 0, st>>>(a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
    else if (k <= 4) permute_bwd_kernel<4, DXR><<<grid, 256, 0, st>>>(a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
    else if (k <= 8) permute_bwd_kernel<8, DXR><<<grid, 256, 0, st>>>(a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
    else if (k <= 16) permute_bwd_kernel<16, DXR><<<grid, 256, 0, st>>>(a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
    else permute_bwd_kernel<32, DXR><<<grid, 256, 0, st>>>(a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
}

bool shape_ok(int64_t T, int d, int E, int k) {
    return T > 0 && d > 0 && E > 0 && k > 0;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute(const int32_t* topk_idx, const moe_bf16* x, int64_t T, int d, int E,
                           int k, int32_t* counts, int64_t* offsets, int64_t* row_offsets,
                           int32_t* perm_token, int32_t* slot_to_row, moe_bf16* X_perm,
                           const float* topk_gate, float* row_gate, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
    if (!topk_idx || !x || !counts || !offsets || !row_offsets || !perm_token || !slot_to_row ||
        !X_perm)
        return MOE_ERR_INVALID_ARG;
    if ((topk_gate == nullptr) != (row_gate == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(T, d, E, k)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(X_perm)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    int* status = device_status_word();
    if (!status) return MOE_ERR_LAUNCH;
    const int64_t nb = hist_blocks(T);
    WsCarver wc(ws, ws_bytes);
    int32_t* bcounts = wc.take<int32_t>(nb * E);
    int32_t* bbase = wc.take<int32_t>(nb * E);
    if (!ws || !wc.ok()) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    hist_kernel<<<(unsigned)nb, kHistThreads, 0, st>>>(topk_idx, T, E, k, bcounts, status);
    scan_kernel<<<1, kScanThreads, 0, st>>>(bcounts, nb, E, bbase, counts, offsets, row_offsets);
    scatter_kernel<<<(unsigned)(nb + (int64_t)E * kPadSplit), kScatterThreads, 0, st>>>(
        topk_idx, T, E, k, nb, bbase, row_offsets, counts, d, perm_token, slot_to_row,
        reinterpret_cast<__nv_bfloat16*>(X_perm), topk_gate, row_gate);
    gather_kernel<<<warp_grid(T), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x),
                                                slot_to_row, T, d, k,
                                                reinterpret_cast<__nv_bfloat16*>(X_perm));
    return launch_status();
}

extern "C" int moe_combine(const moe_bf16* Y_perm, const float* topk_gate,
                           const int32_t* slot_to_row, const moe_bf16* Y_shared, int64_t T,
                           int d, int k, moe_bf16* out, moe_stream_t stream) {
    if (!Y_perm || !slot_to_row || !out) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(T, d, 1, k)) return MOE_ERR_INVALID_ARG;
    if (k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(Y_perm) || !aligned16(out) || (Y_shared && !aligned16(Y_shared)))
        return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    combine_kernel<<<warp_grid(T), 256, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(Y_perm), topk_gate, slot_to_row,
        reinterpret_cast<const __nv_bfloat16*>(Y_shared), T, d, k,
        reinterpret_cast<__nv_bfloat16*>(out));
    return launch_status();
}

extern "C" int moe_bias_update(const int32_t* counts, int E, int64_t T, int k, float gamma,
                               float* b, moe_stream_t stream) {
    if (!counts || !b || E <= 0 || T <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    bias_update_kernel<<<(unsigned)cdiv(E, 256), 256, 0, (cudaStream_t)stream>>>(counts, E, T, k,
                                                                                gamma, b);
    return launch_status();
}

extern "C" int moe_bias_update_proportional(const int32_t* counts, int E, int64_t T, int k,
                                            float gamma, float* b, moe_stream_t stream) {
    if (!counts || !b || E <= 0 || T <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    bias_update_proportional_kernel<<<(unsigned)cdiv(E, 256), 256, 0, (cudaStream_t)stream>>>(
        counts, E, T, k, gamma, b);
    return launch_status();
}

extern "C" int moe_combine_bwd(const moe_bf16* dY, const moe_bf16* Y_perm,
                               const float* topk_gate, const int32_t* slot_to_row,
                               const int64_t* row_offsets, const int32_t* perm_token,
                               int64_t T, int d, int E, int k, moe_bf16* dY_perm, float* dg,
                               moe_stream_t stream) {
    if (!dY || !slot_to_row || !row_offsets || !perm_token || !dY_perm)
        return MOE_ERR_INVALID_ARG;
    if ((Y_perm == nullptr) != (dg == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(T, d, E, k)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(dY) || (Y_perm && !aligned16(Y_perm)) || !aligned16(dY_perm))
        return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const __nv_bfloat16* dYb = reinterpret_cast<const __nv_bfloat16*>(dY);
    const __nv_bfloat16* Yb = reinterpret_cast<const __nv_bfloat16*>(Y_perm);
    __nv_bfloat16* dYp = reinterpret_cast<__nv_bfloat16*>(dY_perm);
    const int64_t tb = warp_grid(T);  // token blocks; then kPadSplit padding blocks per expert
    const unsigned g = (unsigned)(tb + (int64_t)E * kPadSplit);
    if (k <= 2) combine_bwd_kernel<2><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token);
    else if (k <= 4) combine_bwd_kernel<4><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token);
    else if (k <= 8) combine_bwd_kernel<8><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token);
    else if (k <= 16) combine_bwd_kernel<16><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token);
    else combine_bwd_kernel<32><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token);
    return launch_status();
}

extern "C" int moe_combine_bwd_fp8(const moe_bf16* dY, const moe_bf16* Y_perm,
                                   const float* topk_gate, const int32_t* slot_to_row,
                                   const int64_t* row_offsets, const int32_t* perm_token,
                                   int64_t T, int d, int E, int k, moe_bf16* dY_perm, float* dg,
                                   uint8_t* dYq, float* sdY, moe_stream_t stream) {
    if (!dY || !Y_perm || !topk_gate || !slot_to_row || !row_offsets || !perm_token ||
        !dY_perm || !dg || !dYq || !sdY)
        return MOE_ERR_INVALID_ARG;
    if (!shape_ok(T, d, E, k)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(dY) || !aligned16(Y_perm) || !aligned16(dY_perm) || !aligned16(dYq))
        return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const __nv_bfloat16* dYb = reinterpret_cast<const __nv_bfloat16*>(dY);
    const __nv_bfloat16* Yb = reinterpret_cast<const __nv_bfloat16*>(Y_perm);
    __nv_bfloat16* dYp = reinterpret_cast<__nv_bfloat16*>(dY_perm);
    const int64_t tb = warp_grid(T);  // token blocks; then kPadSplit padding blocks per expert
    const unsigned g = (unsigned)(tb + (int64_t)E * kPadSplit);
    if (k <= 2) combine_bwd_kernel<2, true><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token, dYq, sdY);
    else if (k <= 4) combine_bwd_kernel<4, true><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token, dYq, sdY);
    else if (k <= 8) combine_bwd_kernel<8, true><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token, dYq, sdY);
    else if (k <= 16) combine_bwd_kernel<16, true><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token, dYq, sdY);
    else combine_bwd_kernel<32, true><<<g, 256, 0, st>>>(dYb, Yb, topk_gate, slot_to_row, T, d, k, dYp, dg, tb, row_offsets, perm_token, dYq, sdY);
    if (launch_pad_rows_fp8(row_offsets, perm_token, d, E, dYq, sdY, st) != MOE_OK)
        return MOE_ERR_LAUNCH;
    return launch_status();
}

extern "C" int moe_row_gates(const float* topk_gate, const int32_t* slot_to_row, int64_t T, int k,
                             int64_t rows, float* row_gate, moe_stream_t stream) {
    if (!topk_gate || !slot_to_row || !row_gate || T <= 0 || k <= 0 || rows <= 0)
        return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(row_gate, 0, sizeof(float) * rows, st) != cudaSuccess) return MOE_ERR_LAUNCH;
    const int64_t n = T * k;
    row_gates_kernel<<<(unsigned)cdiv(n, 256), 256, 0, st>>>(topk_gate, slot_to_row, n, rows, row_gate);
    return launch_status();
}

extern "C" int moe_gate_grad(const float* gate_part, const int32_t* slot_to_row, int64_t T, int k,
                             int f, float* dg, moe_stream_t stream) {
    if (!gate_part || !slot_to_row || !dg || T <= 0 || k <= 0 || f <= 0 || f % 64 != 0)
        return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    const int64_t n = T * k;
    gate_grad_kernel<<<(unsigned)cdiv(n, 256), 256, 0, (cudaStream_t)stream>>>(gate_part, f / 64,
                                                                              slot_to_row, n, dg);
    return launch_status();
}

extern "C" int moe_permute_bwd(const moe_bf16* dX_perm, const int32_t* slot_to_row,
                               const moe_bf16* dx_shared, const float* dlogits,
                               const float* W_r, const float* dx_router, int64_t T, int d, int E,
                               int k, moe_bf16* dx, moe_stream_t stream) {
    if (!dX_perm || !slot_to_row || !dx) return MOE_ERR_INVALID_ARG;
    if ((dlogits == nullptr) != (W_r == nullptr)) return MOE_ERR_INVALID_ARG;
    if (dx_router && dlogits) return MOE_ERR_INVALID_ARG;  // the router term once
    if (dx_router && !aligned16(dx_router)) return MOE_ERR_INVALID_ARG;
    if (!shape_ok(T, d, E, k)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(dX_perm) || !aligned16(dx) || (dx_shared && !aligned16(dx_shared)) ||
        (W_r && !aligned16(W_r)))
        return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const __nv_bfloat16* a = reinterpret_cast<const __nv_bfloat16*>(dX_perm);
    const __nv_bfloat16* sh = reinterpret_cast<const __nv_bfloat16*>(dx_shared);
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(dx);
    const unsigned grid = warp_grid(T);
    if (dx_router)
        launch_permute_bwd<true>(grid, st, a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
    else
        launch_permute_bwd<false>(grid, st, a, slot_to_row, sh, dlogits, W_r, dx_router, T, d, E, k, o);
    return launch_status();
}

// ------------------------------------------------------------------------------------
// moe_permute_noalloc: the same launches as moe_permute, with the two per-chunk count
// tables in a library-owned static device array instead of the caller's workspace, for
// callers that have no way to allocate device memory (see the header).

namespace {

constexpr int kNoallocMaxInts = MOE_PERMUTE_NOALLOC_MAX_INTS;
constexpr int kNoallocMaxDevices = 64;

// [0, kNoallocMaxInts): per-chunk counts; [kNoallocMaxInts, 2 kNoallocMaxInts): chunk bases.
static __device__ __align__(256) int32_t g_permute_scratch[2 * kNoallocMaxInts];

// Per device: the context the address was looked up in (by its driver-assigned id, which
// is never reused) and the address. A new context on the device (after cudaDeviceReset, or
// a primary context released and created again) may place the array elsewhere, so the
// address is looked up again whenever the current context's id differs.
struct ScratchAddr {
    unsigned long long ctx_id;
    int32_t* ptr;
};
ScratchAddr g_permute_scratch_addr[kNoallocMaxDevices] = {};
std::mutex g_permute_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the current context, or 0 when the driver cannot give one (then the address is
// looked up on every call).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_permute_scratch in the current device's context, looked up once per
// context. In host code the symbol name is only a host-side handle, so the address must
// come from the runtime before a kernel can be given it.
int32_t* permute_scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return nullptr;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lk(g_permute_scratch_mu);
    ScratchAddr& a = g_permute_scratch_addr[dev];
    if (!a.ptr || id == 0 || a.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        a.ptr = static_cast<int32_t*>(p);
        a.ctx_id = id;
    }
    return a.ptr;
}

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_idx, const moe_bf16* x, int64_t T, int d,
                                   int E, int k, int32_t* counts, int64_t* offsets,
                                   int64_t* row_offsets, int32_t* perm_token,
                                   int32_t* slot_to_row, moe_bf16* X_perm,
                                   moe_stream_t stream) {
    if (!topk_idx || !x || !counts || !offsets || !row_offsets || !perm_token || !slot_to_row ||
        !X_perm)
        return MOE_ERR_INVALID_ARG;
    if (!shape_ok(T, d, E, k)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > E || k > 32 || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(X_perm)) return MOE_ERR_INVALID_ARG;
    const int64_t nb = hist_blocks(T);
    if (nb * E > kNoallocMaxInts) return MOE_ERR_TOO_LARGE;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    int* status = device_status_word();
    if (!status) return MOE_ERR_LAUNCH;
    int32_t* scratch = permute_scratch_on_current_device();
    if (!scratch) return MOE_ERR_LAUNCH;
    int32_t* bcounts = scratch;
    int32_t* bbase = scratch + kNoallocMaxInts;
    cudaStream_t st = (cudaStream_t)stream;
    hist_kernel<<<(unsigned)nb, kHistThreads, 0, st>>>(topk_idx, T, E, k, bcounts, status);
    scan_kernel<<<1, kScanThreads, 0, st>>>(bcounts, nb, E, bbase, counts, offsets, row_offsets);
    scatter_kernel<<<(unsigned)(nb + (int64_t)E * kPadSplit), kScatterThreads, 0, st>>>(
        topk_idx, T, E, k, nb, bbase, row_offsets, counts, d, perm_token, slot_to_row,
        reinterpret_cast<__nv_bfloat16*>(X_perm), nullptr, nullptr);
    gather_kernel<<<warp_grid(T), 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x),
                                                slot_to_row, T, d, k,
                                                reinterpret_cast<__nv_bfloat16*>(X_perm));
    return launch_status();
}
