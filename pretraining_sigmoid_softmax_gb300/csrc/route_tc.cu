// Router contractions on the tensor cores (tcgen05, TMEM, TMA), for routers of up to 128
// experts: the logits l = x W_r^T with the top-k choice, gates and softmax statistics in the
// epilogue, and the W_r gradient dW_r = dlogits^T x.
//
// Router: "The whole stack, in the open" (Apex-3), "What's inside", row "Fine-grained MoE"
// (sigmoid router, per-expert selection bias, no loss term); KempnerForge README,
// "Features" (softmax top-k router, router z-loss); handbook summary, section 2.5 (router
// logits in fp32).
//
// fp32 through bf16 tensor cores. The fp32 operand (W_r forward, the logit gradient
// backward) is split into three bf16 pieces that sum to it within 2^-24 relative (see
// split3_bf16); the other operand (x) is bf16 already. Every product of two bf16 values is
// exact in fp32; the tensor core sums each piece's products in fp32 and the three partial
// sums are added in fp32 (largest first), so the result is an fp32 contraction of the exact
// operands, as the router's definition asks. The contraction is thin (E <= 128 outputs per token), so after the split
// it is bound by reading x once from HBM rather than by arithmetic.
//
// Logits kernel: persistent, one CTA per SM, 128-token tiles. Warp 0 issues TMA loads of
// the x tile (128 tokens x 64 of d) and of the three W_r pieces (epad experts x 64 of d,
// back to back: a 3 epad-row operand) into a ring of stages; warp 1 issues one tcgen05.mma
// (M = 128, N = 3 epad, K = 16; two of half the width when 3 epad > 256) per K step, which
// leaves the three partial logits side by side in TMEM. Warps 4-7 each own 32 tokens (one
// TMEM lane per token): a first pass adds the partials, writes the logits and parks each
// logit and selection value (or key) back in TMEM (tcgen05.st). Sigmoid routing with k <= 8
// (its own kernel instance) then reads them back eight experts at a time into an insertion
// network; otherwise k passes each pick the best expert not yet taken. Both follow the order
// "larger value, then lower index" - the definition's total order.
//
// dW_r kernel: the transposed product dW_r^T[j][e] = sum_t x[t][j] dlogits[t][e], as
// 128-column tiles of d (M) by np experts (N), K running over tokens. The token axis is
// split so that the grid fills the GPU; each (tile, split) unit writes its partial sums,
// which a fixed-order reduction adds. Both operands are MN-major (x rows and gradient rows
// are contiguous along j and e).
//
// Every mbarrier wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT, stops every
// role of the CTA, and the CTA frees its tensor memory before it returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "router.cuh"
#include "sizes.h"
#include "tmap.h"

namespace moe {
namespace {

constexpr int kTcThreads = 256;
constexpr int kTcSmemBudget = 200 * 1024;
constexpr int kTcMisc = 256;  // barriers, TMEM slot, abort flag

// dst[p][r][c] for p = 0..2, r < rows_pad, c < cols: the bf16 pieces of src[r][c] (zero for
// r >= rows).
__global__ void split3_rows_kernel(const float* __restrict__ src, int rows, int cols, int rows_pad,
                                   __nv_bfloat16* __restrict__ dst) {
    const int64_t n = (int64_t)rows_pad * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float v = (i / cols) < rows ? src[i] : 0.f;
        __nv_bfloat16 p0, p1, p2;
        split3_bf16(v, p0, p1, p2);
        dst[i] = p0;
        dst[n + i] = p1;
        dst[2 * n + i] = p2;
    }
}

// dst[p][t][e] for p = 0, 1, t < T, e < np: the first two bf16 pieces of src[t][e] (zero for
// e >= E); piece p starts at dst + p * pstride.
__global__ void split2_cols_kernel(const float* __restrict__ src, int64_t T, int E, int np,
                                   int64_t pstride, __nv_bfloat16* __restrict__ dst) {
    const int64_t n = T * np;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / np;
        const int e = (int)(i % np);
        const float v = e < E ? src[t * E + e] : 0.f;
        __nv_bfloat16 p0, p1, p2;
        split3_bf16(v, p0, p1, p2);
        dst[i] = p0;
        dst[pstride + i] = p1;
    }
}

struct TcRing {
    uint8_t* a;
    uint8_t* b;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint32_t* tmem_slot;
    int* abort_flag;
    uint8_t* extra;  // after the misc block
};

template <int STAGES, int A_BYTES, int B_BYTES>
__device__ __forceinline__ TcRing carve_ring(uint8_t* raw) {
    TcRing r;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    r.a = base;
    r.b = base + (size_t)STAGES * A_BYTES;
    uint8_t* misc = base + (size_t)STAGES * (A_BYTES + B_BYTES);
    r.full = reinterpret_cast<uint64_t*>(misc);
    r.empty = r.full + STAGES;
    r.tfull = r.empty + STAGES;
    r.tempty = r.tfull + 2;
    r.tmem_slot = reinterpret_cast<uint32_t*>(r.tempty + 2);
    r.abort_flag = reinterpret_cast<int*>(r.tmem_slot + 1);
    r.extra = misc + kTcMisc;
    return r;
}

// Barrier setup and TMEM allocation (warp 2); every thread returns the TMEM base.
template <int STAGES, int TMEM_COLS>
__device__ __forceinline__ uint32_t ring_setup(const TcRing& R, int tid, int warp) {
    static_assert((STAGES * 2 + 4) * 8 + 8 <= kTcMisc, "misc block");
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&R.full[s]), 1);
            mbar_init(smem_u32(&R.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&R.tfull[b]), 1);
            mbar_init(smem_u32(&R.tempty[b]), 4);  // one arrive per epilogue warp
        }
        *R.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(R.tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *R.tmem_slot;
}

template <int TMEM_COLS>
__device__ __forceinline__ void ring_teardown(const TcRing& R, uint32_t tmem_base, int warp) {
    __syncwarp();
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(R.abort_flag)) {  // let copies in flight land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------------ logits + choice

struct LogitParams {
    int64_t T;
    int64_t ntiles;
    int d, E, k, mode;
    int vec_logits;  // logits rows can take 16-byte stores
    const float* bias;
    float* logits;
    int32_t* topk_idx;
    float* topk_gate;
    float* topk_score;
    float* lse;
    double* z_part;
    int* status;
    uint64_t wait_limit_ns;
};

template <int EPAD>
struct LogitCfg {
    static constexpr int A_BYTES = 128 * 128;       // 128 tokens x 64 bf16 of d
    static constexpr int B_BYTES = 3 * EPAD * 128;  // 3 pieces x EPAD experts x 64 bf16 of d
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (kTcSmemBudget / STAGE_BYTES) > 6 ? 6 : (kTcSmemBudget / STAGE_BYTES);
    // The three pieces sit back to back in a stage, a 3*EPAD-row B tile: one MMA of
    // N = 3*EPAD per K step (two of half that when it exceeds 256) accumulates the three
    // partial logits side by side in TMEM; the epilogue adds them.
    static constexpr int NTOT = 3 * EPAD;
    static constexpr int NMMA = NTOT <= 256 ? 1 : 2;
    static constexpr int NPER = NTOT / NMMA;
    static constexpr int NBUF = 2 * NTOT <= 512 ? 2 : 1;  // accumulators in flight
    static constexpr int TMEM_COLS = NBUF * NTOT <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_mma(NPER, 128, false, false);
    static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + kTcMisc + sizeof(float) * EPAD;
    static_assert(EPAD % 32 == 0 && EPAD >= 32 && EPAD <= 128, "expert tile");
    static_assert(STAGES >= 2, "pipeline depth");
};

// Widest choice made by the insertion network (RouteTopK) in one pass.
constexpr int kNetK = 8;

// The first pass over one token's three partial logits in TMEM (columns [0, EPAD), [EPAD,
// 2 EPAD), [2 EPAD, 3 EPAD) of its lane), 32 experts at a time: adds the partials into the
// logit l, forms the selection value (sigmoid(l) + b, or l; a NaN never wins), calls
// f(e, l, value) for every expert e < E in increasing order, and writes the logits row.
// Executed by all 32 lanes of the warp together (tcgen05.ld is warp-collective); `live`
// masks the stores of rows past the last token.
template <int EPAD, typename F>
__device__ __forceinline__ void route_first_pass(uint32_t t_acc, int64_t t, bool live, bool sig,
                                                 const LogitParams& P, const float* sbias, F&& f) {
    constexpr int NCH = EPAD / 32;
    const int E = P.E;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        uint32_t p0[32], p1[32], p2[32];
        tmem_ld32(t_acc + 32 * c, p0);
        tmem_ld32(t_acc + EPAD + 32 * c, p1);
        tmem_ld32(t_acc + 2 * EPAD + 32 * c, p2);
        tmem_ld_wait();
        uint32_t lv[32], vv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int e = 32 * c + j;
            const float l = (__uint_as_float(p0[j]) + __uint_as_float(p1[j])) + __uint_as_float(p2[j]);
            float val = sig ? route_select_sigmoid(l) + sbias[e] : l;
            if (val != val) val = -INFINITY;
            lv[j] = __float_as_uint(l);
            vv[j] = __float_as_uint(val);
        }
        if (live && P.logits) {
            float* row = P.logits + t * E;
            if (P.vec_logits) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (32 * c + 4 * q < E)
                        *reinterpret_cast<float4*>(row + 32 * c + 4 * q) =
                            make_float4(__uint_as_float(lv[4 * q]), __uint_as_float(lv[4 * q + 1]),
                                        __uint_as_float(lv[4 * q + 2]), __uint_as_float(lv[4 * q + 3]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (32 * c + j < E) row[32 * c + j] = __uint_as_float(lv[j]);
            }
        }
        f(c, lv, vv);
    }
}

// Sigmoid routing with k <= kNetK: the first pass parks each expert's logit and selection key
// in TMEM (over the consumed accumulator); a rolled loop then reads them back eight experts
// at a time and pushes each, in index order, into a kNetK-slot insertion network, which
// leaves the k best in the choice's order ("larger value, then lower index"). Scores are the
// sigmoids of their logits, gates the scores over their sum. The loop is kept rolled so the
// epilogue's code stays small: fully unrolled over 64 or 128 experts it is tens of KB of
// straight-line code per tile, which competes with the producer's and MMA issuer's loops for
// the instruction cache.
template <int EPAD>
__device__ __forceinline__ void route_epilogue_net(uint32_t t_acc, int64_t t, bool live,
                                                   const LogitParams& P, const float* sbias) {
    const int E = P.E, k = P.k;
    const uint32_t t_l = t_acc;         // logits (over the first partial)
    const uint32_t t_v = t_acc + EPAD;  // selection keys (over the second)
    route_first_pass<EPAD>(t_acc, t, live, true, P, sbias, [&](int c, uint32_t (&lv)[32], uint32_t (&vv)[32]) {
#pragma unroll
        for (int j = 0; j < 32; ++j) vv[j] = (uint32_t)route_key(__uint_as_float(vv[j]));
        tmem_st32(t_l + 32 * c, lv);
        tmem_st32(t_v + 32 * c, vv);
    });
    tmem_st_wait();
    RouteTopK<kNetK> top;
    top.init();
#pragma unroll 1
    for (int e0 = 0; e0 < E; e0 += 8) {
        uint32_t kv[8], lv[8];
        tmem_ld8(t_v + e0, kv);
        tmem_ld8(t_l + e0, lv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (e0 + j < E) top.push((int)kv[j], e0 + j, __uint_as_float(lv[j]));
    }
    if (!live) return;
    int32_t* oi = P.topk_idx + t * k;
    float* os = P.topk_score + t * k;
    float* og = P.topk_gate + t * k;
    float sc[kNetK];
    float ssum = 0.f;
#pragma unroll
    for (int i = 0; i < kNetK; ++i) {
        sc[i] = 0.f;
        if (i < k) {
            sc[i] = route_sigmoid(top.l[i]);
            ssum += sc[i];
            oi[i] = top.e[i];
            os[i] = sc[i];
        }
    }
#pragma unroll
    for (int i = 0; i < kNetK; ++i)
        if (i < k) og[i] = sc[i] / ssum;
}

// Every other router (softmax, or k > kNetK): the first pass parks each logit and selection
// value back in TMEM (tcgen05.st), then k passes each pick the best expert not yet taken, in
// the order "larger value, then lower index" - the definition's total order. Softmax also
// forms the normaliser over all experts and returns lse^2 for the z-loss.
template <int EPAD>
__device__ __forceinline__ double route_epilogue(uint32_t t_acc, int64_t t, bool live,
                                                 const LogitParams& P, const float* sbias) {
    constexpr int NCH = EPAD / 32;
    const int E = P.E, k = P.k;
    const bool sig = P.mode == MOE_MODE_SIGMOID;
    const uint32_t t_l = t_acc;          // logits (over the first partial)
    const uint32_t t_v = t_acc + EPAD;   // selection values (over the second)
    float mx = -INFINITY, sum = 0.f;
    route_first_pass<EPAD>(t_acc, t, live, sig, P, sbias, [&](int c, uint32_t (&lv)[32], uint32_t (&vv)[32]) {
        if (!sig) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (32 * c + j < E) mx = fmaxf(mx, __uint_as_float(lv[j]));
        }
        tmem_st32(t_l + 32 * c, lv);
        tmem_st32(t_v + 32 * c, vv);
    });
    tmem_st_wait();
    if (!sig) {  // softmax normaliser over all experts
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            uint32_t lv[32];
            tmem_ld32(t_l + 32 * c, lv);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (32 * c + j < E) sum += expf(__uint_as_float(lv[j]) - mx);
        }
    }
    uint32_t taken[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) taken[c] = 0u;
    int32_t* oi = P.topk_idx + t * k;
    float* os = P.topk_score + t * k;
    float* og = P.topk_gate + t * k;
    float ssum = 0.f;
    for (int i = 0; i < k; ++i) {
        float bv = -INFINITY, bl = 0.f;
        int be = 0x7fffffff;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            uint32_t vv[32], lv[32];
            tmem_ld32(t_v + 32 * c, vv);
            tmem_ld32(t_l + 32 * c, lv);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int e = 32 * c + j;
                const float val = __uint_as_float(vv[j]);
                if (e < E && !((taken[c] >> j) & 1u) && route_better(val, e, bv, be)) {
                    bv = val;
                    be = e;
                    bl = __uint_as_float(lv[j]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c)
            if (c == (be >> 5)) taken[c] |= 1u << (be & 31);
        const float s = sig ? route_sigmoid(bl) : expf(bl - mx) / sum;
        ssum += s;
        if (live) {
            oi[i] = be;
            os[i] = s;
            if (!sig) og[i] = s;
        }
    }
    if (sig) {
        if (live)
            for (int i = 0; i < k; ++i) og[i] = os[i] / ssum;
        return 0.0;
    }
    const float l_se = mx + logf(sum);
    if (live) P.lse[t] = l_se;
    return live ? (double)l_se * (double)l_se : 0.0;
}

template <int EPAD, bool NET>
__global__ void __launch_bounds__(kTcThreads, 1)
    route_logits_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                           const LogitParams P) {
    using C = LogitCfg<EPAD>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const TcRing R = carve_ring<C::STAGES, C::A_BYTES, C::B_BYTES>(smem_raw);
    float* sbias = reinterpret_cast<float*>(R.extra);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < EPAD; i += kTcThreads)
        sbias[i] = (P.mode == MOE_MODE_SIGMOID && i < P.E) ? P.bias[i] : 0.f;
    const uint32_t tmem_base = ring_setup<C::STAGES, C::TMEM_COLS>(R, tid, warp);
    volatile int* abort_flag = R.abort_flag;
    const int kiters = P.d / 64;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        tma_prefetch_desc(&mx);
        tma_prefetch_desc(&mw);
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t tile = blockIdx.x; tile < P.ntiles; tile += gridDim.x) {
            bool ok = true;
            for (int kb = 0; kb < kiters; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&R.empty[stage]), phase ^ 1u, abort_flag, P.status,
                                       P.wait_limit_ns, 40)) {
                    ok = false;
                    break;
                }
                const uint32_t bar = smem_u32(&R.full[stage]);
                mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
                tma_load_2d(smem_u32(R.a + (size_t)stage * C::A_BYTES), &mx, bar, kb * 64,
                            (int32_t)(tile * 128));
                const uint32_t b_dst = smem_u32(R.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int p = 0; p < 3; ++p) tma_load_2d(b_dst + p * EPAD * 128, &mw, bar, kb * 64, p * EPAD);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        for (int64_t tile = blockIdx.x; tile < P.ntiles; tile += gridDim.x, ++local) {
            const int buf = C::NBUF == 2 ? (local & 1) : 0;
            const uint32_t use = C::NBUF == 2 ? ((local >> 1) & 1) : (local & 1);
            if (!mbar_wait_bounded(smem_u32(&R.tempty[buf]), use ^ 1u, abort_flag, P.status,
                                   P.wait_limit_ns, 41))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * C::NTOT;
            bool ok = true;
            for (int kb = 0; kb < kiters; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&R.full[stage]), phase, abort_flag, P.status,
                                       P.wait_limit_ns, 42)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = smem_u32(R.a + (size_t)stage * C::A_BYTES);
                const uint32_t b_s = smem_u32(R.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 4 steps of 16 K-elements (32 bytes)
                    const uint64_t adesc = sdesc_sw128(a_s + kk * 32, 16, 1024);
#pragma unroll
                    for (int m = 0; m < C::NMMA; ++m) {
                        const uint64_t bdesc = sdesc_sw128(b_s + m * C::NPER * 128 + kk * 32, 16, 1024);
                        umma_bf16(d_tmem + m * C::NPER, adesc, bdesc, C::IDESC, (kb | kk) ? 1u : 0u);
                    }
                }
                umma_commit(smem_u32(&R.empty[stage]));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(smem_u32(&R.tfull[buf]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;  // TMEM lanes 32q .. 32q+31
        int local = 0;
        for (int64_t tile = blockIdx.x; tile < P.ntiles; tile += gridDim.x, ++local) {
            const int buf = C::NBUF == 2 ? (local & 1) : 0;
            const uint32_t use = C::NBUF == 2 ? ((local >> 1) & 1) : (local & 1);
            bool ok = mbar_wait_bounded(smem_u32(&R.tfull[buf]), use, abort_flag, P.status,
                                        P.wait_limit_ns, 43);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_acc = tmem_base + buf * C::NTOT + ((uint32_t)(32 * q) << 16);
            const int64_t t = tile * 128 + 32 * q + lane;
            double z = 0.0;
            if constexpr (NET)
                route_epilogue_net<EPAD>(t_acc, t, t < P.T, P, sbias);
            else
                z = route_epilogue<EPAD>(t_acc, t, t < P.T, P, sbias);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&R.tempty[buf]));
            if (P.mode == MOE_MODE_SOFTMAX) {  // fixed-order sum of the warp's 32 tokens
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                if (lane == 0) P.z_part[tile * 4 + q] = z;
            }
        }
    }
    ring_teardown<C::TMEM_COLS>(R, tmem_base, warp);
}

template <int EPAD>
int launch_logits(const CUtensorMap& mx, const CUtensorMap& mw, const LogitParams& P, cudaStream_t st) {
    using C = LogitCfg<EPAD>;
    static_assert(C::SMEM_BYTES <= 227 * 1024, "shared memory");
    const bool net = P.mode == MOE_MODE_SIGMOID && P.k <= kNetK;
    auto kern = net ? route_logits_tc_kernel<EPAD, true> : route_logits_tc_kernel<EPAD, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    const int64_t grid = P.ntiles < sm_count() ? P.ntiles : sm_count();
    kern<<<(unsigned)grid, kTcThreads, C::SMEM_BYTES, st>>>(mx, mw, P);
    return launch_status();
}

// ------------------------------------------------------------------------ W_r gradient

struct DwrParams {
    int64_t T;
    int d, E;
    int mtiles;    // d / 128
    int nsplit;    // token splits
    int kb_total;  // 64-token blocks
    float* part;   // [nsplit][E][d]
    int* status;
    uint64_t wait_limit_ns;
};

template <int NP>
struct DwrCfg {
    static constexpr int A_BYTES = 2 * 8192;        // 64 tokens x 128 of d, two 64-wide boxes
    static constexpr int B_BYTES = 3 * NP * 128;    // 3 pieces x 64 tokens x NP experts
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (kTcSmemBudget / STAGE_BYTES) > 6 ? 6 : (kTcSmemBudget / STAGE_BYTES);
    static constexpr int TMEM_COLS = 2 * NP;
    static constexpr uint32_t IDESC = idesc_mma(NP, 128, true, true);
    static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + kTcMisc;
    static_assert(NP == 64 || NP == 128, "expert tile");
};

struct DwrUnit {
    int mt, s, kb_lo, kb_hi;
};

__device__ __forceinline__ DwrUnit dwr_unit(int64_t u, const DwrParams& P) {
    DwrUnit w;
    w.mt = (int)(u % P.mtiles);
    w.s = (int)(u / P.mtiles);
    w.kb_lo = (int)((int64_t)w.s * P.kb_total / P.nsplit);
    w.kb_hi = (int)((int64_t)(w.s + 1) * P.kb_total / P.nsplit);
    return w;
}

template <int NP>
__global__ void __launch_bounds__(kTcThreads, 1)
    route_dwr_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap ml0,
                        const __grid_constant__ CUtensorMap ml1, const __grid_constant__ CUtensorMap ml2,
                        const DwrParams P) {
    using C = DwrCfg<NP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const TcRing R = carve_ring<C::STAGES, C::A_BYTES, C::B_BYTES>(smem_raw);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t tmem_base = ring_setup<C::STAGES, C::TMEM_COLS>(R, tid, warp);
    volatile int* abort_flag = R.abort_flag;
    const int64_t nunits = (int64_t)P.mtiles * P.nsplit;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        tma_prefetch_desc(&mx);
        tma_prefetch_desc(&ml0);
        tma_prefetch_desc(&ml1);
        tma_prefetch_desc(&ml2);
        const CUtensorMap* ml[3] = {&ml0, &ml1, &ml2};
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
            const DwrUnit w = dwr_unit(u, P);
            bool ok = true;
            for (int kb = w.kb_lo; kb < w.kb_hi; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&R.empty[stage]), phase ^ 1u, abort_flag, P.status,
                                       P.wait_limit_ns, 44)) {
                    ok = false;
                    break;
                }
                const uint32_t bar = smem_u32(&R.full[stage]);
                mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
                const uint32_t a_dst = smem_u32(R.a + (size_t)stage * C::A_BYTES);
                const int32_t t0 = kb * 64, j0 = w.mt * 128;
                tma_load_2d(a_dst, &mx, bar, j0, t0);
                tma_load_2d(a_dst + 8192, &mx, bar, j0 + 64, t0);
                const uint32_t b_dst = smem_u32(R.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int p = 0; p < 3; ++p)
#pragma unroll
                    for (int g = 0; g < NP / 64; ++g)
                        tma_load_2d(b_dst + p * NP * 128 + g * 8192, ml[p], bar, 64 * g, t0);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, ++local) {
            const DwrUnit w = dwr_unit(u, P);
            const int buf = local & 1;
            if (!mbar_wait_bounded(smem_u32(&R.tempty[buf]), ((local >> 1) & 1) ^ 1u, abort_flag,
                                   P.status, P.wait_limit_ns, 45))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * NP;
            bool ok = true;
            for (int kb = w.kb_lo; kb < w.kb_hi; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&R.full[stage]), phase, abort_flag, P.status,
                                       P.wait_limit_ns, 46)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = smem_u32(R.a + (size_t)stage * C::A_BYTES);
                const uint32_t b_s = smem_u32(R.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 4 steps of 16 tokens (2048 bytes of k-rows)
                    const uint64_t adesc = sdesc_sw128(a_s + kk * 2048, 8192, 1024);
#pragma unroll
                    for (int p = 0; p < 3; ++p) {
                        const uint64_t bdesc = sdesc_sw128(b_s + p * NP * 128 + kk * 2048, 8192, 1024);
                        umma_bf16(d_tmem, adesc, bdesc, C::IDESC,
                                  (kb > w.kb_lo || kk > 0 || p > 0) ? 1u : 0u);
                    }
                }
                umma_commit(smem_u32(&R.empty[stage]));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(smem_u32(&R.tfull[buf]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;
        int local = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, ++local) {
            const DwrUnit w = dwr_unit(u, P);
            const int buf = local & 1;
            bool ok = mbar_wait_bounded(smem_u32(&R.tfull[buf]), (local >> 1) & 1, abort_flag,
                                        P.status, P.wait_limit_ns, 47);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_acc = tmem_base + buf * NP + ((uint32_t)(32 * q) << 16);
            const int j = w.mt * 128 + 32 * q + lane;
            float* out = P.part + (size_t)w.s * P.E * P.d + j;
#pragma unroll
            for (int c = 0; c < NP / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(t_acc + 32 * c, v);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int e = 32 * c + jj;
                    if (e < P.E) out[(size_t)e * P.d] = __uint_as_float(v[jj]);  // coalesced over j
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&R.tempty[buf]));
        }
    }
    ring_teardown<C::TMEM_COLS>(R, tmem_base, warp);
}

template <int NP>
int launch_dwr(const CUtensorMap& mx, const CUtensorMap* ml, const DwrParams& P, cudaStream_t st) {
    using C = DwrCfg<NP>;
    static_assert(C::SMEM_BYTES <= 227 * 1024, "shared memory");
    auto kern = route_dwr_tc_kernel<NP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    const int64_t units = (int64_t)P.mtiles * P.nsplit;
    const int64_t grid = units < sm_count() ? units : sm_count();
    kern<<<(unsigned)grid, kTcThreads, C::SMEM_BYTES, st>>>(mx, ml[0], ml[1], ml[2], P);
    return launch_status();
}

// ------------------------------------------------------------ router input gradient
// dx_r[t][j] = sum_e dlogits[t][e] W_r[e][j] on the tensor cores, for dense logit gradients
// (softmax router, balancing losses), where the input-gradient kernel's row loop over W_r
// would read E rows of d fp32 from L2 per token. With the three-piece split d = d0 + d1 + d2
// and w = w0 + w1 + w2, the product keeps d0 w0 + d0 w1 + d1 w0: the dropped terms are
// below 3 * 2^-16 of each product, far under the bf16 rounding of the dx they feed. The
// three kept terms are three K segments (np experts each) of one GEMM: M = 128 tokens,
// N = BN columns of d, K = 3 np; A (the logit-gradient pieces, [T, np]) K-major, B (the W_r
// pieces, [np, d]) MN-major. The fp32 result is staged per warp in 32 x 32 boxes (128-byte
// swizzle) and written by TMA stores, which clip rows past T.

struct RdxParams {
    int64_t T;
    int d, np;
    int64_t ntiles;  // ceil(T / 128) * (d / BN)
    int* status;
    uint64_t wait_limit_ns;
};

template <int BN>
struct RdxCfg {
    static constexpr int A_BYTES = 128 * 128;          // 128 tokens x 64 experts, K-major
    static constexpr int B_BYTES = (BN / 64) * 8192;   // 64 experts x BN columns, MN-major
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 3;
    static constexpr int TMEM_COLS = 2 * BN;           // two accumulators
    static constexpr uint32_t IDESC = idesc_mma(BN, 128, false, true);
    static constexpr int OUT_BUF = 32 * 128;           // 32 rows x 32 fp32
    static constexpr size_t SMEM_BYTES =
        1024 + (size_t)STAGES * STAGE_BYTES + kTcMisc + 1024 + 4 * 2 * OUT_BUF;
    static_assert(BN == 128 || BN == 256, "column tile");
};

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    router_dx_tc_kernel(const __grid_constant__ CUtensorMap ml0, const __grid_constant__ CUtensorMap ml1,
                        const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mo,
                        const RdxParams P) {
    using C = RdxCfg<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const TcRing R = carve_ring<C::STAGES, C::A_BYTES, C::B_BYTES>(smem_raw);
    uint8_t* ob = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(R.extra) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t tmem_base = ring_setup<C::STAGES, C::TMEM_COLS>(R, tid, warp);
    volatile int* abort_flag = R.abort_flag;
    const int ntn = P.d / BN;
    const int kb_seg = P.np / 64;    // k-blocks per segment
    const int nkb = 3 * kb_seg;      // segments: (d0, w0), (d0, w1), (d1, w0)

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        tma_prefetch_desc(&ml0);
        tma_prefetch_desc(&ml1);
        tma_prefetch_desc(&mw);
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t tile = blockIdx.x; tile < P.ntiles; tile += gridDim.x) {
            const int32_t t0 = (int32_t)((tile / ntn) * 128), n0 = (int32_t)(tile % ntn) * BN;
            bool ok = true;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&R.empty[stage]), phase ^ 1u, abort_flag, P.status,
                                       P.wait_limit_ns, 48)) {
                    ok = false;
                    break;
                }
                const int seg = kb / kb_seg, e0 = (kb % kb_seg) * 64;
                const CUtensorMap* ma = seg == 2 ? &ml1 : &ml0;  // d1 in the third segment
                const int32_t wrow = (seg == 1 ? P.np : 0) + e0;  // w1 in the second
                const uint32_t bar = smem_u32(&R.full[stage]);
                mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
                tma_load_2d(smem_u32(R.a + (size_t)stage * C::A_BYTES), ma, bar, e0, t0);
                const uint32_t b_dst = smem_u32(R.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int g = 0; g < BN / 64; ++g) tma_load_2d(b_dst + g * 8192, &mw, bar, n0 + 64 * g, wrow);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        for (int64_t tile = blockIdx.x; tile < P.ntiles; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            if (!mbar_wait_bounded(smem_u32(&R.tempty[buf]), ((local >> 1) & 1) ^ 1u, abort_flag,
                                   P.status, P.wait_limit_ns, 49))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * BN;
            bool ok = true;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&R.full[stage]), phase, abort_flag, P.status,
                                       P.wait_limit_ns, 50)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = smem_u32(R.a + (size_t)stage * C::A_BYTES);
                const uint32_t b_s = smem_u32(R.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 16 experts per step
                    const uint64_t adesc = sdesc_sw128(a_s + kk * 32, 16, 1024);
                    const uint64_t bdesc = sdesc_sw128(b_s + kk * 2048, 8192, 1024);
                    umma_bf16(d_tmem, adesc, bdesc, C::IDESC, (kb | kk) ? 1u : 0u);
                }
                umma_commit(smem_u32(&R.empty[stage]));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(smem_u32(&R.tfull[buf]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;
        int local = 0;
        uint32_t n = 0;  // chunks staged by this warp (output buffer parity)
        for (int64_t tile = blockIdx.x; tile < P.ntiles; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            bool ok = mbar_wait_bounded(smem_u32(&R.tfull[buf]), (local >> 1) & 1, abort_flag,
                                        P.status, P.wait_limit_ns, 51);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_acc = tmem_base + buf * BN + ((uint32_t)(32 * q) << 16);
            const int32_t row0 = (int32_t)((tile / ntn) * 128) + 32 * q;
            const int32_t n0 = (int32_t)(tile % ntn) * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c, ++n) {
                uint32_t v[32];
                tmem_ld32(t_acc + 32 * c, v);
                tmem_ld_wait();
                uint8_t* ob_w = ob + ((size_t)q * 2 + (n & 1)) * C::OUT_BUF;
                if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)  // 128-byte swizzle: piece j of row r at j ^ (r & 7)
                    *reinterpret_cast<uint4*>(ob_w + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                        make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&mo, smem_u32(ob_w), n0 + 32 * c, row0);
                    bulk_commit();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&R.tempty[buf]));
        }
        if (lane == 0) bulk_wait<0>();
    }
    ring_teardown<C::TMEM_COLS>(R, tmem_base, warp);
}

template <int BN>
int launch_rdx(const CUtensorMap* ml, const CUtensorMap& mw, const CUtensorMap& mo,
               const RdxParams& P, cudaStream_t st) {
    using C = RdxCfg<BN>;
    static_assert(C::SMEM_BYTES <= 227 * 1024, "shared memory");
    auto kern = router_dx_tc_kernel<BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    const int64_t grid = P.ntiles < sm_count() ? P.ntiles : sm_count();
    kern<<<(unsigned)grid, kTcThreads, C::SMEM_BYTES, st>>>(ml[0], ml[1], mw, mo, P);
    return launch_status();
}

}  // namespace

int launch_route_logits_tc(const __nv_bfloat16* x, const float* W_r, const float* b, int64_t T,
                           int d, int E, int k, int mode, float* logits, int32_t* topk_idx,
                           float* topk_gate, float* topk_score, float* lse, double* z_part,
                           int64_t* nz, __nv_bfloat16* w3, cudaStream_t st) {
    const int epad = route_tc_epad(E);
    if (!epad || d % 64 != 0) return MOE_ERR_UNSUPPORTED;
    const int64_t n = (int64_t)epad * d;
    const int sblocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    split3_rows_kernel<<<sblocks, 256, 0, st>>>(W_r, E, d, epad, w3);
    if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    CUtensorMap mx, mw;
    if (!make_tmap_bf16_2d(&mx, x, d, T, 64, 128) || !make_tmap_bf16_2d(&mw, w3, d, 3 * (uint64_t)epad, 64, epad))
        return MOE_ERR_LAUNCH;
    LogitParams P{};
    P.T = T;
    P.ntiles = route_tc_tiles(T);
    P.d = d;
    P.E = E;
    P.k = k;
    P.mode = mode;
    P.vec_logits = (logits && E % 4 == 0 && aligned16(logits)) ? 1 : 0;
    P.bias = b;
    P.logits = logits;
    P.topk_idx = topk_idx;
    P.topk_gate = topk_gate;
    P.topk_score = topk_score;
    P.lse = lse;
    P.z_part = z_part;
    P.status = device_status_word();
    P.wait_limit_ns = wait_limit_ns();
    *nz = 4 * P.ntiles;
    if (epad == 32) return launch_logits<32>(mx, mw, P, st);
    if (epad == 64) return launch_logits<64>(mx, mw, P, st);
    return launch_logits<128>(mx, mw, P, st);
}

int launch_route_dwr_tc(const __nv_bfloat16* x, const __nv_bfloat16* dl3, int64_t pstride,
                        int64_t T, int d, int E, float* part, int64_t* nsplit, cudaStream_t st) {
    const int np = route_tc_np(E);
    if (!np || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    DwrParams P{};
    P.T = T;
    P.d = d;
    P.E = E;
    P.mtiles = d / 128;
    P.kb_total = (int)cdiv(T, 64);
    // enough (tile, split) units for about four per SM, within the scratch's split count
    int64_t s = cdiv(4 * (int64_t)sm_count(), P.mtiles);
    if (s > route_tc_splits_max(T)) s = route_tc_splits_max(T);
    if (s < 1) s = 1;
    P.nsplit = (int)s;
    P.part = part;
    P.status = device_status_word();
    P.wait_limit_ns = wait_limit_ns();
    *nsplit = s;
    CUtensorMap mx, ml[3];
    if (!make_tmap_bf16_2d(&mx, x, d, T, 64, 64)) return MOE_ERR_LAUNCH;
    for (int p = 0; p < 3; ++p)
        if (!make_tmap_bf16_2d(&ml[p], dl3 + (size_t)p * pstride, np, T, 64, 64)) return MOE_ERR_LAUNCH;
    if (np == 64) return launch_dwr<64>(mx, ml, P, st);
    return launch_dwr<128>(mx, ml, P, st);
}

int launch_router_dx_tc(const float* dlogits, const float* W_r, int64_t T, int d, int E,
                        __nv_bfloat16* dl2, int64_t pstride, __nv_bfloat16* w3, float* dx_r,
                        cudaStream_t st) {
    const int np = route_tc_np(E);
    if (!np || d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    {
        const int64_t m = T * np;
        const int blocks = (int)((m + 255) / 256 < 4096 ? (m + 255) / 256 : 4096);
        split2_cols_kernel<<<blocks, 256, 0, st>>>(dlogits, T, E, np, pstride, dl2);
        if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    }
    const __nv_bfloat16* dl3 = dl2;
    const int64_t n = (int64_t)np * d;
    const int sblocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    split3_rows_kernel<<<sblocks, 256, 0, st>>>(W_r, E, d, np, w3);  // [3][np][d], zero past E
    if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    const int BN = d % 256 == 0 ? 256 : 128;
    CUtensorMap ml[2], mw, mo;
    for (int p = 0; p < 2; ++p)
        if (!make_tmap_bf16_2d(&ml[p], dl3 + (size_t)p * pstride, np, T, 64, 128)) return MOE_ERR_LAUNCH;
    if (!make_tmap_bf16_2d(&mw, w3, d, 3 * (uint64_t)np, 64, 64) ||
        !make_tmap_f32_2d(&mo, dx_r, d, T, 32, 32))
        return MOE_ERR_LAUNCH;
    RdxParams P{};
    P.T = T;
    P.d = d;
    P.np = np;
    P.ntiles = route_tc_tiles(T) * (d / BN);
    P.status = device_status_word();
    P.wait_limit_ns = wait_limit_ns();
    if (BN == 256) return launch_rdx<256>(ml, mw, mo, P, st);
    return launch_rdx<128>(ml, mw, mo, P, st);
}

}  // namespace moe
