// SwiGLU experts as grouped GEMMs on the sm_100-family tensor cores (tcgen05, TMEM, TMA).
//
// "The whole stack, in the open" (Apex-3), "What's inside", row "Fine-grained MoE": the
// experts run as grouped GEMMs. Handbook summary, section 2.5: a bias-free SwiGLU expert
// has three weight matrices (gate, up, down).
//
// One persistent kernel template serves every GEMM of the layer:
//   G1  [a|u] = X W_g^T, X W_u^T      two accumulators, SwiGLU in the epilogue (A, U, H out)
//   G2  Y = H W_d^T
//   B2  dH = dY W_d, SwiGLU backward in the epilogue (dA, dU out)
//   B4  dX = dA W_g + dU W_u          K split over two operand pairs
//   B3  dW_d[e] = dY_e^T H_e           weight gradients: K runs over expert e's rows
//   B5  dW_g[e] = dA_e^T X_e, dW_u[e] = dU_e^T X_e
// Row tiles are 128 rows of the expert-major layout, whose segments are padded to 128
// rows, so every tile belongs to one expert and is found from row_offsets on the device
// (no host synchronisation). Roles per CTA (384 threads, or 640 with sixteen epilogue warps,
// one CTA per SM):
//   warp 0  TMA producer (one thread): operand tiles into a ring of shared-memory stages;
//   warp 1  MMA issuer (one thread): tcgen05.mma 128 x N x 16 steps into a TMEM accumulator;
//   warp 2  allocates / frees tensor memory (two accumulators, double-buffered);
//   warps 4-11 epilogue: tcgen05.ld of TMEM lanes 0-127 (one output row per thread; warps w
//            and w + 4 share a lane quadrant and take one half of the columns each), the
//            fused elementwise step, bf16 outputs. Token-major outputs (G1, G2, B2, B4) are
//            packed into swizzled shared-memory boxes and written by TMA stores; B2 reads
//            its saved a and u through TMA-staged boxes; weight gradients store per thread.
//            Two warps per quadrant double the loads and stores in flight; GEMMs with a
//            reduction of at most 1024 (G1) or 512 (G2) take four per quadrant (warps 4-19), as their main
//            loop is shorter than eight warps' epilogue of the previous tile.
// Pair mode (a cluster of two CTAs on two SMs): the leading CTA issues
// tcgen05.mma.cta_group::2 over a 256-row tile; each CTA stages its own 128 rows of A and
// half of the tile's B columns, so per SM the shared-memory operand traffic and the TMA
// bytes per FLOP drop by a third compared with a 128 x 256 tile on one SM. Both CTAs' TMA
// loads complete on the leader's "full" barriers, the leader's commits arrive on both
// CTAs' barriers (multicast), and both epilogues release the accumulator to the leader.
// Operand tiles use the 128-byte swizzle. K-major tiles are TMA boxes of 64 K-elements x
// rows; MN-major tiles are boxes of 64 MN-elements x 64 k-rows. Every wait on an mbarrier
// is bounded in time; a wait that runs out records MOE_ERR_TIMEOUT, stops every role of
// the CTA and the kernel frees its tensor memory before returning.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "sizes.h"
#include "tmap.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;        // bf16 K elements per stage (128 bytes per row)
constexpr int BK_FP8 = 128;   // E4M3 K elements per stage (also 128 bytes per row)
constexpr int kEpiWarps = 8;  // default: two per TMEM lane quadrant, each half the columns
constexpr int kSmemBudget = 200 * 1024;

enum Epi : int { kEpiSwigluFwd = 0, kEpiStore = 1, kEpiSwigluBwd = 2 };
// SwiGLU backward: each epilogue warp stages the saved a and u of its 32 rows by TMA, kAuCols
// columns per chunk, kAuBufs chunks deep; the ring of operand stages gets what is left of
// kSmemBudgetAu.
constexpr int kAuCols = 16;
constexpr int kAuBufs = 2;
constexpr int kSmemBudgetAu = 220 * 1024;
// Token-major epilogues stage their outputs in shared memory, 16 columns x 32 rows per warp
// and output, and write them with TMA stores: two buffers deep, or one for the SwiGLU
// backward, whose operand ring then keeps a fifth stage (what bounds it at K = 4096).
constexpr int kOutCols = 16;

template <int BN_, bool A_MN_, bool B_MN_, bool DUAL_, int EPI_, bool TWO_K_, bool WGRAD_,
          bool PAIR_ = false, bool FP8_ = false, int OC_ = kOutCols, int EW_ = kEpiWarps>
struct Cfg {
    // epilogue warps: 8 (two per TMEM lane quadrant), or 16 for GEMMs whose reduction is so
    // short that the epilogue, not the tensor cores, sets the pace (at most 96 registers)
    static constexpr int EW = EW_;
    static constexpr int THREADS = 128 + 32 * EW;
    static_assert(EW == 8 || EW == 16, "epilogue warps");
    static constexpr bool FP8 = FP8_;        // E4M3 operands with row / column scales
    static constexpr int KB = FP8 ? BK_FP8 : BK;  // K elements per stage
    static constexpr int BN = BN_;           // output columns per tile (per B matrix if DUAL)
    static constexpr bool A_MN = A_MN_;
    static constexpr bool B_MN = B_MN_;
    static constexpr bool DUAL = DUAL_;      // two B operands -> gate and up accumulators (G1)
    static constexpr int EPI = EPI_;
    static constexpr bool TWO_K = TWO_K_;    // K = [K0 from (a0,b0)] ++ [K1 from (a1,b1)]
    static constexpr bool WGRAD = WGRAD_;    // M = weight rows, K = expert's token rows
    static constexpr bool PAIR = PAIR_;      // CTA pair: 256-row tiles, B split between CTAs
    static constexpr int MMA_N = DUAL ? 2 * BN : BN;         // accumulator columns per row
    static constexpr int BROWS = PAIR ? MMA_N / 2 : MMA_N;   // B rows staged by this CTA
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;        // rows of one (pair) tile
    static constexpr int A_BYTES = BM * 128;     // 128-byte rows in either type
    static constexpr int B_BYTES = BROWS * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // this CTA's bytes per K block
    static constexpr bool AU = EPI == kEpiSwigluBwd;
    static constexpr int AU_BUF_BYTES = 2 * 32 * kAuCols * 2;  // a and u: 32 rows x kAuCols
    static constexpr int AU_BYTES = AU ? EW * kAuBufs * AU_BUF_BYTES : 0;
    static constexpr bool TS = !WGRAD;  // token-major outputs leave by TMA stores
    static constexpr int NOUT = EPI == kEpiSwigluFwd ? 3 : EPI == kEpiSwigluBwd ? 2 : 1;
    // output columns per staged chunk: 16, or 32 (single-output epilogues of short-K GEMMs,
    // where the per-chunk fence and store issue dominate) at the same shared-memory size
    static constexpr int OCOLS = OC_;
    static_assert(OCOLS == 16 || (OCOLS == 32 && NOUT == 1 && !AU), "output chunk width");
    static constexpr int OUT_BOX_BYTES = 32 * OCOLS * 2;             // one output, one chunk
    static constexpr int OUT_BUF_BYTES = NOUT * OUT_BOX_BYTES;       // one chunk, every output
    static constexpr int OUT_DEPTH = (AU || OCOLS == 32 || EW == 16) ? 1 : 2;  // chunks per warp
    static constexpr int OUT_BYTES = TS ? EW * OUT_DEPTH * OUT_BUF_BYTES : 0;
    static constexpr int BUDGET = (AU || TS ? kSmemBudgetAu : kSmemBudget) - AU_BYTES - OUT_BYTES;
    static constexpr int STAGES = (BUDGET / STAGE_BYTES) > 6 ? 6 : (BUDGET / STAGE_BYTES);
    static constexpr int ACC_COLS = MMA_N;
    static constexpr int TMEM_COLS = 2 * ACC_COLS;  // two accumulator buffers
    // DUAL: the W_g and W_u boxes form one 2*BN-row B tile (on one CTA, back to back; in a
    // pair, W_g on the leader and W_u on the peer), so one instruction fills gate columns
    // [0, BN) and up columns [BN, 2BN).
    static constexpr uint32_t IDESC = idesc_mma(MMA_N, TILE_M, A_MN, B_MN, FP8);
    static_assert(!FP8 || (!A_MN && !B_MN && !WGRAD && !TWO_K), "FP8: forward K-major GEMMs");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "tensor memory columns");
    static_assert(BN % 64 == 0 && MMA_N <= 256 && BROWS % 64 == 0, "tile width");
    static constexpr size_t MISC_BYTES = 512 + sizeof(int64_t) * (kMaxExperts + 1) +
                                         sizeof(int32_t) * kMaxExperts +
                                         sizeof(int32_t) * (kMaxExperts + 1);
    static constexpr size_t SMEM_BYTES =
        1024 + (size_t)STAGES * STAGE_BYTES + AU_BYTES + OUT_BYTES + MISC_BYTES;
    static_assert((2 * STAGES + 4 + EW * kAuBufs) * 8 + 8 <= 512, "barrier block");

};

struct Params {
    const int64_t* row_offsets;  // padded expert segments, or null = one dense expert
    const int32_t* expert_order; // weight gradients: experts in descending row count
    int64_t rows;                // extent of the token dimension
    int E;
    int N;      // output columns
    int K0;     // token-major: reduction length of operand pair 0
    int K1;     // token-major: reduction length of operand pair 1 (TWO_K)
    int M_out;  // weight gradients: rows of each expert's output
    int nprob;  // weight gradients: (a0,out0) and, if 2, (a1,out1)
    int kb_per_expert;  // B operand rows per expert (MN-major weights: K extent per expert)
    // weight gradients: the outputs of problems 0 and 1 (token-major outputs leave through
    // the output tensor maps instead)
    __nv_bfloat16* out0;
    __nv_bfloat16* out1;
    const float* sa;           // FP8: scale of each A row (indexed by the global row)
    const float* sb0;          // FP8: scale of each B row (output channel), first B operand
    const float* sb1;          // FP8: second B operand (W_u of G1)
    const float* row_scale;    // gate folded into the expert: G1 writes g*h, B2 forms g*dh
    float* gate_part;          // B2 with row_scale: per row, (dy W_d) . h per 64 columns
    int ld_out;                // B2: output columns; gate_part holds ld_out / 64 per row
    // B4 with the router's input-gradient term in the rows: row += r1_row[row] * r1_col[e][col]
    // (the slot's logit gradient times its expert's router row, both fp32)
    const float* r1_row;
    const float* r1_col;
    int* status;
    uint64_t wait_limit_ns;
};

struct TileInfo {
    int e;       // expert
    int p;       // weight-gradient problem (0 or 1)
    int64_t m0;  // token-major: first row; weight gradients: first output row
    int n0;      // first output column
    int64_t k_lo;  // weight gradients: first token row of the expert
    int k_iters;   // 64-wide K blocks
    int64_t row_end;  // token-major: rows at or past this are not stored
};

struct SmemLayout {
    uint8_t* a;        // STAGES x A tile
    uint8_t* b;        // STAGES x B tile(s)
    uint64_t* full;    // STAGES
    uint64_t* empty;   // STAGES
    uint64_t* tfull;   // 2
    uint64_t* tempty;  // 2
    uint32_t* tmem_slot;
    int* abort_flag;
    int64_t* offs;     // E + 1
    int32_t* order;    // E
    int32_t* ptp;      // E + 1: exclusive prefix of pair tiles per expert (pair, token-major)
    uint8_t* au;       // SwiGLU backward: EW x kAuBufs staged (a | u) chunks
    uint64_t* au_full; // EW x kAuBufs
    uint8_t* ob;       // TMA-store epilogues: EW x OUT_DEPTH staged output chunks
};

template <class C>
__device__ __forceinline__ SmemLayout carve(uint8_t* raw) {
    SmemLayout s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = base + (size_t)C::STAGES * C::A_BYTES;
    s.au = base + (size_t)C::STAGES * C::STAGE_BYTES;  // 1024-aligned: stage sizes are
    s.ob = s.au + C::AU_BYTES;  // 1024-aligned: the a/u buffers are whole KB
    uint8_t* misc = s.ob + C::OUT_BYTES;
    s.full = reinterpret_cast<uint64_t*>(misc);
    s.empty = s.full + C::STAGES;
    s.tfull = s.empty + C::STAGES;
    s.tempty = s.tfull + 2;
    s.au_full = s.tempty + 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.au_full + (C::AU ? C::EW * kAuBufs : 0));
    s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
    s.offs = reinterpret_cast<int64_t*>(misc + 512);
    s.order = reinterpret_cast<int32_t*>(s.offs + kMaxExperts + 1);
    s.ptp = s.order + kMaxExperts;
    return s;
}

__device__ __forceinline__ int64_t cdiv_dev(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <class C>
__device__ __forceinline__ int64_t total_tiles(const Params& P, const SmemLayout& S) {
    const int n_tiles = P.N / C::BN;
    if constexpr (C::WGRAD) {
        return (int64_t)P.E * P.nprob * (P.M_out / C::TILE_M) * n_tiles;
    } else {
        int64_t mt;
        if (!P.row_offsets) mt = cdiv_dev(P.rows, C::TILE_M);
        else if (C::PAIR) mt = S.ptp[P.E];
        else mt = S.offs[P.E] / BM;
        return mt * n_tiles;
    }
}

// Last expert e in [0, E) with key[e] <= v (key non-decreasing). Among equal keys (empty
// experts) the last one is the expert that owns the rows.
template <class K>
__device__ __forceinline__ int last_le(const K* key, int E, int64_t v) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)key[mid] <= v) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Tile `tile` as seen by CTA `rank` of its pair (rank 0 outside pair mode).
template <class C>
__device__ __forceinline__ TileInfo decode(int64_t tile, const Params& P, const SmemLayout& S,
                                           uint32_t rank) {
    TileInfo ti;
    const int n_tiles = P.N / C::BN;
    const int64_t half = C::PAIR ? (int64_t)rank * BM : 0;
    if constexpr (C::WGRAD) {
        const int m_tiles = P.M_out / C::TILE_M;
        const int64_t per_e = (int64_t)P.nprob * m_tiles * n_tiles;
        const int oi = (int)(tile / per_e);
        int64_t rem = tile % per_e;
        ti.e = S.order[oi];
        ti.p = (int)(rem / (m_tiles * n_tiles));
        rem %= (m_tiles * n_tiles);
        ti.m0 = (rem / n_tiles) * C::TILE_M + half;
        ti.n0 = (int)(rem % n_tiles) * C::BN;
        int64_t lo = 0, hi = P.rows;
        if (P.row_offsets) {
            lo = S.offs[ti.e];
            hi = S.offs[ti.e + 1];
        }
        ti.k_lo = lo;
        ti.k_iters = (int)cdiv_dev(hi - lo, BK);
        ti.row_end = P.M_out;
    } else {
        const int64_t mt = tile / n_tiles;
        ti.n0 = (int)(tile % n_tiles) * C::BN;
        ti.p = 0;
        ti.k_lo = 0;
        ti.e = 0;
        if (!P.row_offsets) {
            ti.m0 = mt * C::TILE_M + half;
            ti.row_end = P.rows;
        } else if constexpr (C::PAIR) {
            // pair tiles of expert e cover its padded segment 256 rows at a time; the
            // second half of a segment's last pair tile may lie past the segment
            ti.e = last_le(S.ptp, P.E, mt);
            ti.m0 = S.offs[ti.e] + (mt - S.ptp[ti.e]) * C::TILE_M + half;
            ti.row_end = S.offs[ti.e + 1];
        } else {
            ti.m0 = mt * BM;
            ti.e = last_le(S.offs, P.E, ti.m0);
            ti.row_end = S.offs[ti.e + 1];
        }
        ti.k_iters = (P.K0 + (C::TWO_K ? P.K1 : 0)) / C::KB;
    }
    return ti;
}

template <class C>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                         int32_t c0, int32_t c1) {
    if constexpr (C::PAIR) tma_load_2d_pair(dst, map, bar, c0, c1);
    else tma_load_2d(dst, map, bar, c0, c1);
}

// Loads of K block `kb` of a tile into this CTA's stage buffers; `bar` is the barrier the
// copies complete on (in pair mode the leader's, as a shared::cluster address).
template <class C>
__device__ __forceinline__ void issue_loads(const TileInfo& ti, int kb, uint32_t a_dst,
                                            uint32_t b_dst, uint32_t bar, const Params& P,
                                            const CUtensorMap* ma0, const CUtensorMap* ma1,
                                            const CUtensorMap* mb0, const CUtensorMap* mb1,
                                            uint32_t rank) {
    const int32_t bhalf = C::PAIR ? (int32_t)rank * C::BROWS : 0;  // this CTA's B columns
    if constexpr (C::WGRAD) {
        const int32_t krow = (int32_t)(ti.k_lo + (int64_t)kb * BK);
        const CUtensorMap* ma = ti.p == 0 ? ma0 : ma1;
        // A: MN-major, two 64-wide boxes along M
        tma_load<C>(a_dst, ma, bar, (int32_t)ti.m0, krow);
        tma_load<C>(a_dst + 8192, ma, bar, (int32_t)ti.m0 + 64, krow);
#pragma unroll
        for (int j = 0; j < C::BROWS / 64; ++j)
            tma_load<C>(b_dst + j * 8192, mb0, bar, ti.n0 + bhalf + 64 * j, krow);
    } else {
        int kk = kb * C::KB;
        const CUtensorMap* ma = ma0;
        const CUtensorMap* mb = mb0;
        int kper = P.kb_per_expert;
        if (C::TWO_K && kk >= P.K0) {
            kk -= P.K0;
            ma = ma1;
            mb = mb1;
        }
        tma_load<C>(a_dst, ma, bar, kk, (int32_t)ti.m0);
        if constexpr (C::B_MN) {
            const int32_t brow = ti.e * kper + kk;
#pragma unroll
            for (int j = 0; j < C::BROWS / 64; ++j)
                tma_load<C>(b_dst + j * 8192, mb, bar, ti.n0 + bhalf + 64 * j, brow);
        } else if constexpr (C::DUAL) {
            const int32_t brow = ti.e * P.N + ti.n0;
            if constexpr (C::PAIR) {
                tma_load<C>(b_dst, rank == 0 ? mb0 : mb1, bar, kk, brow);
            } else {
                tma_load<C>(b_dst, mb0, bar, kk, brow);
                tma_load<C>(b_dst + C::BN * 128, mb1, bar, kk, brow);
            }
        } else {
            tma_load<C>(b_dst, mb, bar, kk, ti.e * P.N + ti.n0 + bhalf);
        }
    }
}

__device__ __forceinline__ uint4 pack_chunk8(const float* v) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// FP8 dequantisation of a 32-column accumulator chunk: value * scale(A row) * scale(B row
// of each output column). With dual=true, `a` takes the first B operand's column scales
// and `b` the second's (G1: gate and up); otherwise only `a` is scaled.
template <int W = 32>
__device__ __forceinline__ void fp8_scale(float* a, float* b, const Params& P, int64_t row,
                                          const TileInfo& ti, int c, bool dual = true) {
    const float sr = __ldg(P.sa + row);
    const int64_t col0 = (int64_t)ti.e * P.N + ti.n0 + c;
    const float4* s0 = reinterpret_cast<const float4*>(P.sb0 + col0);
#pragma unroll
    for (int q = 0; q < W / 4; ++q) {
        const float4 v = __ldg(s0 + q);
        a[4 * q] *= sr * v.x;
        a[4 * q + 1] *= sr * v.y;
        a[4 * q + 2] *= sr * v.z;
        a[4 * q + 3] *= sr * v.w;
    }
    if (dual) {
        const float4* s1 = reinterpret_cast<const float4*>(P.sb1 + col0);
#pragma unroll
        for (int q = 0; q < W / 4; ++q) {
            const float4 v = __ldg(s1 + q);
            b[4 * q] *= sr * v.x;
            b[4 * q + 1] *= sr * v.y;
            b[4 * q + 2] *= sr * v.z;
            b[4 * q + 3] *= sr * v.w;
        }
    }
}

// Weight-gradient epilogue: columns [c_lo, c_hi) of this thread's output row (a weight row;
// always inside the output, as M_out and N are whole tiles). An expert with no rows gives
// zeros.
template <class C>
__device__ __forceinline__ void epilogue_wgrad(const TileInfo& ti, uint32_t t_acc, int row_in_tile,
                                               const Params& P, int c_lo, int c_hi) {
    static_assert(C::WGRAD, "weight-gradient tiles only");
    const int64_t row = ti.m0 + row_in_tile;
    __nv_bfloat16* out = (ti.p == 0 ? P.out0 : P.out1) + ((int64_t)ti.e * P.M_out + row) * P.N + ti.n0;
    for (int c = c_lo; c < c_hi; c += 32) {
        float v[32];
        if (ti.k_iters > 0) {
            uint32_t r[32];
            tmem_ld32(t_acc + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = pack_chunk8(v + 8 * q);
    }
}

// ------------------------------------------------------- epilogues with TMA stores
// Each epilogue warp owns 32 rows x (BN / 2) columns of the tile and walks them in chunks of
// kOutCols. Per chunk its lanes pack their rows of every output into a shared-memory buffer
// laid out as the 32-byte-swizzled TMA box (kOutCols x 32 rows), and lane 0 stores the boxes;
// a buffer is rewritten only after the store that read it two chunks earlier is done.
// A 128-row half of a pair tile that lies past the expert's segment stores nothing (such a
// half is wholly inside or wholly outside, as segments are padded to 128 rows); rows past
// the end of the output tensor are clipped by the stores themselves.

// Byte offset of 16-byte piece j of row r in a 32-byte-swizzled box of 32-byte rows.
__device__ __forceinline__ int sw32_offset(int r, int j) { return r * 32 + ((j ^ ((r >> 2) & 1)) << 4); }
// ... and in a 64-byte-swizzled box of 64-byte rows (32 bf16 columns).
__device__ __forceinline__ int sw64_offset(int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); }

template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[W]) {
    if constexpr (W == 32) tmem_ld32(taddr, r);
    else if constexpr (W == 16) tmem_ld16(taddr, r);
    else tmem_ld8(taddr, r);
}


template <class C>
__device__ __forceinline__ void epilogue_tma_store(const SmemLayout& S, const TileInfo& ti,
                                                   uint32_t t_acc, int q, int lane, int slot,
                                                   int c_lo, int ncols, const Params& P,
                                                   const CUtensorMap* mo0, const CUtensorMap* mo1,
                                                   const CUtensorMap* mo2, uint32_t& n) {
    constexpr int W = C::OCOLS;
    if (ti.m0 >= ti.row_end) return;  // warp-uniform: the whole half is past the segment
    const int64_t row0 = ti.m0 + 32 * q;
    // rows past row_end (the tail of an unpadded layout) are clipped by the store; their FP8
    // row scale is read from the last row instead
    const int64_t row = row0 + lane < ti.row_end ? row0 + lane : ti.row_end - 1;
    for (int i = 0; i < ncols / W; ++i, ++n) {
        const int c = c_lo + i * W;
        float v[C::NOUT][W];
        if constexpr (C::EPI == kEpiSwigluFwd) {
            uint32_t g[W], u[W];
            tmem_ld_cols<W>(t_acc + c, g);
            tmem_ld_cols<W>(t_acc + C::BN + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < W; ++j) {
                v[0][j] = __uint_as_float(g[j]);
                v[1][j] = __uint_as_float(u[j]);
            }
            if constexpr (C::FP8) fp8_scale<W>(v[0], v[1], P, row, ti, c);
            const float rg = P.row_scale ? __ldg(P.row_scale + row) : 1.0f;
#pragma unroll
            for (int j = 0; j < W; ++j)
                v[2][j] = v[0][j] / (1.0f + __expf(-v[0][j])) * v[1][j] * rg;
        } else {
            uint32_t r[W];
            tmem_ld_cols<W>(t_acc + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < W; ++j) v[0][j] = __uint_as_float(r[j]);
            if constexpr (C::FP8) fp8_scale<W>(v[0], v[0], P, row, ti, c, /*dual=*/false);
            if constexpr (C::EPI == kEpiStore && !C::WGRAD) {
                if (P.r1_row) {  // the slot's router term, one fp32 FMA per element
                    const float g = __ldg(P.r1_row + row);
                    const float4* w = reinterpret_cast<const float4*>(
                        P.r1_col + (int64_t)ti.e * P.N + ti.n0 + c);
#pragma unroll
                    for (int j = 0; j < W / 4; ++j) {
                        const float4 w4 = __ldg(w + j);
                        v[0][4 * j] = fmaf(g, w4.x, v[0][4 * j]);
                        v[0][4 * j + 1] = fmaf(g, w4.y, v[0][4 * j + 1]);
                        v[0][4 * j + 2] = fmaf(g, w4.z, v[0][4 * j + 2]);
                        v[0][4 * j + 3] = fmaf(g, w4.w, v[0][4 * j + 3]);
                    }
                }
            }
        }
        uint8_t* buf = S.ob + ((size_t)slot * C::OUT_DEPTH + n % C::OUT_DEPTH) * C::OUT_BUF_BYTES;
        if (lane == 0) bulk_wait_read<C::OUT_DEPTH - 1>();  // the store that last read it is done
        __syncwarp();
#pragma unroll
        for (int o = 0; o < C::NOUT; ++o)
#pragma unroll
            for (int j = 0; j < W / 8; ++j)
                *reinterpret_cast<uint4*>(buf + o * C::OUT_BOX_BYTES +
                                          (W == 32 ? sw64_offset(lane, j) : sw32_offset(lane, j))) =
                    pack_chunk8(v[o] + 8 * j);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            const CUtensorMap* mo[3] = {mo0, mo1, mo2};
#pragma unroll
            for (int o = 0; o < C::NOUT; ++o)
                tma_store_2d(mo[o], smem_u32(buf + o * C::OUT_BOX_BYTES), ti.n0 + c, (int32_t)row0);
            bulk_commit();
        }
    }
}

// ------------------------------------------------- SwiGLU backward with staged a and u
// Each epilogue warp owns 32 rows x (BN / 2) columns of the tile and walks them in chunks of
// kAuCols. The chunk's saved a and u arrive by TMA (boxes of kAuCols x 32 rows, swizzled
// so that the row-per-lane reads below hit distinct banks) into one of the warp's kAuBufs
// buffers; lane 0 issues the copy of chunk n + kAuBufs once the warp is done with chunk n,
// and a tile's first chunks before its accumulator is ready.

// Byte offset of 16-byte piece j of row r in a staged (a or u) chunk.
__device__ __forceinline__ int au_offset(int r, int j) {
    if constexpr (kAuCols == 32) return r * 64 + ((j ^ ((r >> 1) & 3)) << 4);  // 64-byte swizzle
    else if constexpr (kAuCols == 16) return r * 32 + ((j ^ ((r >> 2) & 1)) << 4);  // 32-byte
    else return r * 16;                                                            // unswizzled
}

template <class C>
__device__ __forceinline__ void au_issue(const SmemLayout& S, const CUtensorMap* ma,
                                         const CUtensorMap* mu, int slot, uint32_t n, int64_t row0,
                                         int col) {
    const int b = (int)(n % kAuBufs);
    const uint32_t dst = smem_u32(S.au + ((size_t)slot * kAuBufs + b) * C::AU_BUF_BYTES);
    const uint32_t bar = smem_u32(&S.au_full[slot * kAuBufs + b]);
    // relaxed: the buffer's previous contents were read into registers and used before the
    // warp synchronised, and the fill orders no earlier store of this thread; a releasing
    // arrive would wait for the warp's dA/dU stores to drain (measured: B2 1.7% slower)
    mbar_arrive_expect_tx_relaxed(bar, C::AU_BUF_BYTES);
    tma_load_2d(dst, ma, bar, col, (int32_t)row0);
    tma_load_2d(dst + C::AU_BUF_BYTES / 2, mu, bar, col, (int32_t)row0);
}

// One tile of this warp's columns [c_lo, c_lo + ncols). `n` counts the warp's chunks over the
// kernel's life (it picks buffer and phase). Returns false when a wait failed (uniform
// across the warp).
template <class C>
__device__ __forceinline__ bool swiglu_bwd_staged(const SmemLayout& S, const TileInfo& ti,
                                                  uint32_t t_acc, int q, int lane, int slot,
                                                  int c_lo, int ncols, const Params& P,
                                                  const CUtensorMap* ma, const CUtensorMap* mu,
                                                  const CUtensorMap* mda, const CUtensorMap* mdu,
                                                  uint32_t& n, volatile int* abort_flag) {
    static_assert(kAuCols == kOutCols, "one staged output chunk per a/u chunk");
    const int nch = ncols / kAuCols;
    const int64_t row0 = ti.m0 + 32 * q;
    const int64_t row = row0 + lane;
    const bool ok_row = row < ti.row_end;
    // padded segments are whole 128-row halves, so a warp's rows are all inside or all past
    // the segment; rows past an unpadded layout's end are clipped by the store
    const bool store = row0 < ti.row_end;
    // gate folded into the expert: dy is the ungated row gradient, dh = g (dy W_d), and the
    // gate's gradient (dy W_d) . h is summed per 64-column group (h recomputed in fp32)
    const float g = (P.row_scale && ok_row) ? __ldg(P.row_scale + row) : 1.0f;
    float gpart = 0.f;
    for (int i = 0; i < nch; ++i, ++n) {
        const int c = c_lo + i * kAuCols;
        const int b = (int)(n % kAuBufs);
        uint32_t acc[kAuCols];
        tmem_ld_cols<kAuCols>(t_acc + c, acc);
        bool ok = mbar_wait_bounded(smem_u32(&S.au_full[slot * kAuBufs + b]), (n / kAuBufs) & 1u,
                                    abort_flag, P.status, P.wait_limit_ns, 34);
        tmem_ld_wait();
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        float dav[kAuCols], duv[kAuCols];
        if (store) {  // lanes past an unpadded layout's end see zero-filled a, u and acc
            const uint8_t* abuf = S.au + ((size_t)slot * kAuBufs + b) * C::AU_BUF_BYTES;
            const uint8_t* ubuf = abuf + C::AU_BUF_BYTES / 2;
            float accf[kAuCols];
#pragma unroll
            for (int j = 0; j < kAuCols; ++j) accf[j] = __uint_as_float(acc[j]);
            // FP8 operands: the dequantised r = (dy codes) (W_d codes) * scale(row) * scale(col)
            if constexpr (C::FP8)
                fp8_scale<kAuCols>(accf, accf, P, ok_row ? row : ti.row_end - 1, ti, c, false);
#pragma unroll
            for (int j = 0; j < kAuCols / 8; ++j) {
                const uint4 a4 = *reinterpret_cast<const uint4*>(abuf + au_offset(lane, j));
                const uint4 u4 = *reinterpret_cast<const uint4*>(ubuf + au_offset(lane, j));
                const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w};
                const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const float a = (h & 1) ? bf16_hi(aw[h >> 1]) : bf16_lo(aw[h >> 1]);
                    const float u = (h & 1) ? bf16_hi(uw[h >> 1]) : bf16_lo(uw[h >> 1]);
                    const float acc_h = accf[8 * j + h];
                    const float sa = 1.0f / (1.0f + __expf(-a));
                    if (P.gate_part) gpart = fmaf(acc_h, a * sa * u, gpart);
                    const float dh = acc_h * g;
                    dav[8 * j + h] = dh * u * sa * (1.0f + a * (1.0f - sa));
                    duv[8 * j + h] = dh * a * sa;
                }
            }
            const int col = ti.n0 + c;
            if (P.gate_part && (col + kAuCols) % 64 == 0) {  // last chunk of a 64-column group
                if (ok_row) P.gate_part[row * (int64_t)(P.ld_out / 64) + col / 64] = gpart;
                gpart = 0.f;
            }
        }
        __syncwarp();  // every lane is done with a/u buffer b
        if (lane == 0 && i + kAuBufs < nch)
            au_issue<C>(S, ma, mu, slot, n + kAuBufs, row0, ti.n0 + c + kAuBufs * kAuCols);
        if (store) {
            uint8_t* ob = S.ob + ((size_t)slot * C::OUT_DEPTH + n % C::OUT_DEPTH) * C::OUT_BUF_BYTES;
            if (lane == 0) bulk_wait_read<C::OUT_DEPTH - 1>();  // the store that last read it is done
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kAuCols / 8; ++j) {
                *reinterpret_cast<uint4*>(ob + sw32_offset(lane, j)) = pack_chunk8(dav + 8 * j);
                *reinterpret_cast<uint4*>(ob + 1024 + sw32_offset(lane, j)) = pack_chunk8(duv + 8 * j);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(mda, smem_u32(ob), ti.n0 + c, (int32_t)row0);
                tma_store_2d(mdu, smem_u32(ob + 1024), ti.n0 + c, (int32_t)row0);
                bulk_commit();
            }
        }
    }
    return true;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap ma0,
                        const __grid_constant__ CUtensorMap ma1,
                        const __grid_constant__ CUtensorMap mb0,
                        const __grid_constant__ CUtensorMap mb1,
                        const __grid_constant__ CUtensorMap mo0,
                        const __grid_constant__ CUtensorMap mo1,
                        const __grid_constant__ CUtensorMap mo2, const Params P) {
    extern __shared__ uint8_t gg_smem_raw[];
    const SmemLayout S = carve<C>(gg_smem_raw);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const uint32_t rank = C::PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // tiles are dealt to CTAs (or to pairs, whose two CTAs take the same tile)
    const int64_t first_tile = C::PAIR ? blockIdx.x / 2 : blockIdx.x;
    const int64_t tile_step = C::PAIR ? gridDim.x / 2 : gridDim.x;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);
            mbar_init(smem_u32(&S.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&S.tfull[b]), 1);
            mbar_init(smem_u32(&S.tempty[b]), C::PAIR ? 2 * C::EW : C::EW);
        }
        if constexpr (C::AU)
            for (int b = 0; b < C::EW * kAuBufs; ++b) mbar_init(smem_u32(&S.au_full[b]), 1);
        *S.abort_flag = 0;
        fence_mbar_init();
    }
    if (P.row_offsets)
        for (int i = tid; i <= P.E; i += C::THREADS) S.offs[i] = P.row_offsets[i];
    if (C::WGRAD)
        for (int i = tid; i < P.E; i += C::THREADS) S.order[i] = P.expert_order ? P.expert_order[i] : i;
    if (warp == 2) {
        if constexpr (C::PAIR) {
            tmem_alloc_pair(smem_u32(S.tmem_slot), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(S.tmem_slot), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    if constexpr (C::PAIR && !C::WGRAD) {
        // pair tiles per expert = ceil(128-row tiles / 2); exclusive prefix in S.ptp
        __syncthreads();
        if (P.row_offsets) {
            int v = 0;
            if (tid < P.E) v = (int)(((S.offs[tid + 1] - S.offs[tid]) / BM + 1) / 2);
            if (tid < kMaxExperts) S.ptp[tid + 1] = v;
            if (tid == 0) S.ptp[0] = 0;
            __syncthreads();
            for (int off = 1; off < kMaxExperts; off <<= 1) {  // inclusive scan of S.ptp[1..256]
                int add = 0;
                if (tid >= off && tid < kMaxExperts) add = S.ptp[tid + 1 - off];
                __syncthreads();
                if (tid < kMaxExperts) S.ptp[tid + 1] += add;
                __syncthreads();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (C::PAIR) cluster_sync();  // the peer's barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *S.tmem_slot;
    volatile int* abort_flag = S.abort_flag;

    // the padded layout: offsets start at 0, never decrease, every segment is a whole number
    // of 128-row tiles and the last ends within the row capacity; anything else is reported
    // and the launch does no work (the same decision in every CTA)
    bool bad_offs = false;
    if (P.row_offsets && tid < P.E) {
        const int64_t lo = S.offs[tid], hi = S.offs[tid + 1];
        bad_offs = hi < lo || (hi - lo) % BM != 0 || (tid == 0 && lo != 0);
    }
    bool layout_ok = !__syncthreads_or(bad_offs);
    if (P.row_offsets && S.offs[P.E] > P.rows) layout_ok = false;
    if (!layout_ok && tid == 0) record_error(P.status, MOE_ERR_BAD_INDEX, 20);
    const int64_t ntiles = layout_ok ? total_tiles<C>(P, S) : 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        tma_prefetch_desc(&ma0);
        tma_prefetch_desc(&mb0);
        if (C::TWO_K || C::WGRAD) tma_prefetch_desc(&ma1);
        if (C::TWO_K || C::DUAL) tma_prefetch_desc(&mb1);
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t tile = first_tile; tile < ntiles; tile += tile_step) {
            const TileInfo ti = decode<C>(tile, P, S, rank);
            bool ok = true;
            for (int kb = 0; kb < ti.k_iters; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&S.empty[stage]), phase ^ 1u, abort_flag, P.status,
                                       P.wait_limit_ns, 30)) {
                    ok = false;
                    break;
                }
                const uint32_t full = smem_u32(&S.full[stage]);
                uint32_t bar = full;
                if constexpr (C::PAIR) {
                    bar = mapa_shared(full, 0);  // both CTAs' copies complete on the leader's
                    if (leader) mbar_arrive_expect_tx(full, 2 * C::STAGE_BYTES);
                } else {
                    mbar_arrive_expect_tx(full, C::STAGE_BYTES);
                }
                issue_loads<C>(ti, kb, smem_u32(S.a + (size_t)stage * C::A_BYTES),
                               smem_u32(S.b + (size_t)stage * C::B_BYTES), bar, P, &ma0, &ma1,
                               &mb0, &mb1, rank);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        for (int64_t tile = first_tile; tile < ntiles; tile += tile_step, ++local) {
            const TileInfo ti = decode<C>(tile, P, S, rank);
            const int buf = local & 1;
            const uint32_t use = (local >> 1) & 1;
            if (!mbar_wait_bounded(smem_u32(&S.tempty[buf]), use ^ 1u, abort_flag, P.status,
                                   P.wait_limit_ns, 31))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + buf * C::ACC_COLS;
            bool ok = true;
            for (int kb = 0; kb < ti.k_iters; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&S.full[stage]), phase, abort_flag, P.status,
                                       P.wait_limit_ns, 32)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = smem_u32(S.a + (size_t)stage * C::A_BYTES);
                const uint32_t b_s = smem_u32(S.b + (size_t)stage * C::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 4 instructions of 32 bytes of K
                    const uint64_t adesc = C::A_MN ? sdesc_sw128(a_s + kk * 2048, 8192, 1024)
                                                   : sdesc_sw128(a_s + kk * 32, 16, 1024);
                    const uint64_t bdesc = C::B_MN ? sdesc_sw128(b_s + kk * 2048, 8192, 1024)
                                                   : sdesc_sw128(b_s + kk * 32, 16, 1024);
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (C::PAIR && C::FP8) umma_fp8_pair(d_tmem, adesc, bdesc, C::IDESC, acc);
                    else if constexpr (C::PAIR) umma_bf16_pair(d_tmem, adesc, bdesc, C::IDESC, acc);
                    else if constexpr (C::FP8) umma_fp8(d_tmem, adesc, bdesc, C::IDESC, acc);
                    else umma_bf16(d_tmem, adesc, bdesc, C::IDESC, acc);
                }
                if constexpr (C::PAIR) umma_commit_pair(smem_u32(&S.empty[stage]), 0x3);
                else umma_commit(smem_u32(&S.empty[stage]));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if constexpr (C::PAIR) umma_commit_pair(smem_u32(&S.tfull[buf]), 0x3);
            else umma_commit(smem_u32(&S.tfull[buf]));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp % 4;  // TMEM lanes 32q .. 32q+31 (a warp's rank in its warpgroup)
        const int row_in_tile = 32 * q + lane;
        constexpr int kCols = C::BN / (C::EW / 4);  // columns per epilogue warp
        static_assert(kCols % 32 == 0, "epilogue column split");
        const int c_lo = ((warp - 4) / 4) * kCols;
        const int slot = warp - 4;
        uint32_t n_au = 0;  // staged a/u chunks consumed by this warp
        int local = 0;
        for (int64_t tile = first_tile; tile < ntiles; tile += tile_step, ++local) {
            const TileInfo ti = decode<C>(tile, P, S, rank);
            const int buf = local & 1;
            const uint32_t ph = (local >> 1) & 1;
            if constexpr (C::AU) {  // this tile's first a/u chunks while the MMA runs
                if (lane == 0)
                    for (int i = 0; i < kAuBufs && i < kCols / kAuCols; ++i)
                        au_issue<C>(S, &ma1, &mb1, slot, n_au + i, ti.m0 + 32 * q,
                                    ti.n0 + c_lo + i * kAuCols);
            }
            bool ok = mbar_wait_bounded(smem_u32(&S.tfull[buf]), ph, abort_flag, P.status,
                                        P.wait_limit_ns, 33);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t t_acc = tmem_base + buf * C::ACC_COLS + ((uint32_t)(32 * q) << 16);
            if constexpr (C::AU) {
                if (!swiglu_bwd_staged<C>(S, ti, t_acc, q, lane, slot, c_lo, kCols, P, &ma1, &mb1,
                                          &mo0, &mo1, n_au, abort_flag))
                    break;
            } else if constexpr (C::TS) {
                epilogue_tma_store<C>(S, ti, t_acc, q, lane, slot, c_lo, kCols, P, &mo0, &mo1, &mo2,
                                      n_au);
            } else {
                epilogue_wgrad<C>(ti, t_acc, row_in_tile, P, c_lo, c_lo + kCols);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (C::PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&S.tempty[buf]), 0));
                else mbar_arrive(smem_u32(&S.tempty[buf]));
            }
        }
        if constexpr (C::TS) {
            if (lane == 0) bulk_wait<0>();  // this warp's stores are complete
        }
    }
    __syncwarp();
    __syncthreads();
    if constexpr (C::PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
    if (*abort_flag) {  // let copies still in flight land before the CTA exits
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
    if (warp == 2) {
        tc_fence_after();
        if constexpr (C::PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Experts in descending padded row count (ties: lower index), for the weight-gradient
// tile order: the longest reductions are scheduled first.
__global__ void expert_order_kernel(const int64_t* __restrict__ row_offsets, int E,
                                    int32_t* __restrict__ order) {
    const int e = threadIdx.x;
    if (e >= E) return;
    const int64_t ce = row_offsets[e + 1] - row_offsets[e];
    int rank = 0;
    for (int j = 0; j < E; ++j) {
        const int64_t cj = row_offsets[j + 1] - row_offsets[j];
        if (cj > ce || (cj == ce && j < e)) ++rank;
    }
    order[rank] = e;
}

// ---------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map over a row-major [outer, inner] matrix of bf16 (or of bytes, for E4M3 codes),
// 128-byte swizzled boxes.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer, bool bytes = false,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto enc = get_encoder();
    if (!enc || !base) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (bytes ? 1 : 2)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return enc(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps for the TMA-store epilogue: boxes of `cols` (16 or 32) x 32 rows over [rows, ld]
// bf16, swizzled as the epilogue lays them out (32- or 64-byte rows).
bool out_maps(CUtensorMap (&mo)[3], const void* o0, const void* o1, const void* o2, uint64_t ld,
              uint64_t rows, int cols = kOutCols) {
    const void* o[3] = {o0, o1 ? o1 : o0, o2 ? o2 : o0};
    const CUtensorMapSwizzle swz = cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    for (int i = 0; i < 3; ++i)
        if (!make_map(&mo[i], o[i], ld, rows, (uint32_t)cols, 32, false, swz)) return false;
    return true;
}

// `mo` (TMA-store configurations only): the output maps from out_maps.
template <class C>
int launch(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
           const CUtensorMap& b1, const Params& P, int64_t max_tiles, cudaStream_t st,
           const CUtensorMap* mo = nullptr) {
    static_assert(C::SMEM_BYTES <= 227 * 1024, "shared memory");
    if (C::TS && !mo) return MOE_ERR_LAUNCH;
    const CUtensorMap& o0 = mo ? mo[0] : a0;
    const CUtensorMap& o1 = mo ? mo[1] : a0;
    const CUtensorMap& o2 = mo ? mo[2] : a0;
    auto kern = grouped_gemm_kernel<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_BYTES) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    if constexpr (C::PAIR) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2));
        int clusters = 0;  // pairs that fit on the GPU at once (one CTA per SM)
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1)
            clusters = sm_count() / 2;
        int64_t pairs = clusters;
        if (max_tiles < pairs) pairs = max_tiles;
        if (pairs < 1) pairs = 1;
        cfg.gridDim = dim3(2 * (unsigned)pairs);
        if (cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, o0, o1, o2, P) != cudaSuccess)
            return MOE_ERR_LAUNCH;
        return launch_status();
    } else {
        int64_t grid = sm_count();
        if (max_tiles < grid) grid = max_tiles;
        if (grid < 1) grid = 1;
        kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, st>>>(a0, a1, b0, b1, o0, o1, o2, P);
        return launch_status();
    }
}

// Configurations of the layer's GEMMs (P: CTA-pair versions).
using CfgG1 = Cfg<128, false, false, true, kEpiSwigluFwd, false, false>;
using CfgG1P = Cfg<128, false, false, true, kEpiSwigluFwd, false, false, true>;
template <int BN> using CfgStoreK = Cfg<BN, false, false, false, kEpiStore, false, false>;
using CfgStoreKP = Cfg<256, false, false, false, kEpiStore, false, false, true>;
// short reductions: sixteen epilogue warps (and 32-column chunks for one output)
using CfgG1P16 = Cfg<128, false, false, true, kEpiSwigluFwd, false, false, true, false, 16, 16>;
using CfgStoreKP32 = Cfg<256, false, false, false, kEpiStore, false, false, true, false, 32, 16>;
template <int BN> using CfgSwigluBwd = Cfg<BN, false, true, false, kEpiSwigluBwd, false, false>;
using CfgSwigluBwdP = Cfg<256, false, true, false, kEpiSwigluBwd, false, false, true>;
using CfgSwigluBwdP16 = Cfg<256, false, true, false, kEpiSwigluBwd, false, false, true, false, 16, 16>;
template <int BN> using CfgDgrad2 = Cfg<BN, false, true, false, kEpiStore, true, false>;
using CfgDgrad2P = Cfg<256, false, true, false, kEpiStore, true, false, true>;
// Reductions this short (K elements) finish their main loop well before eight epilogue warps
// have stored the tile, so those GEMMs take sixteen: G1 (three outputs) up to K = 1024, G2
// (one output, 32-column chunks) up to K = 512. Measured on one box, the small fine-grained
// layer's forward went from 0.156 to 0.137 ms; at K = 768-1024 sixteen warps for G2 (which
// cost an operand stage) were 3% slower, and B4 at K = 512 gained nothing.
constexpr int kShortK = 1024;
constexpr int kShortKOneOut = 512;
constexpr int kShortKB2 = 1024;
template <int BN> using CfgWgrad = Cfg<BN, true, true, false, kEpiStore, false, true>;
using CfgWgradP = Cfg<256, true, true, false, kEpiStore, false, true, true>;
// E4M3 forward GEMMs (rowwise scales)
using CfgG1P8 = Cfg<128, false, false, true, kEpiSwigluFwd, false, false, true, true>;
using CfgStoreKP8 = Cfg<256, false, false, false, kEpiStore, false, false, true, true>;
using CfgStoreK8 = Cfg<128, false, false, false, kEpiStore, false, false, false, true>;
// E4M3 data gradients (B2 on the upstream gradient's codes and W_d's transposed column codes)
using CfgSwigluBwdP8 = Cfg<256, false, false, false, kEpiSwigluBwd, false, false, true, true>;
using CfgSwigluBwd8 = Cfg<128, false, false, false, kEpiSwigluBwd, false, false, false, true>;

Params base_params(const int64_t* row_offsets, int64_t rows, int E) {
    Params P{};
    P.row_offsets = row_offsets;
    P.rows = rows;
    P.E = E;
    P.status = device_status_word();
    P.wait_limit_ns = wait_limit_ns();
    return P;
}

int64_t token_tiles_max(int64_t rows, int N, int BN) { return cdiv(rows, BM) * (N / BN); }

bool gemm_shape_ok(int d, int f) { return d % 128 == 0 && f % 128 == 0 && d > 0 && f > 0; }

}  // namespace

bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                       uint32_t box_inner, uint32_t box_outer) {
    return make_map(m, base, inner, outer, box_inner, box_outer);
}

bool make_tmap_f32_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_inner, uint32_t box_outer) {
    auto enc = get_encoder();
    if (!enc || !base) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_expert_fwd(const moe_bf16* X, const int64_t* row_offsets, int E, int64_t rows,
                              int d, int f, const moe_bf16* W_g, const moe_bf16* W_u,
                              const moe_bf16* W_d, moe_bf16* A, moe_bf16* U, moe_bf16* H,
                              moe_bf16* Y, const float* row_gate, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (!X || !W_g || !W_u || !W_d || !A || !U || !H || !Y) return MOE_ERR_INVALID_ARG;
    if (E <= 0 || rows <= 0 || (!row_offsets && E != 1)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || !gemm_shape_ok(d, f)) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[8] = {X, W_g, W_u, W_d, A, U, H, Y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    if (!device_status_word()) return MOE_ERR_LAUNCH;
    cudaStream_t st = (cudaStream_t)stream;
    CUtensorMap mx, mwg, mwu, mh, mwd;
    if (!make_map(&mx, X, d, rows, 64, 128) || !make_map(&mwg, W_g, d, (uint64_t)E * f, 64, 128) ||
        !make_map(&mwu, W_u, d, (uint64_t)E * f, 64, 128) || !make_map(&mh, H, f, rows, 64, 128))
        return MOE_ERR_LAUNCH;
    // G1: a, u, h
    Params P = base_params(row_offsets, rows, E);
    P.N = f;
    P.K0 = d;
    P.row_scale = row_gate;
    CUtensorMap moa[3], moy[3];
    if (!out_maps(moa, A, U, H, f, rows) || !out_maps(moy, Y, nullptr, nullptr, d, rows))
        return MOE_ERR_LAUNCH;
    int rc = d <= kShortK
                 ? launch<CfgG1P16>(mx, mx, mwg, mwu, P, token_tiles_max(rows, f, 128), st, moa)
                 : launch<CfgG1P>(mx, mx, mwg, mwu, P, token_tiles_max(rows, f, 128), st, moa);
    if (rc != MOE_OK) return rc;
    // G2: y = h W_d^T
    Params Q = base_params(row_offsets, rows, E);
    Q.N = d;
    Q.K0 = f;
    if (d % 256 == 0) {  // CTA pair: each CTA stages 128 of the tile's 256 W_d rows
        if (!make_map(&mwd, W_d, f, (uint64_t)E * d, 64, 128)) return MOE_ERR_LAUNCH;
        if (f <= kShortKOneOut) {
            CUtensorMap moy32[3];
            if (!out_maps(moy32, Y, nullptr, nullptr, d, rows, 32)) return MOE_ERR_LAUNCH;
            rc = launch<CfgStoreKP32>(mh, mh, mwd, mwd, Q, token_tiles_max(rows, d, 256), st, moy32);
        } else {
            rc = launch<CfgStoreKP>(mh, mh, mwd, mwd, Q, token_tiles_max(rows, d, 256), st, moy);
        }
    } else {
        if (!make_map(&mwd, W_d, f, (uint64_t)E * d, 64, 128)) return MOE_ERR_LAUNCH;
        rc = launch<CfgStoreK<128>>(mh, mh, mwd, mwd, Q, token_tiles_max(rows, d, 128), st, moy);
    }
    return rc;
}

static int weight_grads(const moe_bf16* dY, const moe_bf16* X, const moe_bf16* H,
                        const moe_bf16* dA, const moe_bf16* dU, const int64_t* row_offsets, int E,
                        int64_t rows, int d, int f, int32_t* order, moe_bf16* dW_g, moe_bf16* dW_u,
                        moe_bf16* dW_d, cudaStream_t st);

extern "C" int moe_expert_bwd(const moe_bf16* dY, const moe_bf16* X, const moe_bf16* A,
                              const moe_bf16* U, const moe_bf16* H, const int64_t* row_offsets,
                              int E, int64_t rows, int d, int f, const moe_bf16* W_g,
                              const moe_bf16* W_u, const moe_bf16* W_d, moe_bf16* dX,
                              moe_bf16* dA, moe_bf16* dU, moe_bf16* dW_g, moe_bf16* dW_u,
                              moe_bf16* dW_d, const float* row_gate, float* gate_part, int parts,
                              const float* dl_rows, const float* W_r, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
    if (!dY || !X || !A || !U || !H || !W_g || !W_u || !W_d || !dX || !dA || !dU || !dW_g ||
        !dW_u || !dW_d)
        return MOE_ERR_INVALID_ARG;
    if ((row_gate == nullptr) != (gate_part == nullptr)) return MOE_ERR_INVALID_ARG;
    if (parts <= 0 || parts > MOE_BWD_ALL) return MOE_ERR_INVALID_ARG;
    if ((dl_rows == nullptr) != (W_r == nullptr)) return MOE_ERR_INVALID_ARG;
    if (W_r && (!row_offsets || !aligned16(W_r))) return MOE_ERR_INVALID_ARG;
    if (E <= 0 || rows <= 0 || (!row_offsets && E != 1)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || !gemm_shape_ok(d, f)) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[14] = {dY, X, A, U, H, W_g, W_u, W_d, dX, dA, dU, dW_g, dW_u, dW_d};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    if (!device_status_word()) return MOE_ERR_LAUNCH;
    WsCarver wc(ws, ws_bytes);
    int32_t* order = wc.take<int32_t>(E + 1);
    if (row_offsets && (!ws || !wc.ok())) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    int rc;

    // B2: dH = dY W_d (W_d[e] is [d, f]: K = d rows, N = f contiguous), SwiGLU backward; the
    // saved a and u are staged by TMA (their maps ride in the second A and B slots)
    if (parts & MOE_BWD_DH) {
        constexpr CUtensorMapSwizzle kAuSwz = kAuCols == 32   ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : kAuCols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                              : CU_TENSOR_MAP_SWIZZLE_NONE;
        CUtensorMap mdy, mwd, msa, msu;
        if (!make_map(&mdy, dY, d, rows, 64, 128) || !make_map(&mwd, W_d, f, (uint64_t)E * d, 64, 64) ||
            !make_map(&msa, A, f, rows, kAuCols, 32, false, kAuSwz) ||
            !make_map(&msu, U, f, rows, kAuCols, 32, false, kAuSwz))
            return MOE_ERR_LAUNCH;
        Params P = base_params(row_offsets, rows, E);
        P.N = f;
        P.K0 = d;
        P.kb_per_expert = d;
        P.ld_out = f;
        P.row_scale = row_gate;
        P.gate_part = gate_part;
        CUtensorMap mod[3];
        if (!out_maps(mod, dA, dU, nullptr, f, rows)) return MOE_ERR_LAUNCH;
        if (f % 256 == 0 && d <= kShortKB2)
            rc = launch<CfgSwigluBwdP16>(mdy, msa, mwd, msu, P, token_tiles_max(rows, f, 256), st, mod);
        else if (f % 256 == 0)
            rc = launch<CfgSwigluBwdP>(mdy, msa, mwd, msu, P, token_tiles_max(rows, f, 256), st, mod);
        else
            rc = launch<CfgSwigluBwd<128>>(mdy, msa, mwd, msu, P, token_tiles_max(rows, f, 128), st,
                                           mod);
        if (rc != MOE_OK) return rc;
    }
    // B4: dX = dA W_g + dU W_u (W_g[e] is [f, d]: K = f rows, N = d contiguous), plus each
    // row's router term when given
    if (parts & MOE_BWD_DX) {
        CUtensorMap mda, mdu, mwg, mwu;
        if (!make_map(&mda, dA, f, rows, 64, 128) || !make_map(&mdu, dU, f, rows, 64, 128) ||
            !make_map(&mwg, W_g, d, (uint64_t)E * f, 64, 64) ||
            !make_map(&mwu, W_u, d, (uint64_t)E * f, 64, 64))
            return MOE_ERR_LAUNCH;
        Params P = base_params(row_offsets, rows, E);
        P.N = d;
        P.K0 = f;
        P.K1 = f;
        P.kb_per_expert = f;
        P.r1_row = dl_rows;
        P.r1_col = W_r;
        CUtensorMap mox[3];
        if (!out_maps(mox, dX, nullptr, nullptr, d, rows)) return MOE_ERR_LAUNCH;
        if (d % 256 == 0)
            rc = launch<CfgDgrad2P>(mda, mdu, mwg, mwu, P, token_tiles_max(rows, d, 256), st, mox);
        else
            rc = launch<CfgDgrad2<128>>(mda, mdu, mwg, mwu, P, token_tiles_max(rows, d, 128), st, mox);
        if (rc != MOE_OK) return rc;
    }
    if (!(parts & MOE_BWD_W)) return MOE_OK;
    return weight_grads(dY, X, H, dA, dU, row_offsets, E, rows, d, f, order, dW_g, dW_u, dW_d, st);
}

// B3 and B5, the weight gradients, from bf16 operands (shared by both expert backward
// entry points): experts scheduled longest first.
static int weight_grads(const moe_bf16* dY, const moe_bf16* X, const moe_bf16* H,
                        const moe_bf16* dA, const moe_bf16* dU, const int64_t* row_offsets, int E,
                        int64_t rows, int d, int f, int32_t* order, moe_bf16* dW_g, moe_bf16* dW_u,
                        moe_bf16* dW_d, cudaStream_t st) {
    int rc;
    if (row_offsets) {
        expert_order_kernel<<<1, kMaxExperts, 0, st>>>(row_offsets, E, order);
        if (launch_status() != MOE_OK) return MOE_ERR_LAUNCH;
    }
    const int32_t* order_ptr = row_offsets ? order : nullptr;
    // B3: dW_d[e] = dY_e^T H_e  (M = d, N = f, K = the expert's rows)
    {
        CUtensorMap mdy, mh;
        if (!make_map(&mdy, dY, d, rows, 64, 64) || !make_map(&mh, H, f, rows, 64, 64))
            return MOE_ERR_LAUNCH;
        Params P = base_params(row_offsets, rows, E);
        P.expert_order = order_ptr;
        P.N = f;
        P.M_out = d;
        P.nprob = 1;
        P.out0 = reinterpret_cast<__nv_bfloat16*>(dW_d);
        const int64_t pair_tiles = (int64_t)E * (d / 256) * (f / 256);
        if (d % 256 == 0 && f % 256 == 0 && 2 * pair_tiles >= sm_count())
            rc = launch<CfgWgradP>(mdy, mdy, mh, mh, P, pair_tiles, st);
        else if (f % 256 == 0 && !(d % 256 == 0 && 2 * pair_tiles < sm_count()))
            rc = launch<CfgWgrad<256>>(mdy, mdy, mh, mh, P, (int64_t)E * (d / BM) * (f / 256), st);
        else  // also when there are few pair tiles: 128-wide tiles on 4x the SMs
            rc = launch<CfgWgrad<128>>(mdy, mdy, mh, mh, P, (int64_t)E * (d / BM) * (f / 128), st);
        if (rc != MOE_OK) return rc;
    }
    // B5: dW_g[e] = dA_e^T X_e, dW_u[e] = dU_e^T X_e  (M = f, N = d)
    {
        CUtensorMap mda, mdu, mxx;
        if (!make_map(&mda, dA, f, rows, 64, 64) || !make_map(&mdu, dU, f, rows, 64, 64) ||
            !make_map(&mxx, X, d, rows, 64, 64))
            return MOE_ERR_LAUNCH;
        Params P = base_params(row_offsets, rows, E);
        P.expert_order = order_ptr;
        P.N = d;
        P.M_out = f;
        P.nprob = 2;
        P.out0 = reinterpret_cast<__nv_bfloat16*>(dW_g);
        P.out1 = reinterpret_cast<__nv_bfloat16*>(dW_u);
        const int64_t pair_tiles = (int64_t)E * 2 * (f / 256) * (d / 256);
        if (d % 256 == 0 && f % 256 == 0 && 2 * pair_tiles >= sm_count())
            rc = launch<CfgWgradP>(mda, mdu, mxx, mxx, P, pair_tiles, st);
        else if (d % 256 == 0 && f % 256 == 0)  // few pair tiles: 128-wide tiles on 4x the SMs
            rc = launch<CfgWgrad<128>>(mda, mdu, mxx, mxx, P, (int64_t)E * 2 * (f / BM) * (d / 128), st);
        else if (d % 256 == 0)
            rc = launch<CfgWgrad<256>>(mda, mdu, mxx, mxx, P, (int64_t)E * 2 * (f / BM) * (d / 256), st);
        else
            rc = launch<CfgWgrad<128>>(mda, mdu, mxx, mxx, P, (int64_t)E * 2 * (f / BM) * (d / 128), st);
    }
    return rc;
}

extern "C" int moe_expert_bwd_fp8(const uint8_t* dYq, const float* sdY, const moe_bf16* dY,
                                  const moe_bf16* X, const moe_bf16* A, const moe_bf16* U,
                                  const moe_bf16* H, const int64_t* row_offsets, int E,
                                  int64_t rows, int d, int f, const uint8_t* Wdq, const float* sWd,
                                  const uint8_t* Wguq, const float* sWgu, moe_bf16* dX,
                                  moe_bf16* dA, moe_bf16* dU, uint8_t* AUq, float* sAU,
                                  moe_bf16* dW_g, moe_bf16* dW_u, moe_bf16* dW_d,
                                  const float* dl_rows, const float* W_r, void* ws,
                                  size_t ws_bytes, moe_stream_t stream) {
    if (!dYq || !sdY || !dY || !X || !A || !U || !H || !Wdq || !sWd || !Wguq || !sWgu || !dX ||
        !dA || !dU || !AUq || !sAU || !dW_g || !dW_u || !dW_d)
        return MOE_ERR_INVALID_ARG;
    if ((dl_rows == nullptr) != (W_r == nullptr)) return MOE_ERR_INVALID_ARG;
    if (W_r && (!row_offsets || !aligned16(W_r))) return MOE_ERR_INVALID_ARG;
    if (E <= 0 || rows <= 0 || (!row_offsets && E != 1)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || !gemm_shape_ok(d, f)) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[14] = {dYq, dY, X, A, U, H, Wdq, Wguq, dX, dA, dU, AUq, dW_g, dW_u};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dW_d) || !aligned16(sWd) || !aligned16(sWgu)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    if (!device_status_word()) return MOE_ERR_LAUNCH;
    WsCarver wc(ws, ws_bytes);
    int32_t* order = wc.take<int32_t>(E + 1);
    if (row_offsets && (!ws || !wc.ok())) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    int rc;
    // B2 on E4M3: r = (dy codes)(W_d column codes, transposed: [E f, d], K-major) times the
    // row and column scales, then the SwiGLU backward on the staged bf16 a and u
    {
        constexpr CUtensorMapSwizzle kAuSwz = kAuCols == 32   ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : kAuCols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                              : CU_TENSOR_MAP_SWIZZLE_NONE;
        CUtensorMap mdy, mwd, msa, msu;
        if (!make_map(&mdy, dYq, d, rows, 128, 128, true) ||
            !make_map(&mwd, Wdq, d, (uint64_t)E * f, 128, 128, true) ||
            !make_map(&msa, A, f, rows, kAuCols, 32, false, kAuSwz) ||
            !make_map(&msu, U, f, rows, kAuCols, 32, false, kAuSwz))
            return MOE_ERR_LAUNCH;
        Params P = base_params(row_offsets, rows, E);
        P.N = f;
        P.K0 = d;
        P.ld_out = f;
        P.sa = sdY;
        P.sb0 = sWd;
        CUtensorMap mod[3];
        if (!out_maps(mod, dA, dU, nullptr, f, rows)) return MOE_ERR_LAUNCH;
        if (f % 256 == 0)
            rc = launch<CfgSwigluBwdP8>(mdy, msa, mwd, msu, P, token_tiles_max(rows, f, 256), st, mod);
        else
            rc = launch<CfgSwigluBwd8>(mdy, msa, mwd, msu, P, token_tiles_max(rows, f, 128), st, mod);
        if (rc != MOE_OK) return rc;
    }
    // [dA | dU] rows -> E4M3 codes under one scale per row (2 f bytes per row)
    rc = launch_quantize_rows_fp8(reinterpret_cast<const __nv_bfloat16*>(dA),
                                  row_offsets ? row_offsets + E : nullptr, rows, f, AUq, sAU, st,
                                  reinterpret_cast<const __nv_bfloat16*>(dU));
    if (rc != MOE_OK) return rc;
    // B4 on E4M3: dX = [dA | dU] codes ([rows, 2f]) x ([W_g; W_u] column codes, transposed:
    // [E d, 2f], K-major), one product over K = 2f, times the row and column scales
    {
        CUtensorMap mau, mwgu;
        if (!make_map(&mau, AUq, 2 * (uint64_t)f, rows, 128, 128, true) ||
            !make_map(&mwgu, Wguq, 2 * (uint64_t)f, (uint64_t)E * d, 128, 128, true))
            return MOE_ERR_LAUNCH;
        Params P = base_params(row_offsets, rows, E);
        P.N = d;
        P.K0 = 2 * f;
        P.sa = sAU;
        P.sb0 = sWgu;
        P.r1_row = dl_rows;
        P.r1_col = W_r;
        CUtensorMap mox[3];
        if (!out_maps(mox, dX, nullptr, nullptr, d, rows)) return MOE_ERR_LAUNCH;
        if (d % 256 == 0)
            rc = launch<CfgStoreKP8>(mau, mau, mwgu, mwgu, P, token_tiles_max(rows, d, 256), st, mox);
        else
            rc = launch<CfgStoreK8>(mau, mau, mwgu, mwgu, P, token_tiles_max(rows, d, 128), st, mox);
        if (rc != MOE_OK) return rc;
    }
    return weight_grads(dY, X, H, dA, dU, row_offsets, E, rows, d, f, order, dW_g, dW_u, dW_d, st);
}

extern "C" int moe_expert_fwd_fp8(const uint8_t* Xq, const float* sX, const int64_t* row_offsets,
                                  int E, int64_t rows, int d, int f, const uint8_t* Wgq,
                                  const float* sWg, const uint8_t* Wuq, const float* sWu,
                                  const uint8_t* Wdq, const float* sWd, moe_bf16* A, moe_bf16* U,
                                  moe_bf16* H, uint8_t* Hq, float* sH, moe_bf16* Y,
                                  const float* row_gate, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (!Xq || !sX || !Wgq || !sWg || !Wuq || !sWu || !Wdq || !sWd || !A || !U || !H || !Hq ||
        !sH || !Y)
        return MOE_ERR_INVALID_ARG;
    if (E <= 0 || rows <= 0 || (!row_offsets && E != 1)) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || !gemm_shape_ok(d, f)) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[9] = {Xq, Wgq, Wuq, Wdq, A, U, H, Hq, Y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!device_supported()) return MOE_ERR_UNSUPPORTED;
    if (!device_status_word()) return MOE_ERR_LAUNCH;
    cudaStream_t st = (cudaStream_t)stream;
    CUtensorMap mx, mwg, mwu, mh, mwd;
    if (!make_map(&mx, Xq, d, rows, 128, 128, true) ||
        !make_map(&mwg, Wgq, d, (uint64_t)E * f, 128, 128, true) ||
        !make_map(&mwu, Wuq, d, (uint64_t)E * f, 128, 128, true) ||
        !make_map(&mh, Hq, f, rows, 128, 128, true) ||
        !make_map(&mwd, Wdq, f, (uint64_t)E * d, 128, 128, true))
        return MOE_ERR_LAUNCH;
    // G1 on E4M3 codes: a, u, h
    Params P = base_params(row_offsets, rows, E);
    P.N = f;
    P.K0 = d;
    P.sa = sX;
    P.sb0 = sWg;
    P.sb1 = sWu;
    P.row_scale = row_gate;
    CUtensorMap moa[3], moy[3];
    if (!out_maps(moa, A, U, H, f, rows) || !out_maps(moy, Y, nullptr, nullptr, d, rows))
        return MOE_ERR_LAUNCH;
    int rc = launch<CfgG1P8>(mx, mx, mwg, mwu, P, token_tiles_max(rows, f, 128), st, moa);
    if (rc != MOE_OK) return rc;
    // h rows -> E4M3 codes for the down projection
    rc = launch_quantize_rows_fp8(reinterpret_cast<const __nv_bfloat16*>(H),
                                  row_offsets ? row_offsets + E : nullptr, rows, f, Hq, sH, st);
    if (rc != MOE_OK) return rc;
    // G2 on E4M3 codes: y
    Params Q = base_params(row_offsets, rows, E);
    Q.N = d;
    Q.K0 = f;
    Q.sa = sH;
    Q.sb0 = sWd;
    if (d % 256 == 0)
        rc = launch<CfgStoreKP8>(mh, mh, mwd, mwd, Q, token_tiles_max(rows, d, 256), st, moy);
    else
        rc = launch<CfgStoreK8>(mh, mh, mwd, mwd, Q, token_tiles_max(rows, d, 128), st, moy);
    return rc;
}
