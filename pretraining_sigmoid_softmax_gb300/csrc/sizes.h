// Host-side launch geometry and scratch sizes shared by the entry points.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kRouteTokensPerCta = 64;     // router forward: tokens per CTA
constexpr int kHistTokensPerCta = 256;     // permute: tokens per histogram chunk
constexpr int kRouteBwdTokensPerSplit = 2048;  // router backward: tokens per dW_r split
constexpr int kMaxExperts = 256;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int64_t route_blocks(int64_t T) { return cdiv(T, kRouteTokensPerCta); }
inline int64_t hist_blocks(int64_t T) { return cdiv(T, kHistTokensPerCta); }
inline int64_t route_bwd_splits(int64_t T) { return cdiv(T, kRouteBwdTokensPerSplit); }

inline size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Router on the tensor cores (E <= 128). Logits: tiles of 128 tokens, the expert axis padded
// to epad columns. W_r gradient: tiles of 128 columns of d by np experts, the token axis split
// in at most route_tc_splits_max pieces. 0 = too wide: the SIMT kernels run instead.
inline int route_tc_epad(int E) { return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 0; }
inline int route_tc_np(int E) { return E <= 64 ? 64 : E <= 128 ? 128 : 0; }
inline int64_t route_tc_tiles(int64_t T) { return cdiv(T, 128); }
inline int64_t route_tc_splits_max(int64_t T) {
    const int64_t kb = cdiv(T, 64);
    return kb < 32 ? kb : 32;
}

// Scratch of each entry point (each region rounded to 256 bytes as WsCarver takes them).
// Router forward: z-loss partial sums (per 64-token block, or per 32-token warp of a
// tensor-core tile) and the three bf16 pieces of W_r.
inline size_t ws_route(int64_t T, int d, int E) {
    int64_t nz = route_blocks(T);
    if (4 * route_tc_tiles(T) > nz) nz = 4 * route_tc_tiles(T);
    const size_t w = route_tc_epad(E) ? (size_t)3 * route_tc_epad(E) * d * 2 : 0;
    return round256(sizeof(double) * nz) + round256(w);
}
inline size_t ws_permute(int64_t T, int E) {
    return 2 * round256(sizeof(int32_t) * hist_blocks(T) * E);
}
// Router backward: W_r-gradient partial sums per token split, and (tensor-core path) the
// three bf16 pieces of the logit gradient, each [T, np].
inline size_t ws_route_bwd(int64_t T, int d, int E) {
    int64_t s = route_bwd_splits(T);
    if (route_tc_np(E) && route_tc_splits_max(T) > s) s = route_tc_splits_max(T);
    const size_t part = round256(sizeof(float) * s * (size_t)E * d);
    // 3 pieces of T * np bf16, each padded to a multiple of 128 elements (256 bytes)
    const size_t pieces = route_tc_np(E) ? round256((size_t)3 * 2 * (((size_t)T * route_tc_np(E) + 127) / 128 * 128)) : 0;
    return part + pieces;
}
inline size_t ws_expert(int E) { return round256(sizeof(int32_t) * (E + 1)) * 2; }
// Balancing losses: partial sums per (sequence, 256-token chunk); there are at most T such
// chunks (one-token sequences), each holding E floats and E counts.
inline size_t ws_aux(int64_t T, int E) {
    return 2 * round256(sizeof(float) * (size_t)T * E);
}

// Router input gradient (tensor cores): two bf16 pieces of the logit gradient and three of W_r.
inline size_t ws_router_dx(int64_t T, int d, int E) {
    const int np = route_tc_np(E);
    if (!np) return 0;
    const size_t pstride = ((size_t)T * np + 127) / 128 * 128;
    return round256(2 * 2 * pstride) + round256((size_t)3 * np * d * 2);
}

inline size_t ws_total(int64_t T, int d, int E, int k) {
    (void)k;
    size_t m = ws_route(T, d, E);
    if (ws_permute(T, E) > m) m = ws_permute(T, E);
    if (ws_route_bwd(T, d, E) > m) m = ws_route_bwd(T, d, E);
    if (ws_expert(E) > m) m = ws_expert(E);
    if (ws_aux(T, E) > m) m = ws_aux(T, E);
    if (ws_router_dx(T, d, E) > m) m = ws_router_dx(T, d, E);
    return m + 256;
}

}  // namespace moe
