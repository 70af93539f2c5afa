// Host-side launch geometry and scratch sizes shared by the entry points.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kRouteTokensPerCta = 64;     // router forward: tokens per CTA
constexpr int kHistTokensPerCta = 1024;    // permute: tokens per histogram chunk
constexpr int kRouteBwdTokensPerSplit = 2048;  // router backward: tokens per dW_r split
constexpr int kMaxExperts = 256;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int64_t route_blocks(int64_t T) { return cdiv(T, kRouteTokensPerCta); }
inline int64_t hist_blocks(int64_t T) { return cdiv(T, kHistTokensPerCta); }
inline int64_t route_bwd_splits(int64_t T) { return cdiv(T, kRouteBwdTokensPerSplit); }

inline size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Scratch of each entry point (each region rounded to 256 bytes as WsCarver takes them).
inline size_t ws_route(int64_t T) { return round256(sizeof(double) * route_blocks(T)); }
inline size_t ws_permute(int64_t T, int E) {
    return 2 * round256(sizeof(int32_t) * hist_blocks(T) * E);
}
inline size_t ws_route_bwd(int64_t T, int d, int E) {
    return round256(sizeof(float) * route_bwd_splits(T) * (size_t)E * d);
}
inline size_t ws_expert(int E) { return round256(sizeof(int32_t) * (E + 1)) * 2; }
// Balancing losses: partial sums per (sequence, 256-token chunk); there are at most T such
// chunks (one-token sequences), each holding E floats and E counts.
inline size_t ws_aux(int64_t T, int E) {
    return 2 * round256(sizeof(float) * (size_t)T * E);
}

inline size_t ws_total(int64_t T, int d, int E, int k) {
    (void)k;
    size_t m = ws_route(T);
    if (ws_permute(T, E) > m) m = ws_permute(T, E);
    if (ws_route_bwd(T, d, E) > m) m = ws_route_bwd(T, d, E);
    if (ws_expert(E) > m) m = ws_expert(E);
    if (ws_aux(T, E) > m) m = ws_aux(T, E);
    return m + 256;
}

}  // namespace moe
