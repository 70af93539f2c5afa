/*
 * moe_gb300.h - C ABI of the GB300 (sm_103a) fine-grained Mixture-of-Experts layer.
 *
 * The layer (forward and backward of one decoder MoE layer on one GPU):
 *   route    : router logits l = x W_r^T in fp32, top-k expert choice, gates;
 *   permute  : every token copied to the rows of its k experts, grouped by expert;
 *   experts  : SwiGLU experts h = silu(x W_g^T) * (x W_u^T), y = h W_d^T as grouped GEMMs;
 *   combine  : out_t = sum_i g_ti y_ti (+ shared expert output);
 *   bias     : aux-loss-free per-expert bias update after backward.
 * Sources: "The whole stack, in the open" (Apex-3), "What's inside", row "Fine-grained MoE"
 * (sigmoid router, per-expert bias balancing the load without a loss term, grouped GEMM
 * experts); KempnerForge README, "Features" (softmax top-k and DeepSeek-V3 sigmoid routers,
 * shared experts, router z-loss); "How to train a large-scale Mixture-of-Experts model from
 * scratch", section 2.5 "First training of MoE" (top-8 of 64 experts, tokens sent to the
 * chosen experts and outputs returned, bias-free SwiGLU experts, fp32 router logits).
 *
 * Conventions for every entry point
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise; the library
 *     never allocates or frees memory. Scratch space is the caller's `ws` buffer of at
 *     least moe_workspace_bytes() bytes (256-byte aligned).
 *   - Row-major layouts. bf16 tensors are passed as `moe_bf16*` (IEEE bfloat16 bits).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream);
 *     no call synchronises. The return value reports host-side argument checks and
 *     launch errors only. Problems found on the device (an expert index out of range,
 *     a bounded wait that ran out) are recorded in a per-device status word read with
 *     moe_device_status().
 *   - Results are deterministic: no floating-point atomics, every reduction has a fixed
 *     order, so two runs on the same inputs give identical bits.
 *   - Shape limits: 1 <= k <= min(E, 32), E <= 256, d % 128 == 0, f % 128 == 0,
 *     T >= 1. Violations return MOE_ERR_UNSUPPORTED; null or inconsistent arguments
 *     MOE_ERR_INVALID_ARG.
 *
 * Permuted ("expert-major") layout
 *   Rows routed to expert e are stored contiguously, in ascending token order, starting
 *   at row_offsets[e]. Each expert's segment is padded with zero rows to a multiple of
 *   MOE_ROW_ALIGN (128) rows so that every 128-row tile of the grouped GEMMs belongs to
 *   a single expert. row_offsets[e+1] - row_offsets[e] = round_up(counts[e], 128).
 *   Buffers in this layout have moe_padded_rows(T, k, E) rows of capacity; rows past
 *   row_offsets[E] are never read or written.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;               /* IEEE bfloat16 bit pattern */
typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t */

#define MOE_ROW_ALIGN 128

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,  /* shape outside the limits above, or not an sm_103 device */
    MOE_ERR_WORKSPACE = 3,    /* ws_bytes smaller than moe_workspace_bytes() */
    MOE_ERR_LAUNCH = 4,       /* a CUDA launch or runtime call failed */
    MOE_ERR_BAD_INDEX = 5,    /* device: an expert index outside [0, E) or a layout overflow */
    MOE_ERR_TIMEOUT = 6,      /* device: a bounded wait inside a kernel ran out */
    MOE_ERR_TOO_LARGE = 7     /* sizes exceed a fixed, library-owned scratch array */
};

enum moe_router_mode {
    MOE_MODE_SIGMOID = 0, /* sigmoid scores, top-k of score + bias, gates renormalised */
    MOE_MODE_SOFTMAX = 1  /* softmax over all experts, top-k of logits, gates not renormalised */
};

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int moe_version(void);

/* Row capacity of a buffer in the permuted layout: round_up(T*k + E*127, 128). */
int64_t moe_padded_rows(int64_t T, int k, int E);

/* Bytes of scratch any one entry point needs for these sizes (the maximum over all). */
size_t moe_workspace_bytes(int64_t T, int d, int E, int k);

/*
 * Device status word of the current device, written by kernels that detect a problem.
 * Synchronises `stream`, stores the first recorded code (MOE_OK if none) in *code and
 * the site that recorded it in *site (may be NULL). Returns MOE_OK or MOE_ERR_LAUNCH.
 */
int moe_device_status(moe_stream_t stream, int* code, int* site);
/* Clears the device status word (enqueued on `stream`). */
int moe_clear_device_status(moe_stream_t stream);

/*
 * Upper limit, in nanoseconds, of every bounded wait inside the grouped-GEMM kernels
 * (default 2e9). A wait that runs out records MOE_ERR_TIMEOUT and the kernel returns
 * after releasing its tensor memory.
 */
void moe_set_wait_limit_ns(uint64_t ns);

/*
 * moe_check_bounded_wait - self-check of the failure path of the bounded device waits (no
 * counterpart on the pages, which name failure detection only as monitoring: DCGM, NaN
 * detection). Enqueues one kernel that waits, with the same bounded wait the grouped-GEMM
 * kernels use, on an mbarrier that nothing arrives on, with no copy or tensor-core work in
 * flight. The wait runs out after limit_ns nanoseconds (0 < limit_ns <= 1e9, else
 * MOE_ERR_INVALID_ARG), records MOE_ERR_TIMEOUT with site 90 in the device status word and
 * the kernel returns; the context stays usable. Clear the word with moe_clear_device_status
 * afterwards.
 */
int moe_check_bounded_wait(uint64_t limit_ns, moe_stream_t stream);

/*
 * moe_route - router forward (R1).
 * Definition: l[t,e] = sum_j x[t,j] * W_r[e,j] in fp32, each sum in a fixed order.
 *   MOE_MODE_SIGMOID: s = 1/(1+exp(-l)); choose the k largest s[e] + b[e] (lower e first
 *     on equal values); topk_score = chosen s; topk_gate = chosen s / sum of chosen s.
 *   MOE_MODE_SOFTMAX: p = softmax(l) over all E; choose the k largest l (lower e first);
 *     topk_gate = topk_score = chosen p (no renormalisation); lse[t] = logsumexp(l[t]);
 *     z_loss[0] = z_coef * mean_t(lse[t]^2).
 * Source: Apex-3 "Fine-grained MoE" row (sigmoid router with selection bias, no loss
 * term); KempnerForge "Features" (softmax top-k router, router z-loss); section 2.5 of
 * the handbook summary (router logits in fp32).
 * In : x [T,d] bf16; W_r [E,d] fp32; b [E] fp32 (sigmoid mode; ignored and may be NULL
 *      in softmax mode).
 * Out: logits [T,E] fp32 (may be NULL in sigmoid mode; required in softmax mode, where
 *      the backward needs it); topk_idx [T,k] int32, slots in descending selection value;
 *      topk_gate [T,k] fp32; topk_score [T,k] fp32; lse [T] fp32 and z_loss [1] fp32
 *      (softmax mode only, required there).
 */
int moe_route(const moe_bf16* x, const float* W_r, const float* b, int64_t T, int d, int E,
              int k, int mode, float z_coef, float* logits, int32_t* topk_idx,
              float* topk_gate, float* topk_score, float* lse, float* z_loss, void* ws,
              size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute - token dispatch (R2): counts, offsets and a stable expert-major copy of x.
 * Definition: counts[e] = number of (t,i) with topk_idx[t,i] == e; offsets = exclusive
 * scan of counts (offsets[E] = T*k); rows of expert e hold the tokens that chose e in
 * ascending token order. Source: section 2.5 of the handbook summary (tokens must be
 * sent to the chosen experts).
 * In : topk_idx [T,k] int32 (each row k distinct experts in [0,E)); x [T,d] bf16.
 * Out: counts [E] int32; offsets [E+1] int64 (unpadded); row_offsets [E+1] int64 (padded
 *      layout, multiples of 128); perm_token [moe_padded_rows] int32 (token of each row,
 *      -1 for padding rows); slot_to_row [T,k] int32 (row of slot (t,i));
 *      X_perm [moe_padded_rows, d] bf16 (x rows in the permuted layout, padding rows 0).
 * Optional (both or neither, else MOE_ERR_INVALID_ARG): topk_gate [T,k] fp32 in, row_gate
 *      [moe_padded_rows] fp32 out: the gate of each row's slot, 0 on padding rows (what
 *      moe_row_gates writes, for the gate folded into the experts), formed in the same pass.
 * An out-of-range index records MOE_ERR_BAD_INDEX; that slot is dropped.
 */
int moe_permute(const int32_t* topk_idx, const moe_bf16* x, int64_t T, int d, int E, int k,
                int32_t* counts, int64_t* offsets, int64_t* row_offsets, int32_t* perm_token,
                int32_t* slot_to_row, moe_bf16* X_perm, const float* topk_gate,
                float* row_gate, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute_noalloc - moe_permute for callers that cannot allocate device memory.
 * The source pages have no counterpart to this entry point; it exists for the library's
 * users. Some callers hold only the input and output buffers of the layer: a plug-in or
 * fixed-signature callback that is handed tensors but no allocator, or a process whose
 * device memory is owned entirely by another allocator. They cannot provide the `ws`
 * scratch that moe_permute needs and cannot call cudaMalloc to make one.
 * This variant takes the same arguments as moe_permute minus `topk_gate`/`row_gate` and
 * `ws`/`ws_bytes`, and gives the same results. Its scratch (two ceil(T/256) x E int32 tables of per-chunk expert
 * counts) lives in a static device array of MOE_PERMUTE_NOALLOC_MAX_INTS int32 per table
 * (8 MiB in total), which every GPU that loads the library holds until the process exits.
 *   - Limit: ceil(T / 256) * E <= MOE_PERMUTE_NOALLOC_MAX_INTS (T up to 4,194,304 tokens
 *     with E = 64, 1,048,576 with E = 256); larger sizes return MOE_ERR_TOO_LARGE before
 *     any device work.
 *   - Allocation: none. It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - Set-up: the first call on each device (made with that device current) looks up the
 *     device address of the static array once; make that first call before any stream
 *     capture on that device. The lookup is repeated only when the device's context has
 *     changed since (e.g. after cudaDeviceReset), which makes the next call a first call
 *     again.
 *   - Sharing: all calls on a device use the same array and it keeps the last call's
 *     contents (nothing in it needs to start at zero: every entry is written before it is
 *     read). Calls that overlap on the GPU (different streams, no ordering between them)
 *     race on the array and give wrong results; order them on one stream.
 */
#define MOE_PERMUTE_NOALLOC_MAX_INTS 1048576
int moe_permute_noalloc(const int32_t* topk_idx, const moe_bf16* x, int64_t T, int d, int E,
                        int k, int32_t* counts, int64_t* offsets, int64_t* row_offsets,
                        int32_t* perm_token, int32_t* slot_to_row, moe_bf16* X_perm,
                        moe_stream_t stream);

/*
 * moe_expert_fwd - SwiGLU experts as grouped GEMMs (G1 + G2), on tcgen05 tensor cores.
 * Definition, for each row p of expert e: a = X[p] W_g[e]^T, u = X[p] W_u[e]^T,
 * h = silu(a) * u, y = h W_d[e]^T; fp32 accumulation, bf16 results.
 * Source: Apex-3 "Fine-grained MoE" (experts run as grouped GEMMs); section 2.5 of the
 * handbook summary (bias-free SwiGLU expert, three weight matrices).
 * In : X [rows,d] bf16; row_offsets [E+1] int64 device array in the padded layout, or
 *      NULL for one dense expert over all `rows` rows (E must be 1; used for the shared
 *      expert with X = x, rows = T); W_g, W_u [E,f,d] bf16; W_d [E,d,f] bf16.
 * Out: A, U, H [rows,f] bf16 (saved for backward); Y [rows,d] bf16.
 * row_gate [rows] fp32 or NULL: with it the row's gate is folded into the expert, h is
 *      written as row_gate[p] * silu(a) * u (one bf16 rounding) and y is therefore the gated
 *      output; a and u are not scaled. The down projection is linear, so this gives the
 *      combine's g * y without a second pass (moe_permute or moe_row_gates builds row_gate).
 * `rows` is the row capacity of X/A/U/H/Y; rows past it are never touched.
 * A row_offsets array that breaks the padded layout (row_offsets[0] != 0, a decrease, a
 * segment that is not a multiple of 128 rows, row_offsets[E] > rows) records
 * MOE_ERR_BAD_INDEX (site 20) and the GEMMs write nothing; the same holds for
 * moe_expert_bwd and moe_expert_fwd_fp8.
 */
int moe_expert_fwd(const moe_bf16* X, const int64_t* row_offsets, int E, int64_t rows, int d,
                   int f, const moe_bf16* W_g, const moe_bf16* W_u, const moe_bf16* W_d,
                   moe_bf16* A, moe_bf16* U, moe_bf16* H, moe_bf16* Y, const float* row_gate,
                   void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_quantize_rows_fp8 - rowwise FP8 (E4M3) quantisation of a GEMM operand, the Apex-3
 * stack's "fp8_rowwise" precision ("The whole stack, in the open", "Run it yourself":
 * --precision fp8_rowwise; KempnerForge "Features": FP8 via E4M3). Reading: per row,
 * scale[r] = fp32(amax_r / 448) (1 for an all-zero row), Q[r,c] = E4M3(fp32(X[r,c] /
 * scale[r])), round to nearest even, saturating at +-448; both divisions IEEE fp32.
 * In : X [rows, cols] bf16; rows_limit: device int64 or NULL; only rows below
 *      min(rows, *rows_limit) are written (pass row_offsets + E for the padded layout).
 * Out: Q [rows, cols] E4M3 codes (bytes); scale [rows] fp32. cols % 128 == 0.
 */
int moe_quantize_rows_fp8(const moe_bf16* X, const int64_t* rows_limit, int64_t rows, int cols,
                          uint8_t* Q, float* scale, moe_stream_t stream);

/*
 * moe_permute_fp8 - the FP8 codes of the expert-major rows from the codes of the tokens.
 * The rowwise codes and scale of a row depend on that row alone, and every expert-major
 * row is a copy of its token's row x[t] (the dispatch of section 2.5 of the handbook
 * summary). So quantising the T token rows once and copying them to the rows gives exactly
 * moe_quantize_rows_fp8 of X_perm, bit for bit, with a k-fold smaller quantisation.
 * In : xq [T, d] codes and sx [T] scales (moe_quantize_rows_fp8 of x); slot_to_row [T,k],
 *      perm_token [rows] and row_offsets [E+1] from moe_permute (padding rows have
 *      perm_token < 0).
 * Out: Xq [rows, d] codes and sX [rows] scales, where rows = row_offsets[E]: the token's
 *      codes and scale on each of its k rows; padding rows get zero codes and scale 1 (the
 *      quantisation of a zero row). Slots with slot_to_row < 0 are skipped.
 * d % 128 == 0, k <= min(E, 32), E <= 256; xq and Xq 16-byte aligned.
 */
int moe_permute_fp8(const uint8_t* xq, const float* sx, const int32_t* slot_to_row,
                    const int32_t* perm_token, const int64_t* row_offsets, int64_t T, int d,
                    int E, int k, uint8_t* Xq, float* sX, moe_stream_t stream);

/*
 * moe_expert_fwd_fp8 - moe_expert_fwd with E4M3 GEMM operands (tcgen05 kind::f8f6f4, fp32
 * accumulation). Each product is dequantised in the epilogue by its A-row scale and its
 * B-row (output-channel) scale; a, u, h, y are bf16 as in moe_expert_fwd. h is quantised
 * per row (into Hq, sH) before the down projection.
 * In : Xq [rows, d] codes and sX [rows] (moe_quantize_rows_fp8 of the expert-major rows);
 *      Wgq, Wuq [E f, d] codes with sWg, sWu [E f]; Wdq [E d, f] codes with sWd [E d]
 *      (moe_quantize_rows_fp8 of the weights viewed as [E f, d] and [E d, f]).
 * Out: A, U, H [rows, f] bf16; Hq [rows, f] codes and sH [rows]; Y [rows, d] bf16.
 * row_gate: as in moe_expert_fwd (h, and so Hq and y, carry the row's gate).
 */
int moe_expert_fwd_fp8(const uint8_t* Xq, const float* sX, const int64_t* row_offsets, int E,
                       int64_t rows, int d, int f, const uint8_t* Wgq, const float* sWg,
                       const uint8_t* Wuq, const float* sWu, const uint8_t* Wdq,
                       const float* sWd, moe_bf16* A, moe_bf16* U, moe_bf16* H, uint8_t* Hq,
                       float* sH, moe_bf16* Y, const float* row_gate, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * moe_quantize_rows2_fp8 - moe_quantize_rows_fp8 of the concatenated rows [X0 | X1]: one
 * scale per row over both halves, codes 2 cols bytes per row (X0's in the first half).
 * Used for the expert input gradient's operand [dA | dU] of moe_expert_bwd_fp8, one product
 * over K = 2f whose row scale must cover both halves.
 * In : X0, X1 [rows, cols] bf16; rows_limit as in moe_quantize_rows_fp8.
 * Out: Q [rows, 2 cols] E4M3 codes; scale [rows] fp32. cols % 128 == 0.
 */
int moe_quantize_rows2_fp8(const moe_bf16* X0, const moe_bf16* X1, const int64_t* rows_limit,
                           int64_t rows, int cols, uint8_t* Q, float* scale, moe_stream_t stream);

/*
 * moe_quantize_cols_fp8 - columnwise FP8 (E4M3) quantisation of a weight operand whose
 * contraction runs over its rows, written transposed so the GEMM reads it K-major.
 * Reading (Apex-3 "fp8_rowwise" precision carried to the backward, as for
 * moe_expert_bwd_fp8): each column n of each of the E matrices gets scale = fp32(amax/448)
 * over its K values (1 for an all-zero column), codes E4M3(fp32(x / scale)) as in
 * moe_quantize_rows_fp8, so Qt[e][n][k] is the code of X[e][k][n].
 * In : X0 [E, K0, N] bf16; X1 [E, K0, N] bf16 or NULL: with X1 the matrices are the stacks
 *      [X0[e]; X1[e]] of K = 2 K0 rows under one scale per column.
 * Out: Qt [E, N, K] codes; scale [E N] fp32. K0 % 128 == 0, N % 64 == 0.
 * W_d [E, d, f] -> (X0 = W_d, K0 = d, N = f): Wdq [E, f, d]; W_g, W_u [E, f, d] ->
 * (X0 = W_g, X1 = W_u, K0 = f, N = d): Wguq [E, d, 2f].
 */
int moe_quantize_cols_fp8(const moe_bf16* X0, const moe_bf16* X1, int E, int K0, int N,
                          uint8_t* Qt, float* scale, moe_stream_t stream);

/*
 * moe_expert_bwd_fp8 - moe_expert_bwd with the two data-gradient GEMMs on E4M3 operands
 * (tcgen05 kind::f8f6f4, fp32 accumulation, scales applied in the epilogues); the weight
 * gradients stay bf16 GEMMs of the stored bf16 tensors.
 * Reading of the Apex-3 stack's fp8_rowwise precision ("The whole stack, in the open", "Run
 * it yourself") for the backward, whose form the pages do not give: each data-gradient
 * operand is scaled along the contraction axis, one scale per row of the left operand and
 * per column of the right one:
 *   r = dYq W_d: dy rows (moe_quantize_rows_fp8 of the expert-major upstream gradient) and
 *       W_d columns (Wdq, sWd: moe_quantize_cols_fp8 of W_d); then the SwiGLU backward on
 *       the stored bf16 a and u gives dA, dU (bf16);
 *   dX = [dA | dU] [W_g; W_u] as one product over K = 2f: the rows of [dA | dU]
 *       (moe_quantize_rows2_fp8, done here into AUq, sAU) and the columns of [W_g; W_u]
 *       (Wguq, sWgu: moe_quantize_cols_fp8 of W_g over W_u);
 *   dW_d = sum dY^T H, dW_g = sum dA^T X, dW_u = sum dU^T X as in moe_expert_bwd.
 * In : dYq [rows, d] codes, sdY [rows]; dY [rows, d] bf16 (the same gradient, for dW_d);
 *      X, A, U, H, row_offsets, E, rows, d, f as in moe_expert_bwd; Wdq [E, f, d], sWd [E f];
 *      Wguq [E, d, 2f], sWgu [E d].
 * Out: dX [rows, d], dA, dU [rows, f] bf16; AUq [rows, 2f] codes and sAU [rows] (the
 *      quantised [dA | dU]); dW_g, dW_u [E, f, d], dW_d [E, d, f] bf16.
 * The gate is not folded here (the FP8 layer combines with its gates); dY is g * dY[t].
 * dl_rows and W_r (both or neither; routed layout only): the router term added to dX's rows
 *      as in moe_expert_bwd, after the rows' scales are applied and before the rounding.
 */
int moe_expert_bwd_fp8(const uint8_t* dYq, const float* sdY, const moe_bf16* dY,
                       const moe_bf16* X, const moe_bf16* A, const moe_bf16* U,
                       const moe_bf16* H, const int64_t* row_offsets, int E, int64_t rows, int d,
                       int f, const uint8_t* Wdq, const float* sWd, const uint8_t* Wguq,
                       const float* sWgu, moe_bf16* dX, moe_bf16* dA, moe_bf16* dU, uint8_t* AUq,
                       float* sAU, moe_bf16* dW_g, moe_bf16* dW_u, moe_bf16* dW_d,
                       const float* dl_rows, const float* W_r, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * moe_combine - gate-weighted sum of the expert outputs (C1).
 * Definition: out[t] = sum_{i<k} topk_gate[t,i] * Y_perm[slot_to_row[t,i]] + Y_shared[t],
 * summed in fp32 in slot order, shared term last, one bf16 rounding. Source: section 2.5
 * of the handbook summary (each expert's output is returned to its token); KempnerForge
 * "Features" (shared experts).
 * In : Y_perm [padded rows, d] bf16; topk_gate [T,k] fp32, or NULL when the rows already
 *      carry their gates (moe_expert_fwd with row_gate): then every weight is 1;
 *      slot_to_row [T,k] int32; Y_shared [T,d] bf16 or NULL.  Out: out [T,d] bf16.
 */
int moe_combine(const moe_bf16* Y_perm, const float* topk_gate, const int32_t* slot_to_row,
                const moe_bf16* Y_shared, int64_t T, int d, int k, moe_bf16* out,
                moe_stream_t stream);

/*
 * moe_bias_update - aux-loss-free load balancing (U1), applied once per step after
 * backward with the step's counts. Definition: b[e] = fp32(b[e] + gamma * sign(T*k/E -
 * counts[e])), sign(0) = 0, the sign taken exactly in integers. Source: Apex-3 "Fine-grained
 * MoE" (a per-expert bias balances the load without a loss term) and the training command
 * on that page (router bias rate 1e-3).
 * In : counts [E] int32.  In/out: b [E] fp32.
 */
int moe_bias_update(const int32_t* counts, int E, int64_t T, int k, float gamma, float* b,
                    moe_stream_t stream);

/*
 * moe_bias_update_proportional - the proportional variant of the bias update, named by the
 * Apex-3 benchmark and training commands ("router_bias_update=proportional", rates 0.01 and
 * 1e-3) on "The whole stack, in the open", "Run it yourself". The page prints no formula;
 * reading: the step is proportional to the relative load deviation,
 *   b[e] = fp32(b[e] + fp32(gamma * r_e)),  r_e = fp32((T*k - E*counts[e]) / (T*k)),
 * with the ratio formed exactly from integers in fp64 and each fp32 operation rounded once.
 * In : counts [E] int32.  In/out: b [E] fp32.
 */
int moe_bias_update_proportional(const int32_t* counts, int E, int64_t T, int k, float gamma,
                                 float* b, moe_stream_t stream);

/*
 * moe_combine_bwd - backward of moe_combine (B1).
 * Definition: dY_perm[slot_to_row[t,i]] = bf16(topk_gate[t,i] * dY[t]);
 * dg[t,i] = sum_j dY[t,j] * Y_perm[slot_to_row[t,i], j] (fp32, fixed order).
 * In : dY [T,d] bf16; Y_perm; topk_gate; slot_to_row; row_offsets [E+1] and perm_token
 *      (to zero the padding rows of dY_perm).
 * Out: dY_perm [padded rows, d] bf16 (padding rows 0); dg [T,k] fp32.
 * Gate folded into the experts: topk_gate NULL makes dY_perm plain copies of dY[t] (the
 * gradient of the gated rows); Y_perm and dg both NULL skip the gate gradient, which
 * moe_expert_bwd and moe_gate_grad then form.
 */
int moe_combine_bwd(const moe_bf16* dY, const moe_bf16* Y_perm, const float* topk_gate,
                    const int32_t* slot_to_row, const int64_t* row_offsets,
                    const int32_t* perm_token, int64_t T, int d, int E, int k,
                    moe_bf16* dY_perm, float* dg, moe_stream_t stream);

/*
 * moe_combine_bwd_fp8 - moe_combine_bwd (with gates and the gate gradient) that also writes
 * the E4M3 codes of every dY_perm row it stores, for moe_expert_bwd_fp8: dYq and sdY equal
 * moe_quantize_rows_fp8 of dY_perm bit for bit (padding rows: zero codes, scale 1), without
 * a second pass over dY_perm. A row is bf16(g * dY[t]) with g >= 0, a monotone function of
 * dY[t], so its amax is bf16(g * amax|dY[t]|) and its scale is known before it is written.
 * In / Out as moe_combine_bwd (Y_perm, topk_gate and dg required), plus dYq [padded rows, d]
 * codes and sdY [padded rows] fp32.
 */
int moe_combine_bwd_fp8(const moe_bf16* dY, const moe_bf16* Y_perm, const float* topk_gate,
                        const int32_t* slot_to_row, const int64_t* row_offsets,
                        const int32_t* perm_token, int64_t T, int d, int E, int k,
                        moe_bf16* dY_perm, float* dg, uint8_t* dYq, float* sdY,
                        moe_stream_t stream);

/*
 * moe_expert_bwd - backward of moe_expert_fwd (B2-B5) on tcgen05 tensor cores.
 * Definition, per row p of expert e, with dy = dY[p]:
 *   dh = dy W_d[e]; da = dh * u * s(a) * (1 + a (1 - s(a))); du = dh * silu(a);
 *   dX[p] = da W_g[e] + du W_u[e];
 *   dW_d[e] = sum_p dy^T h;  dW_g[e] = sum_p da^T X[p];  dW_u[e] = sum_p du^T X[p].
 * fp32 accumulation; bf16 results. An expert with no rows gets zero weight gradients.
 * In : dY, X [rows, d] bf16; A, U, H [rows, f] bf16 (from moe_expert_fwd); row_offsets as
 *      in moe_expert_fwd (NULL = one dense expert over `rows` rows); W_g, W_u, W_d.
 *      Padding rows of dY and X must be zero (moe_permute and moe_combine_bwd do this).
 * Out: dX [rows, d] bf16; dA, dU [rows, f] bf16 (the SwiGLU input gradients, kept as
 *      operands of the weight-gradient GEMMs); dW_g, dW_u [E,f,d] bf16; dW_d [E,d,f] bf16.
 * Gate folded into the experts (row_gate and gate_part both given, else both NULL): dY is
 *      the gradient of the gated rows (moe_combine_bwd without gates), H is the gated h of
 *      moe_expert_fwd, and with r = dy W_d[e]: dh = row_gate[p] * r (so dW_d = sum dy^T H
 *      needs no change) and gate_part[p, j] = sum over columns 64j .. 64j+63 of
 *      r * silu(a) * u, in column order (h recomputed in fp32 from a and u): the gate's
 *      gradient in f/64 partial sums. gate_part is [rows, f/64] fp32.
 * parts: which products to run, any union of MOE_BWD_DH (dh and dA, dU; with the gate
 *      folded, gate_part), MOE_BWD_DX (dX, from dA and dU) and MOE_BWD_W (the weight
 *      gradients, from dY, X, H, dA, dU); MOE_BWD_ALL for the whole backward. A caller that
 *      needs the gate's gradient before dX (to form the router term below) runs MOE_BWD_DH
 *      first and the rest after, on the same stream. Other values: MOE_ERR_INVALID_ARG.
 * Router term in the rows (dl_rows and W_r both given, else both NULL; routed layout only):
 *      dX[p] += dl_rows[p] * W_r[e] for each row p of expert e, in fp32 before the row is
 *      rounded, where dl_rows [rows] fp32 holds the logit gradient of each row's slot
 *      (moe_route_bwd writes it) and W_r [E, d] fp32 is the router weight (16-byte
 *      aligned). With sigmoid routing and no balancing losses this is the whole router
 *      input gradient, so moe_permute_bwd then takes neither dlogits nor dx_router.
 */
#define MOE_BWD_DH 1
#define MOE_BWD_DX 2
#define MOE_BWD_W 4
#define MOE_BWD_ALL 7
int moe_expert_bwd(const moe_bf16* dY, const moe_bf16* X, const moe_bf16* A,
                   const moe_bf16* U, const moe_bf16* H, const int64_t* row_offsets, int E,
                   int64_t rows, int d, int f, const moe_bf16* W_g, const moe_bf16* W_u,
                   const moe_bf16* W_d, moe_bf16* dX, moe_bf16* dA, moe_bf16* dU,
                   moe_bf16* dW_g, moe_bf16* dW_u, moe_bf16* dW_d, const float* row_gate,
                   float* gate_part, int parts, const float* dl_rows, const float* W_r,
                   void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_row_gates - each slot's gate at its row of the expert-major layout, for folding the
 * gate into the experts (the combine's weights, moved before the down projection: section
 * 2.5 of the handbook summary weights each expert's output by its gate).
 * Definition: row_gate[slot_to_row[t,i]] = topk_gate[t,i]; every other row (padding) 0.
 * In : topk_gate [T,k] fp32; slot_to_row [T,k] int32 (from moe_permute); rows = the layout's
 *      row capacity (moe_padded_rows).  Out: row_gate [rows] fp32.
 * moe_permute forms the same table in its own pass when given topk_gate and row_gate (rows
 * past the padded layout's end are then left as they were); this call serves callers that
 * permute without them.
 */
int moe_row_gates(const float* topk_gate, const int32_t* slot_to_row, int64_t T, int k,
                  int64_t rows, float* row_gate, moe_stream_t stream);

/*
 * moe_gate_grad - the gate gradient from moe_expert_bwd's partial sums.
 * Definition: dg[t,i] = sum_{j < f/64} gate_part[slot_to_row[t,i], j], in order of j; equal
 * to sum_j dY[t,j] y[t,i,j] (the combine's gate gradient) since y = h W_d^T.
 * In : gate_part [rows, f/64] fp32; slot_to_row [T,k].  Out: dg [T,k] fp32. f % 64 == 0.
 */
int moe_gate_grad(const float* gate_part, const int32_t* slot_to_row, int64_t T, int k, int f,
                  float* dg, moe_stream_t stream);

/*
 * moe_route_bwd - router backward (R1b). No gradient reaches the bias or the choice.
 * Definition: MOE_MODE_SIGMOID: S = sum_i topk_score[t,i]; ds_i = (dg_i - sum_j g_j dg_j)/S;
 *   dlogits[t, idx_i] = ds_i * s_i * (1 - s_i), other experts 0.
 *   MOE_MODE_SOFTMAX: p = exp(l - lse); dlogits[t,e] = p_e * (dg[slot of e, or 0] -
 *   sum_i g_i dg_i) + (2 z_coef / T) * lse[t] * p_e (z-loss with weight 1).
 *   dW_r = dlogits^T x (fp32, fixed-order split reduction over tokens).
 * In : dg [T,k] fp32; x [T,d] bf16; topk_idx, topk_gate, topk_score [T,k]; logits [T,E]
 *      and lse [T] (softmax mode; may be NULL in sigmoid mode); dlogits_extra [T,E] fp32 or
 *      NULL: a further logit gradient (the balancing losses') added before dW_r is formed.
 * Out: dlogits [T,E] fp32 (consumed by moe_permute_bwd for the router's dx term);
 *      dW_r [E,d] fp32.
 * Optional (both or neither; MOE_MODE_SIGMOID without dlogits_extra, where a token's logit
 *      gradient is zero off its chosen experts; else MOE_ERR_INVALID_ARG): slot_to_row
 *      [T,k] int32 in, dl_rows [rows] fp32 out: dl_rows[slot_to_row[t,i]] =
 *      dlogits[t, topk_idx[t,i]], for moe_expert_bwd's router term in the rows. Other
 *      entries of dl_rows are left as they were.
 */
int moe_route_bwd(const float* dg, const moe_bf16* x, const int32_t* topk_idx,
                  const float* topk_gate, const float* topk_score, const float* logits,
                  const float* lse, const float* dlogits_extra, int64_t T, int d, int E, int k,
                  int mode, float z_coef, float* dlogits, float* dW_r,
                  const int32_t* slot_to_row, float* dl_rows, void* ws, size_t ws_bytes,
                  moe_stream_t stream);

/*
 * moe_aux_loss - load-balancing losses of the router (forward).
 * The pages name two such losses without printing their formulas: Megatron's "aux_loss"
 * with coefficient 1e-3, recorded as exactly 1 for a one-expert model (handbook summary,
 * section 2.5), and the sequence-wise loss "seq_aux_alpha=1e-3" of the Apex-3 training
 * command ("The whole stack, in the open", "Run it yourself"; KempnerForge roadmap,
 * "sequence aux loss"). Reading, with pi[t,e] the per-token probabilities over all experts
 * (softmax of the logits in MOE_MODE_SOFTMAX; sigmoid scores normalised to sum 1 in
 * MOE_MODE_SIGMOID) and c the chosen-expert counts:
 *   aux_loss[0] = switch_coef * E * sum_e f_e P_e,  f_e = c_e / (T k),  P_e = mean_t pi[t,e];
 *   aux_loss[1] = seq_coef * mean over the T/seq_len sequences s of sum_e f[s,e] P[s,e],
 *                 f[s,e] = E c[s,e] / (k seq_len),  P[s,e] = mean over s of pi[t,e].
 * In : logits [T,E] fp32 (from moe_route); topk_idx [T,k]. T % seq_len == 0.
 * Out: aux_loss [2] fp32; aux_f [E + (T/seq_len) E] fp32 (f_e then f[s,e], consumed by
 *      moe_aux_loss_bwd). Sums are in a fixed order (fp64 for the final reductions).
 */
int moe_aux_loss(const float* logits, const int32_t* topk_idx, int64_t T, int E, int k,
                 int mode, int64_t seq_len, float switch_coef, float seq_coef, float* aux_loss,
                 float* aux_f, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_aux_loss_bwd - gradient of aux_loss[0] + aux_loss[1] with respect to the logits (the
 * counts get none). With g_e = switch_coef E f_e / T + seq_coef f[s,e] / (T/seq_len * seq_len):
 * softmax mode pi (g - <g, pi>); sigmoid mode (g - <g, pi>) / S * s (1 - s), S = sum of s.
 * In : logits [T,E]; aux_f from moe_aux_loss.  Out: dlogits_aux [T,E] fp32, to be passed to
 * moe_route_bwd as dlogits_extra so that it reaches dW_r and the input gradient.
 */
int moe_aux_loss_bwd(const float* logits, const float* aux_f, int64_t T, int E, int mode,
                     int64_t seq_len, float switch_coef, float seq_coef, float* dlogits_aux,
                     moe_stream_t stream);

/*
 * moe_router_dx - the router's term of the input gradient, dx_r = dlogits W_r, on the tensor
 * cores, for dense logit gradients (the softmax router, or the balancing losses), where
 * moe_permute_bwd's own row loop would read E rows of W_r per token.
 * Definition: dx_r[t,j] = sum_e dlogits[t,e] W_r[e,j]. Both fp32 operands are split into bf16
 * pieces (d0 + d1 + d2, w0 + w1 + w2, each piece the rounding of what the previous ones leave)
 * and the products d0 w0 + d0 w1 + d1 w0 are accumulated in fp32; the dropped terms are below
 * 3 * 2^-16 of each product. Source: section 2.5 of the handbook summary (router logits in
 * fp32; the router's gradient reaches the input through x W_r^T).
 * In : dlogits [T,E] fp32 (from moe_route_bwd); W_r [E,d] fp32. E <= 128, d % 128 == 0.
 * Out: dx_r [T,d] fp32 (16-byte aligned). Scratch: ws (moe_workspace_bytes).
 */
int moe_router_dx(const float* dlogits, const float* W_r, int64_t T, int d, int E, float* dx_r,
                  void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute_bwd - input gradient of the layer (B6).
 * Definition: dx[t] = sum_{i<k} dX_perm[slot_to_row[t,i]] + dx_shared[t] + r[t]
 *                     (fp32 in that order, one bf16 rounding), with the router's term
 *                     r[t] = sum_e dlogits[t,e] * W_r[e] (formed here, from the nonzero logit
 *                     gradients of the token) or r = dx_router (formed by moe_router_dx).
 * In : dX_perm [padded rows, d] bf16; slot_to_row [T,k]; dx_shared [T,d] bf16 or NULL;
 *      dlogits [T,E] fp32 and W_r [E,d] fp32, or both NULL; dx_router [T,d] fp32 or NULL
 *      (not together with dlogits).
 * Out: dx [T,d] bf16.
 */
int moe_permute_bwd(const moe_bf16* dX_perm, const int32_t* slot_to_row,
                    const moe_bf16* dx_shared, const float* dlogits, const float* W_r,
                    const float* dx_router, int64_t T, int d, int E, int k, moe_bf16* dx,
                    moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
