"""fp64 CPU oracle of the fine-grained Mixture-of-Experts layer, forward and backward.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the benchmark's CPU
baseline leg may import this module. The product path never calls it and shares no code
with it.

What the layer computes (the method as the source pages state it):

* "The whole stack, in the open" (Apex-3), section "What's inside", row "Fine-grained MoE":
  a sigmoid router picks the top experts, a per-expert bias balances the load without a
  loss term, and the experts run as grouped GEMMs.
* KempnerForge README, section "Features" (Mixture-of-Experts bullet) and "AI / NeuroAI use
  cases" (sparse architecture research): softmax top-k and DeepSeek-V3 sigmoid routers,
  shared experts, fine-grained experts and router z-loss.
* "How to train a large-scale Mixture-of-Experts model from scratch" (the handbook summary),
  section 2.5 "First training of MoE": the router chooses 8 of 64 experts for each token,
  tokens are sent to the chosen experts and the experts' outputs are returned; a SwiGLU
  expert without bias has three weight matrices; the router logits are computed in fp32
  (``--moe-router-dtype fp32``).

The pages print no formula for the router, the gates, the bias rule, the z-loss or SwiGLU.
The readings taken where they are silent are the workload definitions:

* sigmoid router: s = sigmoid(l), choose the top k of s + b, lower expert index first on
  exact ties; gates = chosen s renormalised to sum 1; b receives no gradient;
* softmax router: p = softmax(l) over all experts, choose the top k of l (same order as p),
  gates = chosen p without renormalisation; z-loss = coef * mean_t(logsumexp(l_t)^2);
* SwiGLU expert: h = silu(x W_g^T) * (x W_u^T), y = h W_d^T;
* shared expert: the same SwiGLU on every token, added with weight 1;
* combine: out_t = sum_i g_ti * y_ti + y_shared_t;
* bias update: b_e <- b_e + gamma * sign(T*k/E - c_e) in fp32, after backward.

Pins (tests/test_oracle_pins.py) hold every function here to facts outside it: k-subset
enumeration with exact ties, closed forms worked by hand (tests/golden), a dense masked
brute force of the forward, central finite differences of the backward, torch's bf16 and
E4M3 conversions, the bias rule's worked example and invariants, the balancing losses' value
of exactly 1 for one expert. tests/test_pins_catch_mistakes.py plants mistakes here one at a
time and checks that a pin fails for each. No function is parity unpinned.

Everything is fp64 numpy; bf16 and fp32 inputs convert to fp64 exactly. Matrix products use
numpy's matmul as a library step. Rows are processed per expert in the order of the
definition; there is no blocking or fusion.

Storage precision. The workloads state "bf16 weights and activations, fp32 accumulate" (and
bf16 outputs and gradients). Every function that produces a tensor the layer hands from one
step to the next takes ``rnd``: ``None`` keeps the exact fp64 value (the plain definition);
``bf16_round`` rounds that stored tensor to bf16 (round to nearest even) at the point it is
materialised, computing it first from unrounded operands:
a, u and h of an expert (h from the unrounded a and u), the expert output y, the shared
expert's a, u, h, y, the layer output, the scaled upstream gradient g * dY of each routed
row, the SwiGLU input gradients da and du (from the stored a and u), each expert's input
gradient, the weight gradients, the shared expert's input gradient and the layer's input
gradient. Router quantities (logits, gates, logit gradients, dW_r) stay fp32-or-better and
are never rounded to bf16.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

SIGMOID = "sigmoid"
SOFTMAX = "softmax"


# ---------------------------------------------------------------------------------------
# conversions

def to64(t) -> np.ndarray:
    """Exact fp64 copy of a host tensor or array (bf16 and fp32 are subsets of fp64)."""
    if hasattr(t, "detach"):
        t = t.detach().cpu().float().numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 value (8 significant bits), ties to even.

    x = m * 2**e with 0.5 <= |m| < 1, so x * 2**(8 - e) has 8 integer bits; rint rounds
    half to even. Below the smallest normal bf16 (2**-126) the spacing stays 2**-133, as for
    bf16 subnormals. Zero stays zero; overflow to infinity is not modelled."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    return np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)


def _r(rnd, x):
    return x if rnd is None else rnd(x)


# ---------------------------------------------------------------------------------------
# FP8 (E4M3) rowwise quantisation of GEMM operands

E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (4 significant bits, ties to even), saturating at
    +-448. Below the smallest normal (2**-6) the spacing stays 2**-9 (subnormals)."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -5)
    q = np.ldexp(np.rint(np.ldexp(x, 4 - e)), e - 4)
    return np.clip(q, -E4M3_MAX, E4M3_MAX)


def quantize_rows_fp8(X: np.ndarray):
    """Rowwise FP8 quantisation (the Apex-3 stack's fp8_rowwise precision): per row,
    scale = fp32(amax / 448) (1 for an all-zero row), q = E4M3(fp32(x / scale)).
    Returns (q, scale); q * scale[:, None] is the dequantised operand. The divisions are
    IEEE fp32 divisions, as the GPU evaluates them."""
    X32 = np.asarray(X, dtype=np.float32)
    amax = np.abs(X32).max(axis=1)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    y = (X32 / scale[:, None]).astype(np.float32)
    return e4m3_round(y), scale.astype(np.float64)


def fp8_dequant_rows(X: np.ndarray) -> np.ndarray:
    q, sc = quantize_rows_fp8(X)
    return q * sc[:, None]


def fp8_dequant_cols(W: np.ndarray) -> np.ndarray:
    """Columnwise FP8 quantisation: each column scaled by its own amax over the rows (the
    rowwise quantisation of W^T), dequantised."""
    return fp8_dequant_rows(np.asarray(W).T).T


def fp8_dgrad_dh(dy: np.ndarray, W_d: np.ndarray) -> np.ndarray:
    """The down projection's data gradient r = dy W_d with FP8 operands (reading of the
    Apex-3 stack's fp8_rowwise precision for the backward): the rows of dy are scaled along
    the contraction axis d (one scale per row), W_d [d, f] per output column j (one scale
    per column, over d), and the products accumulate exactly."""
    return fp8_dequant_rows(dy) @ fp8_dequant_cols(W_d)


def fp8_dgrad_dx(da: np.ndarray, du: np.ndarray, W_g: np.ndarray, W_u: np.ndarray) -> np.ndarray:
    """The expert's input gradient dX = da W_g + du W_u as one product over K = 2f with FP8
    operands: each row of [da | du] gets one scale over its 2f elements, each column i of
    [W_g; W_u] (2f x d) one scale over its 2f elements, and the products accumulate
    exactly."""
    AU = fp8_dequant_rows(np.concatenate([da, du], axis=1))
    W = fp8_dequant_cols(np.concatenate([W_g, W_u], axis=0))
    return AU @ W


def sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def silu(z: np.ndarray) -> np.ndarray:
    return z * sigmoid(z)


# ---------------------------------------------------------------------------------------
# router (forward)

def router_logits(x: np.ndarray, W_r: np.ndarray) -> np.ndarray:
    """l[t, e] = sum_j x[t, j] * W_r[e, j] (router logits, fp32 router per section 2.5)."""
    return x @ W_r.T


def _top_k_desc(score: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, largest first, lower index first on ties."""
    T, E = score.shape
    index = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((index, -score), axis=-1)  # primary key: -score, then index
    return order[:, :k]


def route_sigmoid(logits: np.ndarray, b: np.ndarray, k: int) -> dict:
    """Sigmoid router with selection bias (Apex-3 "Fine-grained MoE"; DeepSeek-V3 sigmoid
    routing in KempnerForge "Features").

    The bias only steers which experts are chosen; gates are the chosen sigmoid scores
    renormalised to sum 1."""
    s = sigmoid(logits)
    v = s + b[None, :]
    idx = _top_k_desc(v, k)
    s_sel = np.take_along_axis(s, idx, axis=1)
    gate = s_sel / s_sel.sum(axis=1, keepdims=True)
    return {"idx": idx, "gate": gate, "score": s_sel, "select_value": v}


def route_softmax(logits: np.ndarray, k: int, z_coef: float) -> dict:
    """Softmax top-k router with router z-loss (KempnerForge "Features").

    p = softmax over all experts; the k largest logits are chosen (the same order as p);
    gates are the chosen p, not renormalised; z = z_coef * mean_t(lse_t^2)."""
    m = logits.max(axis=1, keepdims=True)
    ex = np.exp(logits - m)
    denom = ex.sum(axis=1, keepdims=True)
    p = ex / denom
    lse = (m + np.log(denom))[:, 0]
    idx = _top_k_desc(logits, k)
    gate = np.take_along_axis(p, idx, axis=1)
    z = z_coef * float(np.mean(lse * lse))
    return {"idx": idx, "gate": gate, "score": gate.copy(), "p": p, "lse": lse, "z_loss": z,
            "select_value": logits}


def route(logits: np.ndarray, mode: str, k: int, b: np.ndarray | None = None,
          z_coef: float = 0.0) -> dict:
    if mode == SIGMOID:
        r = route_sigmoid(logits, b, k)
    elif mode == SOFTMAX:
        r = route_softmax(logits, k, z_coef)
    else:
        raise ValueError(mode)
    r["logits"] = logits
    return r


def near_tie_tokens(select_value: np.ndarray, k: int, gap: float = 1e-6) -> np.ndarray:
    """Tokens whose sorted top-(k+1) selection values have an adjacent gap below ``gap``.

    On such tokens an fp32 and an fp64 evaluation of the selection value may order the
    experts differently; they are reported and left out of bit-exact index checks."""
    E = select_value.shape[1]
    kk = min(k + 1, E)
    srt = -np.sort(-select_value, axis=1)[:, :kk]
    if kk < 2:
        return np.zeros(select_value.shape[0], dtype=bool)
    return (np.abs(np.diff(srt, axis=1)) < gap).any(axis=1)


def select_brute_force(v_row: np.ndarray, k: int) -> tuple:
    """Chosen expert set of one token by enumerating every k-subset: the set with the
    largest total selection value; among equal totals, the lexicographically smallest
    sorted index tuple. Returns the indices ordered by descending value, lower index
    first on ties. Only for tiny E."""
    E = v_row.shape[0]
    best, best_sum = None, -math.inf
    for comb in itertools.combinations(range(E), k):
        tot = float(sum(v_row[list(comb)]))
        if tot > best_sum:
            best, best_sum = comb, tot
    return tuple(sorted(best, key=lambda e: (-v_row[e], e)))


# ---------------------------------------------------------------------------------------
# dispatch (token permutation)

def dispatch(idx: np.ndarray, E: int) -> dict:
    """Send every (token, slot) to its expert: per-expert counts, exclusive-scan offsets,
    and rows ordered by (expert, token), which is unique because a token's k experts are
    distinct (section 2.5: tokens must be sent to the selected experts)."""
    T, k = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    tok = np.repeat(np.arange(T), k)
    slot = np.tile(np.arange(k), T)
    e_flat = idx.reshape(-1)
    order = np.lexsort((tok, e_flat))  # primary key expert, then token
    perm_token = tok[order]
    perm_slot = slot[order]
    slot_to_row = np.empty((T, k), dtype=np.int64)
    slot_to_row[perm_token, perm_slot] = np.arange(T * k)
    return {"counts": counts, "offsets": offsets, "perm_token": perm_token,
            "perm_slot": perm_slot, "slot_to_row": slot_to_row}


# ---------------------------------------------------------------------------------------
# experts and combine

def swiglu_expert_fp8(rows: np.ndarray, W_g: np.ndarray, W_u: np.ndarray, W_d: np.ndarray,
                      rnd=None):
    """The SwiGLU expert with FP8 rowwise GEMM operands (row scales for the activations,
    per-output-channel scales for the weights, fp32-exact accumulation): x and the rows of
    W_g, W_u, W_d are quantised; h is stored (rnd) and then quantised per row for the down
    projection."""
    xq = fp8_dequant_rows(rows)
    a = xq @ fp8_dequant_rows(W_g).T
    u = xq @ fp8_dequant_rows(W_u).T
    h = _r(rnd, silu(a) * u)
    y = _r(rnd, fp8_dequant_rows(h) @ fp8_dequant_rows(W_d).T)
    return _r(rnd, a), _r(rnd, u), h, y


def swiglu_expert(rows: np.ndarray, W_g: np.ndarray, W_u: np.ndarray, W_d: np.ndarray,
                  rnd=None, row_gate: np.ndarray | None = None):
    """One bias-free SwiGLU expert (three weight matrices, section 2.5):
    a = x W_g^T, u = x W_u^T, h = silu(a) * u, y = h W_d^T. Returns the stored a, u, h, y.

    ``row_gate`` (one value per row) moves the combine's gate weight before the down
    projection: h is stored as g * silu(a) * u, so y is the gated output g * (h W_d^T). In
    exact arithmetic this is the same product (W_d is linear); with ``rnd`` it models a
    layout that stores the gated h."""
    a = rows @ W_g.T
    u = rows @ W_u.T
    hv = silu(a) * u
    if row_gate is not None:
        hv = row_gate[:, None] * hv
    h = _r(rnd, hv)
    y = _r(rnd, h @ W_d.T)
    return _r(rnd, a), _r(rnd, u), h, y


def experts_forward(x_perm: np.ndarray, offsets: np.ndarray, W_g, W_u, W_d, rnd=None,
                    fp8: bool = False, row_gate: np.ndarray | None = None) -> dict:
    """Each expert applied to its own contiguous segment of the permuted rows (``row_gate``:
    each row's gate folded into its expert, as in ``swiglu_expert``)."""
    expert = swiglu_expert_fp8 if fp8 else swiglu_expert
    N = x_perm.shape[0]
    f = W_g.shape[1]
    d_out = W_d.shape[1]
    A = np.zeros((N, f)); U = np.zeros((N, f)); H = np.zeros((N, f)); Y = np.zeros((N, d_out))
    for e in range(W_g.shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            kw = {} if row_gate is None else {"row_gate": row_gate[lo:hi]}
            A[lo:hi], U[lo:hi], H[lo:hi], Y[lo:hi] = expert(x_perm[lo:hi], W_g[e], W_u[e],
                                                            W_d[e], rnd, **kw)
    return {"A": A, "U": U, "H": H, "Y_perm": Y}


def combine(Y_perm: np.ndarray, gate: np.ndarray, slot_to_row: np.ndarray,
            Y_shared: np.ndarray | None, rnd=None) -> np.ndarray:
    """out_t = sum over slots of gate * expert output, plus the shared expert's output
    (section 2.5: each expert's output is returned to the token)."""
    T, k = gate.shape
    out = np.zeros((T, Y_perm.shape[1]))
    for i in range(k):
        out += gate[:, i:i + 1] * Y_perm[slot_to_row[:, i]]
    if Y_shared is not None:
        out += Y_shared
    return _r(rnd, out)


# ---------------------------------------------------------------------------------------
# whole layer, forward

def layer_forward(inp: dict, mode: str, k: int, z_coef: float = 0.0,
                  logits: np.ndarray | None = None, idx: np.ndarray | None = None,
                  rnd=None, aux: tuple | None = None, fp8: bool = False,
                  fold_gate: bool = False, fp8_dgrad: bool = False,
                  router_rows: bool = False) -> dict:
    """Full forward of the layer from fp64 copies of the inputs.

    ``logits`` replaces the fp64 router logits (used to replay the GPU's fp32 logits, so
    that index checks compare selections made from identical logits). ``idx`` replaces
    the chosen experts (used so value checks do not cascade from a near-tie).
    ``fold_gate`` applies each slot's gate inside its expert (before the linear down
    projection) and combines without weights: the same value in exact arithmetic, and with
    ``rnd`` the rounding of a layout that stores the gated h and y. ``fp8_dgrad`` marks the
    layer whose backward data-gradient products take FP8 operands (``layer_backward``).
    ``router_rows`` marks a backward that adds the router's input-gradient term to each
    slot's expert row before that row is stored (``layer_backward``): sigmoid routing
    without balancing losses only, where the logit gradient of a token is nonzero only at
    its chosen experts."""
    x = inp["x"]
    E = inp["W_r"].shape[0]
    if logits is None:
        logits = router_logits(x, inp["W_r"])
    r = route(logits, mode, k, inp.get("b"), z_coef)
    if idx is not None:
        r = _regate(r, logits, idx, mode, inp.get("b"), z_coef)
    disp = dispatch(r["idx"], E)
    x_perm = x[disp["perm_token"]]
    if fold_gate and fp8:
        raise ValueError("the FP8 expert model quantises the ungated h; fold_gate is bf16 only")
    row_gate = r["gate"][disp["perm_token"], disp["perm_slot"]] if fold_gate else None
    ex = experts_forward(x_perm, disp["offsets"], inp["W_g"], inp["W_u"], inp["W_d"], rnd, fp8,
                         row_gate=row_gate)
    shared = None
    if "Ws_g" in inp:
        shared = (swiglu_expert_fp8 if fp8 else swiglu_expert)(x, inp["Ws_g"], inp["Ws_u"],
                                                               inp["Ws_d"], rnd)
    out = combine(ex["Y_perm"], np.ones_like(r["gate"]) if fold_gate else r["gate"],
                  disp["slot_to_row"], None if shared is None else shared[3], rnd)
    if fp8_dgrad and fold_gate:
        raise ValueError("the FP8 data gradients take the ungated rows; fold_gate is bf16 only")
    if router_rows and (mode != SIGMOID or aux is not None):
        raise ValueError("the router term fits the expert rows only for sparse logit gradients")
    res = {**r, **disp, **ex, "X_perm": x_perm, "out": out, "mode": mode, "k": k,
           "z_coef": z_coef, "rnd": rnd, "aux": aux, "row_gate": row_gate,
           "fp8_dgrad": fp8_dgrad, "router_rows": router_rows}
    if aux is not None:  # (seq_len, switch_coef, seq_coef)
        a = aux_losses(logits, r["idx"], mode, *aux)
        res["aux_switch"], res["aux_seq"] = a["switch"], a["seq"]
    if shared is not None:
        res["shared"] = dict(zip("AUHY", shared))
    return res


def _regate(r: dict, logits, idx, mode, b, z_coef) -> dict:
    """Gates and scores for a given choice of experts (replay of a selection)."""
    idx = np.asarray(idx, dtype=np.int64)
    r = dict(r)
    r["idx"] = idx
    if mode == SIGMOID:
        s = sigmoid(logits)
        s_sel = np.take_along_axis(s, idx, axis=1)
        r["score"] = s_sel
        r["gate"] = s_sel / s_sel.sum(axis=1, keepdims=True)
    else:
        r["gate"] = np.take_along_axis(r["p"], idx, axis=1)
        r["score"] = r["gate"].copy()
    return r


def layer_forward_dense_masked(inp: dict, mode: str, k: int, z_coef: float = 0.0) -> np.ndarray:
    """Brute-force forward: every expert on every token, then out = sum_e m[t, e] y_e(x_t)
    with m the gate of a chosen expert and 0 elsewhere. No permutation at all; an
    independent path to the same definition."""
    x = inp["x"]
    logits = router_logits(x, inp["W_r"])
    r = route(logits, mode, k, inp.get("b"), z_coef)
    T = x.shape[0]
    E = inp["W_r"].shape[0]
    m = np.zeros((T, E))
    for i in range(k):
        m[np.arange(T), r["idx"][:, i]] = r["gate"][:, i]
    out = np.zeros_like(x)
    for e in range(E):
        _, _, _, y = swiglu_expert(x, inp["W_g"][e], inp["W_u"][e], inp["W_d"][e])
        out += m[:, e:e + 1] * y
    if "Ws_g" in inp:
        out += swiglu_expert(x, inp["Ws_g"], inp["Ws_u"], inp["Ws_d"])[3]
    return out


def loss(fwd: dict, dY: np.ndarray) -> float:
    """Scalar whose gradient the backward computes: <out, dY> plus the z-loss and the
    balancing losses when present (weight 1 each)."""
    L = float(np.sum(fwd["out"] * dY))
    if fwd["mode"] == SOFTMAX:
        L += fwd["z_loss"]
    if fwd.get("aux") is not None:
        L += fwd["aux_switch"] + fwd["aux_seq"]
    return L


# ---------------------------------------------------------------------------------------
# backward

def swiglu_backward(dh: np.ndarray, a: np.ndarray, u: np.ndarray):
    """d/da and d/du of h = silu(a) * u."""
    sa = sigmoid(a)
    da = dh * u * sa * (1.0 + a * (1.0 - sa))
    du = dh * silu(a)
    return da, du


def expert_backward(dy: np.ndarray, x: np.ndarray, a: np.ndarray, u: np.ndarray,
                    h: np.ndarray, W_g: np.ndarray, W_u: np.ndarray, W_d: np.ndarray,
                    rnd=None, row_gate: np.ndarray | None = None,
                    fp8_dgrad: bool = False) -> dict:
    """Backward of one SwiGLU expert over its rows, given the upstream gradient of its
    output and the stored a, u, h of the forward:
    dh = dy W_d, (da, du) from the SwiGLU derivative, dx = da W_g + du W_u,
    dW_d = dy^T h, dW_g = da^T x, dW_u = du^T x.

    With ``row_gate`` (the gate folded into the expert, h stored gated): dy is the gradient
    of the gated output, r = dy W_d, dh = g * r, dW_d = dy^T h (h already carries g), and
    the gate's gradient per row is dg = sum_j r_j silu(a_j) u_j (returned as "dg_row").

    ``fp8_dgrad``: the two data-gradient products (r and dx) take FP8 operands
    (``fp8_dgrad_dh``, ``fp8_dgrad_dx``, the latter on the stored da and du); the weight
    gradients stay products of the stored bf16 tensors."""
    r = fp8_dgrad_dh(dy, W_d) if fp8_dgrad else dy @ W_d
    dh = r if row_gate is None else row_gate[:, None] * r
    da, du = swiglu_backward(dh, a, u)
    da, du = _r(rnd, da), _r(rnd, du)
    dx = fp8_dgrad_dx(da, du, W_g, W_u) if fp8_dgrad else da @ W_g + du @ W_u
    res = {"dA": da, "dU": du, "dX": _r(rnd, dx), "dX_exact": dx,
           "dW_d": _r(rnd, dy.T @ h), "dW_g": _r(rnd, da.T @ x), "dW_u": _r(rnd, du.T @ x)}
    if row_gate is not None:
        res["dg_row"] = np.sum(r * silu(a) * u, axis=1)
    return res


def router_backward(dg: np.ndarray, route_res: dict, x: np.ndarray, W_r: np.ndarray,
                    mode: str, z_coef: float, T_norm: int | None = None,
                    dl_extra: np.ndarray | None = None) -> dict:
    """Gradient of the loss with respect to the router logits, W_r and x, given the
    gradient with respect to the gates. No gradient flows through the choice of experts
    or into the bias. ``T_norm`` is the token count of the z-loss mean (default: the rows
    given)."""
    idx, gate = route_res["idx"], route_res["gate"]
    T, k = idx.shape
    if T_norm is None:
        T_norm = T
    E = W_r.shape[0]
    dl = np.zeros((T, E))
    rows = np.arange(T)
    if mode == SIGMOID:
        s = route_res["score"]
        S = s.sum(axis=1, keepdims=True)
        gdg = (gate * dg).sum(axis=1, keepdims=True)
        ds = (dg - gdg) / S
        for i in range(k):
            dl[rows, idx[:, i]] += ds[:, i] * s[:, i] * (1.0 - s[:, i])
    else:
        p, lse = route_res["p"], route_res["lse"]
        pdg = (gate * dg).sum(axis=1, keepdims=True)
        sel = np.zeros((T, E))
        for i in range(k):
            sel[rows, idx[:, i]] = dg[:, i]
        dl = p * (sel - pdg) + (2.0 * z_coef / T_norm) * lse[:, None] * p
    if dl_extra is not None:
        dl = dl + dl_extra
    return {"dlogits": dl, "dW_r": dl.T @ x, "dx_r": dl @ W_r}


def layer_backward(inp: dict, fwd: dict, dY: np.ndarray, T_norm: int | None = None,
                   dl_extra: np.ndarray | None = None, weight_grads: bool = True) -> dict:
    """Gradients of ``loss`` with respect to x, every weight and the router (stored in the
    precision the forward used).

    For a forward over a subset of a batch's tokens (each token's output and input gradient
    depend only on its own routing, rows and upstream gradient): ``T_norm`` is the batch's
    token count that the z-loss mean divides by, ``dl_extra`` the batch's balancing-loss
    logit gradient rows of these tokens (it replaces the subset's own, whose counts would
    be the subset's), and ``weight_grads=False`` skips the weight gradients, which only the
    whole batch gives."""
    rnd = fwd.get("rnd")
    f8 = bool(fwd.get("fp8_dgrad"))
    idx, gate, s2r = fwd["idx"], fwd["gate"], fwd["slot_to_row"]
    T, k = idx.shape
    E = inp["W_r"].shape[0]
    offs = fwd["offsets"]
    tok = fwd["perm_token"]
    slot = fwd["perm_slot"]
    row_gate = fwd.get("row_gate")
    if row_gate is None:
        dY_perm, dg = combine_backward(dY, fwd["Y_perm"], gate, s2r, tok, slot, rnd)
    else:  # gate folded into the experts: rows get the token gradient itself
        dY_perm, dg = dY[tok], np.zeros((T, k))
    # experts backward
    N, d = fwd["X_perm"].shape
    f = inp["W_g"].shape[1]
    dX_perm = np.zeros((N, d))
    if weight_grads:
        dW_g = np.zeros(inp["W_g"].shape); dW_u = np.zeros(inp["W_u"].shape)
        dW_d = np.zeros(inp["W_d"].shape)
    dA = np.zeros((N, f)); dU = np.zeros((N, f))
    rows_term = bool(fwd.get("router_rows"))
    dX_exact = np.zeros((N, d)) if rows_term else None
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        g = expert_backward(dY_perm[lo:hi], fwd["X_perm"][lo:hi], fwd["A"][lo:hi],
                            fwd["U"][lo:hi], fwd["H"][lo:hi], inp["W_g"][e], inp["W_u"][e],
                            inp["W_d"][e], rnd,
                            row_gate=None if row_gate is None else row_gate[lo:hi],
                            fp8_dgrad=f8)
        if row_gate is not None:
            dg[tok[lo:hi], slot[lo:hi]] = g["dg_row"]
        dX_perm[lo:hi], dA[lo:hi], dU[lo:hi] = g["dX"], g["dA"], g["dU"]
        if rows_term:
            dX_exact[lo:hi] = g["dX_exact"]
        if weight_grads:
            dW_g[e], dW_u[e], dW_d[e] = g["dW_g"], g["dW_u"], g["dW_d"]
    res = {"dY_perm": dY_perm, "dg": dg, "dA": dA, "dU": dU, "dX_perm": dX_perm}
    if weight_grads:
        res.update(dW_g=dW_g, dW_u=dW_u, dW_d=dW_d)
    if "shared" in fwd:
        sh = fwd["shared"]
        g = expert_backward(dY, inp["x"], sh["A"], sh["U"], sh["H"], inp["Ws_g"], inp["Ws_u"],
                            inp["Ws_d"], rnd, fp8_dgrad=f8)
        if weight_grads:
            res["dWs_d"], res["dWs_g"], res["dWs_u"] = g["dW_d"], g["dW_g"], g["dW_u"]
        res["dx_shared"] = g["dX"]
    dl_aux = dl_extra
    if dl_aux is None and fwd.get("aux") is not None:
        dl_aux = aux_losses_backward(fwd["logits"], idx, fwd["mode"], *fwd["aux"])
    rb = router_backward(dg, fwd, inp["x"], inp["W_r"], fwd["mode"], fwd["z_coef"],
                         T_norm=T_norm, dl_extra=dl_aux)
    res.update(rb)
    if rows_term:
        # each chosen slot's row carries its token's router term dl[t, e] W_r[e] before the
        # row is stored; the token sum then has no separate router summand (the same value
        # in exact arithmetic: the logit gradient is zero off the chosen experts)
        terms = slot_router_terms(rb["dlogits"], idx, inp["W_r"])
        for i in range(k):
            rws = s2r[:, i]
            dX_perm[rws] = _r(rnd, dX_exact[rws] + terms[:, i])
        res["dX_perm"] = dX_perm
        res["dx"] = input_gradient(dX_perm, s2r, res.get("dx_shared"), None, rnd)
    else:
        res["dx"] = input_gradient(dX_perm, s2r, res.get("dx_shared"), rb["dx_r"], rnd)
    return res


def slot_router_terms(dlogits: np.ndarray, idx: np.ndarray, W_r: np.ndarray) -> np.ndarray:
    """[T, k, d]: each chosen slot's share of the router's input gradient dl W_r, i.e.
    dl[t, idx[t, i]] W_r[idx[t, i]]. Their sum over the slots is dl W_r whenever dl is zero
    off the chosen experts."""
    T = idx.shape[0]
    return dlogits[np.arange(T)[:, None], idx][:, :, None] * W_r[idx]


def combine_backward(dY, Y_perm, gate, slot_to_row, perm_token, perm_slot, rnd=None):
    """Backward of the combine: each routed row receives its gate times the token's
    upstream gradient; the gate gradient is the inner product of the upstream gradient
    with that row's expert output."""
    T, k = gate.shape
    dY_perm = _r(rnd, gate[perm_token, perm_slot][:, None] * dY[perm_token])
    dg = np.zeros((T, k))
    for i in range(k):
        dg[:, i] = np.sum(dY * Y_perm[slot_to_row[:, i]], axis=1)
    return dY_perm, dg


def input_gradient(dX_perm, slot_to_row, dx_shared, dx_router, rnd=None):
    """dx_t = sum over the token's slots of its rows' input gradients, plus the shared
    expert's and the router's input gradients."""
    T, k = slot_to_row.shape
    dx = np.zeros((T, dX_perm.shape[1]))
    for i in range(k):
        dx += dX_perm[slot_to_row[:, i]]
    if dx_shared is not None:
        dx += dx_shared
    if dx_router is not None:
        dx += dx_router
    return _r(rnd, dx)


# ---------------------------------------------------------------------------------------
# load-balancing auxiliary losses

def router_probs(logits: np.ndarray, mode: str) -> np.ndarray:
    """Per-token probability vector over all experts used by the balancing losses: the
    softmax in softmax mode; the sigmoid scores normalised to sum 1 in sigmoid mode."""
    if mode == SOFTMAX:
        m = logits.max(axis=1, keepdims=True)
        ex = np.exp(logits - m)
        return ex / ex.sum(axis=1, keepdims=True)
    s = sigmoid(logits)
    return s / s.sum(axis=1, keepdims=True)


def aux_losses(logits: np.ndarray, idx: np.ndarray, mode: str, seq_len: int,
               switch_coef: float, seq_coef: float) -> dict:
    """Load-balancing losses (handbook summary, section 2.5: --moe-router-load-balancing-type
    aux_loss with coefficient 1e-3, recorded as exactly 1 for a one-expert model; Apex-3
    training command: seq_aux_alpha=1e-3; KempnerForge roadmap: sequence aux loss).

    Readings (no formula on the pages):
      switch = switch_coef * E * sum_e f_e P_e, f_e = c_e / (T k), P_e = mean_t pi[t, e];
      seq    = seq_coef * mean over sequences s of sum_e f[s,e] P[s,e],
               f[s,e] = E c[s,e] / (k L), P[s,e] = mean over the sequence of pi[t, e],
    with pi the per-token probabilities of ``router_probs`` and c the chosen-expert counts.
    Both equal their coefficient times 1 for E = 1, k = 1."""
    T, E = logits.shape
    k = idx.shape[1]
    pi = router_probs(logits, mode)
    onehot = np.zeros((T, E))
    for i in range(k):
        onehot[np.arange(T), idx[:, i]] = 1.0
    f = onehot.sum(axis=0) / (T * k)
    P = pi.mean(axis=0)
    switch_unscaled = E * float(np.sum(f * P))
    B = T // seq_len
    fs = E * onehot.reshape(B, seq_len, E).sum(axis=1) / (k * seq_len)
    Ps = pi.reshape(B, seq_len, E).mean(axis=1)
    seq_unscaled = float(np.mean(np.sum(fs * Ps, axis=1)))
    return {"switch": switch_coef * switch_unscaled, "seq": seq_coef * seq_unscaled,
            "switch_unscaled": switch_unscaled, "seq_unscaled": seq_unscaled,
            "f": f, "f_seq": fs, "pi": pi}


def aux_losses_backward(logits: np.ndarray, idx: np.ndarray, mode: str, seq_len: int,
                        switch_coef: float, seq_coef: float) -> np.ndarray:
    """Gradient of switch + seq with respect to the logits (the counts f are piecewise
    constant and receive none)."""
    T, E = logits.shape
    a = aux_losses(logits, idx, mode, seq_len, switch_coef, seq_coef)
    B = T // seq_len
    g = switch_coef * E * a["f"][None, :] / T + \
        (seq_coef / B) * np.repeat(a["f_seq"], seq_len, axis=0) / seq_len
    pi = a["pi"]
    gpi = np.sum(g * pi, axis=1, keepdims=True)
    if mode == SOFTMAX:
        return pi * (g - gpi)
    s = sigmoid(logits)
    S = s.sum(axis=1, keepdims=True)
    return (g - gpi) / S * s * (1.0 - s)


# ---------------------------------------------------------------------------------------
# aux-loss-free bias update

def bias_update(counts: np.ndarray, b: np.ndarray, T: int, k: int, gamma: float) -> np.ndarray:
    """b_e <- b_e + gamma * sign(mean load - c_e), evaluated in fp32 with one rounding.

    Under-loaded experts get a larger bias and so are chosen more often; the bias never
    enters a loss (Apex-3 "Fine-grained MoE": the bias balances the load without a loss
    term). mean load = T*k/E."""
    E = b.shape[0]
    mean = np.float64(T) * k / E
    sgn = np.sign(mean - counts.astype(np.float64)).astype(np.float32)
    return (np.asarray(b, dtype=np.float32) + np.float32(gamma) * sgn).astype(np.float32)


def bias_update_proportional(counts: np.ndarray, b: np.ndarray, T: int, k: int,
                             gamma: float) -> np.ndarray:
    """Proportional variant (the Apex-3 commands' router_bias_update=proportional, whose
    formula the page does not print). Reading: the step is proportional to the relative
    load deviation, b_e <- b_e + gamma * (mean - c_e) / mean with mean = T*k/E.

    Evaluated as: r_e = (T*k - E*c_e) / (T*k) exactly in fp64 (integers), rounded once to
    fp32; then fp32(gamma * r_e) and fp32(b_e + that), each one fp32 rounding."""
    E = b.shape[0]
    N = np.float64(T) * k
    r = ((N - np.float64(E) * counts.astype(np.float64)) / N).astype(np.float32)
    step = (np.float32(gamma) * r).astype(np.float32)
    return (np.asarray(b, dtype=np.float32) + step).astype(np.float32)


# ---------------------------------------------------------------------------------------
# sampled evaluation for workloads too large to run whole on the CPU

def token_forward(inp: dict, t: int, experts, gates, rnd=None, fp8: bool = False,
                  fold_gate: bool = False) -> np.ndarray:
    """out_t for one token given its chosen experts and gates (``fold_gate``: each gate
    applied inside its expert, as in ``layer_forward``)."""
    expert = swiglu_expert_fp8 if fp8 else swiglu_expert
    x_t = inp["x"][t:t + 1]
    out = np.zeros((1, inp["x"].shape[1]))
    for e, g in zip(experts, gates):
        if fold_gate:
            out += swiglu_expert(x_t, inp["W_g"][e], inp["W_u"][e], inp["W_d"][e], rnd,
                                 row_gate=np.array([g]))[3]
        else:
            out += g * expert(x_t, inp["W_g"][e], inp["W_u"][e], inp["W_d"][e], rnd)[3]
    if "Ws_g" in inp:
        out += expert(x_t, inp["Ws_g"], inp["Ws_u"], inp["Ws_d"], rnd)[3]
    return _r(rnd, out[0])


def token_backward(inp: dict, t: int, logits_t: np.ndarray, experts, mode: str, k: int,
                   dY_t: np.ndarray, z_coef: float, T: int, rnd=None,
                   dl_extra_t: np.ndarray | None = None, fp8: bool = False,
                   fold_gate: bool = False) -> dict:
    """Gradient rows of one token: dx_t, dg_t and the router logit gradient for it.

    A token's dx depends only on its own routing, experts and upstream gradient, so it can
    be evaluated alone. ``T`` is the batch size that normalises the z-loss mean.
    ``dl_extra_t`` adds a logit gradient row for the token (the balancing losses', which
    depend on batch-wide counts)."""
    x_t = inp["x"][t:t + 1]
    lg = logits_t[None, :]
    r = route(lg, mode, k, inp.get("b"), z_coef)
    r = _regate(r, lg, np.asarray([experts]), mode, inp.get("b"), z_coef)
    gate = r["gate"][0]
    dx = np.zeros((1, x_t.shape[1]))
    dg = np.zeros((1, k))
    expert = swiglu_expert_fp8 if fp8 else swiglu_expert
    for i, e in enumerate(experts):
        a, u, h, y = expert(x_t, inp["W_g"][e], inp["W_u"][e], inp["W_d"][e], rnd)
        if fold_gate:  # dY_t itself reaches the gated expert; dg from r = dY_t W_d
            rr = dY_t[None, :] @ inp["W_d"][e]
            dg[0, i] = float(np.sum(rr * silu(a) * u))
            dH = gate[i] * rr
        else:
            dg[0, i] = float(np.sum(dY_t * y[0]))
            dH = _r(rnd, gate[i] * dY_t[None, :]) @ inp["W_d"][e]
        dA, dU = swiglu_backward(dH, a, u)
        dA, dU = _r(rnd, dA), _r(rnd, dU)
        dx += _r(rnd, dA @ inp["W_g"][e] + dU @ inp["W_u"][e])
    if "Ws_g" in inp:
        a, u, h, y = expert(x_t, inp["Ws_g"], inp["Ws_u"], inp["Ws_d"], rnd)
        dA, dU = swiglu_backward(dY_t[None, :] @ inp["Ws_d"], a, u)
        dA, dU = _r(rnd, dA), _r(rnd, dU)
        dx += _r(rnd, dA @ inp["Ws_g"] + dU @ inp["Ws_u"])
    rb = router_backward(dg, r, x_t, inp["W_r"], mode, z_coef, T_norm=T,
                         dl_extra=None if dl_extra_t is None else dl_extra_t[None, :])
    dx += rb["dx_r"]
    return {"dx": _r(rnd, dx[0]), "dg": dg[0], "dlogits": rb["dlogits"][0]}


def _gemm_operands(X, Wg, Wu, fp8):
    """The operands the gate/up products see: the bf16 values, or their E4M3 rowwise
    dequantisations when fp8."""
    if fp8:
        return fp8_dequant_rows(X), fp8_dequant_rows(Wg), fp8_dequant_rows(Wu)
    return X, Wg, Wu


def expert_weight_grad_entries(inp: dict, e: int, tokens: np.ndarray, slots_gate: np.ndarray,
                               dY: np.ndarray, entries_d, entries_gu, rnd=None,
                               fp8: bool = False, fold_gate: bool = False) -> dict:
    """Chosen entries of dW_d[e], dW_g[e] and dW_u[e].

    ``tokens`` are the tokens routed to expert e in ascending order and ``slots_gate`` their
    gates for e. ``entries_d`` lists (i, j) of dW_d[e][i, j] = sum_p dY_perm[p, i] h[p, j];
    ``entries_gu`` lists (j, i) of dW_g[e][j, i] = sum_p dA[p, j] x_perm[p, i] (and dW_u)."""
    X = inp["x"][tokens]
    # fold_gate: the rows carry the token gradient itself and the gate sits in h and dh
    g = slots_gate if fold_gate else np.ones(len(tokens))
    dYp = dY[tokens] if fold_gate else _r(rnd, slots_gate[:, None] * dY[tokens])
    Wg, Wu, Wd = inp["W_g"][e], inp["W_u"][e], inp["W_d"][e]
    res = {"dW_d": [], "dW_g": [], "dW_u": []}
    Xo, Wgo, Wuo = _gemm_operands(X, Wg, Wu, fp8)
    for (i, j) in entries_d:
        a, u = Xo @ Wgo[j], Xo @ Wuo[j]
        h = _r(rnd, g * silu(a) * u)
        res["dW_d"].append(float(_r(rnd, np.sum(dYp[:, i] * h))))
    for (j, i) in entries_gu:
        a, u = _r(rnd, Xo @ Wgo[j]), _r(rnd, Xo @ Wuo[j])
        dh = g * (dYp @ Wd[:, j])
        da, du = swiglu_backward(dh, a, u)
        res["dW_g"].append(float(_r(rnd, np.sum(_r(rnd, da) * X[:, i]))))
        res["dW_u"].append(float(_r(rnd, np.sum(_r(rnd, du) * X[:, i]))))
    return res


def shared_weight_grad_entries(inp: dict, dY: np.ndarray, entries_d, entries_gu, rnd=None,
                               fp8: bool = False) -> dict:
    """Chosen entries of the shared expert's weight gradients (every token, weight 1)."""
    X = inp["x"]
    Wg, Wu, Wd = inp["Ws_g"], inp["Ws_u"], inp["Ws_d"]
    res = {"dWs_d": [], "dWs_g": [], "dWs_u": []}
    Xo, Wgo, Wuo = _gemm_operands(X, Wg, Wu, fp8)
    for (i, j) in entries_d:
        a, u = Xo @ Wgo[j], Xo @ Wuo[j]
        h = _r(rnd, silu(a) * u)
        res["dWs_d"].append(float(_r(rnd, np.sum(dY[:, i] * h))))
    for (j, i) in entries_gu:
        a, u = _r(rnd, Xo @ Wgo[j]), _r(rnd, Xo @ Wuo[j])
        da, du = swiglu_backward(dY @ Wd[:, j], a, u)
        res["dWs_g"].append(float(_r(rnd, np.sum(_r(rnd, da) * X[:, i]))))
        res["dWs_u"].append(float(_r(rnd, np.sum(_r(rnd, du) * X[:, i]))))
    return res


def expert_weight_grads(inp: dict, e: int, X: np.ndarray, gates: np.ndarray, dY_rows: np.ndarray,
                        rnd=None, fp8: bool = False, fold_gate: bool = False,
                        fp8_dgrad: bool = False) -> dict:
    """The whole weight gradients dW_g[e], dW_u[e], dW_d[e] of one expert.

    ``X`` holds the rows of the tokens routed to expert e in ascending token order, ``gates``
    their gates for e and ``dY_rows`` their upstream gradients. Only these rows enter expert
    e's weight gradients, so this is the whole layer's dW[e]: the combine's backward gives
    each row g * dY (``fold_gate``: the row keeps dY and the gate sits inside the expert),
    then the expert's own backward."""
    expert = swiglu_expert_fp8 if fp8 else swiglu_expert
    Wg, Wu, Wd = inp["W_g"][e], inp["W_u"][e], inp["W_d"][e]
    if fold_gate:
        a, u, h, _ = swiglu_expert(X, Wg, Wu, Wd, rnd, row_gate=gates)
        g = expert_backward(dY_rows, X, a, u, h, Wg, Wu, Wd, rnd, row_gate=gates)
    else:
        a, u, h, _ = expert(X, Wg, Wu, Wd, rnd)
        dy = _r(rnd, gates[:, None] * dY_rows)
        g = expert_backward(dy, X, a, u, h, Wg, Wu, Wd, rnd, fp8_dgrad=fp8_dgrad)
    return {"dW_g": g["dW_g"], "dW_u": g["dW_u"], "dW_d": g["dW_d"]}


def shared_weight_grad_units(inp: dict, dY: np.ndarray, units, rnd=None,
                             fp8: bool = False, fp8_dgrad: bool = False) -> dict:
    """Whole weight rows of chosen hidden units j of the shared expert (every token, weight
    1): dWs_g[j, :], dWs_u[j, :] (the units' input weights) and dWs_d[:, j] (their output
    weights). The units' a, u and h over all tokens need only their own weight rows:
    a = x W_g[units]^T, dh = dY W_d[:, units], then the SwiGLU derivative and the sums over
    tokens."""
    X = inp["x"]
    units = np.asarray(list(units), dtype=np.int64)
    Xo, Wgo, Wuo = _gemm_operands(X, inp["Ws_g"], inp["Ws_u"], fp8)
    av, uv = Xo @ Wgo[units].T, Xo @ Wuo[units].T
    a, u = _r(rnd, av), _r(rnd, uv)
    h = _r(rnd, silu(av) * uv)  # from the unrounded a and u, as the forward stores it
    if fp8_dgrad:  # the units' columns of the FP8 product (column scales are per column)
        dh = fp8_dequant_rows(dY) @ fp8_dequant_cols(inp["Ws_d"])[:, units]
    else:
        dh = dY @ inp["Ws_d"][:, units]
    da, du = swiglu_backward(dh, a, u)
    return {"dWs_g": _r(rnd, _r(rnd, da).T @ X), "dWs_u": _r(rnd, _r(rnd, du).T @ X),
            "dWs_d": _r(rnd, dY.T @ h)}
