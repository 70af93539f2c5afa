"""The oracle's pins have teeth: each plausible mistake planted in the oracle (a dropped
term, a wrong sign, a swapped operand, a wrong tie rule, a missing gate) makes at least one
pin of ``test_oracle_pins.py`` fail an assertion. CPU only.

Every mutant below is the oracle function with one deliberate error, installed with
monkeypatch for the length of one test; the whole pin suite then runs against it."""
import importlib.util
import itertools
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

_HERE = os.path.dirname(os.path.abspath(__file__))
_spec = importlib.util.spec_from_file_location("_oracle_pin_suite", os.path.join(_HERE, "test_oracle_pins.py"))
P = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(P)

# the unmutated functions, for mutants that wrap them
ORIG = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def _pin_cases():
    """Every pin of the suite with each of its parametrisations."""
    cases = []
    for name in sorted(dir(P)):
        fn = getattr(P, name)
        if not (name.startswith("test_") and callable(fn)):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = [s.strip() for s in mark.args[0].split(",")]
            rows = [v if len(names) > 1 else (v,) for v in mark.args[1]]
            grids.append([dict(zip(names, r)) for r in rows])
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            cases.append((name, fn, kw))
    return cases


PINS = _pin_cases()


def _failing_pins():
    """Pins whose checks reject the oracle as it stands. A pin that stops on some other
    error (a shape the mistake breaks) is not counted: a mistake must fail a check."""
    failed = []
    for name, fn, kw in PINS:
        try:
            fn(**kw)
        except AssertionError:
            failed.append(name)
        except Exception:  # noqa: BLE001
            pass
    return failed


# --------------------------------------------------------------------------------- mutants

def _silu_wrong_sign(z):
    return z / (1.0 + np.exp(z))


def _sigmoid_wrong_sign(z):
    return 1.0 / (1.0 + np.exp(z))


def _swiglu_bwd_drops_sigmoid_derivative(dh, a, u):
    sa = ORIG["sigmoid"](a)
    return dh * u * sa, dh * ORIG["silu"](a)


def _swiglu_bwd_du_without_a(dh, a, u):
    da, _ = ORIG["swiglu_backward"](dh, a, u)
    return da, dh * ORIG["sigmoid"](a)


def _route_sigmoid_unrenormalised(logits, b, k):
    r = ORIG["route_sigmoid"](logits, b, k)
    r["gate"] = r["score"].copy()
    return r


def _route_sigmoid_gate_from_biased_value(logits, b, k):
    r = ORIG["route_sigmoid"](logits, b, k)
    v = np.take_along_axis(r["select_value"], r["idx"], axis=1)
    r["gate"] = v / v.sum(axis=1, keepdims=True)
    return r


def _route_sigmoid_ignores_bias(logits, b, k):
    return ORIG["route_sigmoid"](logits, np.zeros_like(b), k)


def _router_logits_transposed_weight(x, W_r):
    return x @ W_r


def _top_k_ties_to_higher_index(score, k):
    T, E = score.shape
    index = np.broadcast_to(np.arange(E), (T, E))
    return np.lexsort((-index, -score), axis=-1)[:, :k]


def _route_softmax_renormalised(logits, k, z_coef):
    r = ORIG["route_softmax"](logits, k, z_coef)
    r["gate"] = r["gate"] / r["gate"].sum(axis=1, keepdims=True)
    r["score"] = r["gate"].copy()
    return r


def _route_softmax_z_of_mean_lse(logits, k, z_coef):
    r = ORIG["route_softmax"](logits, k, z_coef)
    r["z_loss"] = z_coef * float(np.mean(r["lse"]))
    return r


def _z_loss_square_of_mean(logits, k, z_coef):
    r = ORIG["route_softmax"](logits, k, z_coef)
    r["z_loss"] = z_coef * float(np.mean(r["lse"])) ** 2
    return r


def _router_bwd(dg, rr, x, W_r, mode, z_coef, T_norm=None, dl_extra=None, *, couple=True,
                zfac=2.0):
    """The router backward restated with two knobs that plant a mistake."""
    idx, gate = rr["idx"], rr["gate"]
    T, k = idx.shape
    T_norm = T if T_norm is None else T_norm
    dl = np.zeros((T, W_r.shape[0]))
    rows = np.arange(T)
    if mode == O.SIGMOID:
        s = rr["score"]
        S = s.sum(axis=1, keepdims=True)
        ds = (dg - (gate * dg).sum(axis=1, keepdims=True) * couple) / S
        for i in range(k):
            dl[rows, idx[:, i]] += ds[:, i] * s[:, i] * (1.0 - s[:, i])
    else:
        p, lse = rr["p"], rr["lse"]
        sel = np.zeros_like(p)
        for i in range(k):
            sel[rows, idx[:, i]] = dg[:, i]
        dl = p * (sel - (gate * dg).sum(axis=1, keepdims=True)) + (zfac * z_coef / T_norm) * lse[:, None] * p
    if dl_extra is not None:
        dl = dl + dl_extra
    return {"dlogits": dl, "dW_r": dl.T @ x, "dx_r": dl @ W_r}


def _router_bwd_without_renormalisation_term(*a, **kw):
    return _router_bwd(*a, couple=False, **kw)


def _router_bwd_z_gradient_missing_factor_two(*a, **kw):
    return _router_bwd(*a, zfac=1.0, **kw)


def _dispatch_rows_by_slot(idx, E):
    T, k = idx.shape
    D = ORIG["dispatch"](idx, E)
    tok = np.repeat(np.arange(T), k)
    slot = np.tile(np.arange(k), T)
    order = np.lexsort((slot, idx.reshape(-1)))  # expert, then slot: not token order
    D["perm_token"], D["perm_slot"] = tok[order], slot[order]
    D["slot_to_row"][D["perm_token"], D["perm_slot"]] = np.arange(T * k)
    return D


def _combine_drops_shared(Y_perm, gate, slot_to_row, Y_shared, rnd=None):
    return ORIG["combine"](Y_perm, gate, slot_to_row, None, rnd)


def _combine_bwd_without_gate(dY, Y_perm, gate, slot_to_row, perm_token, perm_slot, rnd=None):
    _, dg = ORIG["combine_backward"](dY, Y_perm, gate, slot_to_row, perm_token, perm_slot, rnd)
    return dY[perm_token], dg


def _expert_bwd_swaps_weight_grads(*a, **kw):
    r = ORIG["expert_backward"](*a, **kw)
    r["dW_g"], r["dW_u"] = r["dW_u"], r["dW_g"]
    return r


def _expert_bwd_folded_gate_grad_from_dh(*a, **kw):
    r = ORIG["expert_backward"](*a, **kw)
    if kw.get("row_gate") is not None:
        r["dg_row"] = r["dg_row"] * kw["row_gate"]
    return r


def _swiglu_expert_gate_squared(rows, W_g, W_u, W_d, rnd=None, row_gate=None):
    return ORIG["swiglu_expert"](rows, W_g, W_u, W_d, rnd,
                                 row_gate=None if row_gate is None else row_gate ** 2)


def _input_gradient_drops_router(dX_perm, slot_to_row, dx_shared, dx_router, rnd=None):
    return ORIG["input_gradient"](dX_perm, slot_to_row, dx_shared, None, rnd)


def _bias_update_wrong_sign(counts, b, T, k, gamma):
    return ORIG["bias_update"](counts, b, T, k, -gamma)


def _bias_update_proportional_over_load(counts, b, T, k, gamma):
    E = b.shape[0]
    mean = np.float64(T) * k / E
    c = np.maximum(counts.astype(np.float64), 1.0)
    step = (np.float32(gamma) * ((mean - c) / c).astype(np.float32)).astype(np.float32)
    return (np.asarray(b, dtype=np.float32) + step).astype(np.float32)


def _aux_switch_without_E(logits, idx, mode, seq_len, switch_coef, seq_coef):
    a = ORIG["aux_losses"](logits, idx, mode, seq_len, switch_coef, seq_coef)
    a["switch_unscaled"] /= logits.shape[1]
    a["switch"] = switch_coef * a["switch_unscaled"]
    return a


def _aux_seq_from_batch_counts(logits, idx, mode, seq_len, switch_coef, seq_coef):
    a = ORIG["aux_losses"](logits, idx, mode, seq_len, switch_coef, seq_coef)
    T, E = logits.shape
    B = T // seq_len
    f_batch = E * a["f"]  # E c_e / (T k): the batch's counts in place of each sequence's
    Ps = a["pi"].reshape(B, seq_len, E).mean(axis=1)
    a["seq_unscaled"] = float(np.mean(np.sum(f_batch[None, :] * Ps, axis=1)))
    a["seq"] = seq_coef * a["seq_unscaled"]
    a["f_seq"] = np.broadcast_to(f_batch, (B, E)).copy()
    return a


def _aux_bwd_drops_sequence_term(logits, idx, mode, seq_len, switch_coef, seq_coef):
    return ORIG["aux_losses_backward"](logits, idx, mode, seq_len, switch_coef, 0.0)


def _e4m3_truncates(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -5)
    q = np.ldexp(np.trunc(np.ldexp(x, 4 - e)), e - 4)
    return np.clip(q, -O.E4M3_MAX, O.E4M3_MAX)


def _bf16_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    m = np.ldexp(x, 8 - e)
    return np.ldexp(np.sign(m) * np.floor(np.abs(m) + 0.5), e - 8)


def _quantize_rows_to_240(X):
    X32 = np.asarray(X, dtype=np.float32)
    amax = np.abs(X32).max(axis=1)
    scale = np.where(amax > 0, (amax / np.float32(240.0)).astype(np.float32), np.float32(1.0))
    return O.e4m3_round((X32 / scale[:, None]).astype(np.float32)), scale.astype(np.float64)


def _fp8_expert(rows, W_g, W_u, W_d, rnd=None, *, weights_by_column=False, x_by_column=False,
                requantise_h=True):
    """The FP8 expert restated with knobs that plant a mistake."""
    deq = ORIG["fp8_dequant_rows"]
    wq = (lambda W: deq(W.T).T) if weights_by_column else deq
    xq = deq(rows.T).T if x_by_column else deq(rows)
    a = xq @ wq(W_g).T
    u = xq @ wq(W_u).T
    h = O._r(rnd, ORIG["silu"](a) * u)
    y = O._r(rnd, (deq(h) if requantise_h else h) @ wq(W_d).T)
    return O._r(rnd, a), O._r(rnd, u), h, y


def _fp8_weights_by_column(*a, **kw):
    return _fp8_expert(*a, weights_by_column=True, **kw)


def _fp8_x_by_column(*a, **kw):
    return _fp8_expert(*a, x_by_column=True, **kw)


def _fp8_h_not_requantised(*a, **kw):
    return _fp8_expert(*a, requantise_h=False, **kw)


def _gemm_operands_unquantised(X, Wg, Wu, fp8):
    return X, Wg, Wu


def _near_tie_ignores_next_value(select_value, k, gap=1e-6):
    srt = -np.sort(-select_value, axis=1)[:, :k]
    if k < 2:
        return np.zeros(select_value.shape[0], dtype=bool)
    return (np.abs(np.diff(srt, axis=1)) < gap).any(axis=1)


def _token_forward_ungated(inp, t, experts, gates, rnd=None, fp8=False, fold_gate=False):
    return ORIG["token_forward"](inp, t, experts, np.ones(len(gates)), rnd, fp8, fold_gate)


def _token_backward_without_shared(inp, *a, **kw):
    return ORIG["token_backward"]({n: v for n, v in inp.items() if not n.startswith("Ws_")}, *a, **kw)


def _weight_grad_entries_ungated(inp, e, tokens, slots_gate, *a, **kw):
    return ORIG["expert_weight_grad_entries"](inp, e, tokens, np.ones_like(slots_gate), *a, **kw)


def _regate_unrenormalised(r, logits, idx, mode, b, z_coef):
    r = ORIG["_regate"](r, logits, idx, mode, b, z_coef)
    if mode == O.SIGMOID:
        r["gate"] = r["score"].copy()
    return r


def _expert_weight_grads_ungated(inp, e, X, gates, *a, **kw):
    return ORIG["expert_weight_grads"](inp, e, X, np.ones_like(gates), *a, **kw)


def _shared_units_dh_from_transposed_weight(inp, dY, units, rnd=None, fp8=False, fp8_dgrad=False):
    wd = inp["Ws_d"]
    if wd.shape[0] != wd.shape[1]:
        wd = np.resize(wd.T, wd.shape)
    return ORIG["shared_weight_grad_units"](dict(inp, Ws_d=wd), dY, units, rnd, fp8, fp8_dgrad)


def _layer_backward_subset_ignores_batch_count(inp, fwd, dY, T_norm=None, dl_extra=None,
                                               weight_grads=True):
    return ORIG["layer_backward"](inp, fwd, dY, None, dl_extra, weight_grads)


def _dgrad_dh_weights_by_row(dy, W_d):
    return O.fp8_dequant_rows(dy) @ O.fp8_dequant_rows(W_d)


def _dgrad_dh_dy_by_column(dy, W_d):
    return O.fp8_dequant_cols(dy) @ O.fp8_dequant_cols(W_d)


def _dgrad_dx_separate_scales(da, du, W_g, W_u):
    return (O.fp8_dequant_rows(da) @ O.fp8_dequant_cols(W_g) +
            O.fp8_dequant_rows(du) @ O.fp8_dequant_cols(W_u))


def _expert_bwd_fp8_dgrad_ignored(*a, fp8_dgrad=False, **kw):
    return ORIG["expert_backward"](*a, **kw)


def _slot_router_terms_without_dlogits(dlogits, idx, W_r):
    return W_r[idx] * 0.1


MUTANTS = {
    "silu with sigmoid(-z)": ("silu", _silu_wrong_sign),
    "router term in the rows without the logit gradient": ("slot_router_terms", _slot_router_terms_without_dlogits),
    "sigmoid with the wrong sign": ("sigmoid", _sigmoid_wrong_sign),
    "SwiGLU backward drops silu's product-rule term": ("swiglu_backward", _swiglu_bwd_drops_sigmoid_derivative),
    "SwiGLU backward du misses the factor a": ("swiglu_backward", _swiglu_bwd_du_without_a),
    "sigmoid gates not renormalised": ("route_sigmoid", _route_sigmoid_unrenormalised),
    "sigmoid gates taken from the biased value": ("route_sigmoid", _route_sigmoid_gate_from_biased_value),
    "selection ignores the bias": ("route_sigmoid", _route_sigmoid_ignores_bias),
    "router logits from the transposed weight": ("router_logits", _router_logits_transposed_weight),
    "ties go to the higher index": ("_top_k_desc", _top_k_ties_to_higher_index),
    "softmax gates renormalised": ("route_softmax", _route_softmax_renormalised),
    "z-loss of mean lse instead of mean lse^2": ("route_softmax", _route_softmax_z_of_mean_lse),
    "z-loss as the square of the mean lse": ("route_softmax", _z_loss_square_of_mean),
    "router backward drops the renormalisation term": ("router_backward", _router_bwd_without_renormalisation_term),
    "z-loss gradient missing its factor 2": ("router_backward", _router_bwd_z_gradient_missing_factor_two),
    "rows within an expert ordered by slot": ("dispatch", _dispatch_rows_by_slot),
    "combine drops the shared expert": ("combine", _combine_drops_shared),
    "combine backward forgets the gate": ("combine_backward", _combine_bwd_without_gate),
    "dW_g and dW_u swapped": ("expert_backward", _expert_bwd_swaps_weight_grads),
    "folded gate gradient taken from dh": ("expert_backward", _expert_bwd_folded_gate_grad_from_dh),
    "folded gate applied twice": ("swiglu_expert", _swiglu_expert_gate_squared),
    "input gradient drops the router term": ("input_gradient", _input_gradient_drops_router),
    "bias update with the wrong sign": ("bias_update", _bias_update_wrong_sign),
    "proportional update relative to the load": ("bias_update_proportional", _bias_update_proportional_over_load),
    "Switch loss without the factor E": ("aux_losses", _aux_switch_without_E),
    "balancing-loss gradient drops the sequence term": ("aux_losses_backward", _aux_bwd_drops_sequence_term),
    "sequence loss from the batch-wide counts": ("aux_losses", _aux_seq_from_batch_counts),
    "E4M3 rounding truncates": ("e4m3_round", _e4m3_truncates),
    "bf16 rounding ties away from zero": ("bf16_round", _bf16_ties_away),
    "FP8 rows scaled to 240": ("quantize_rows_fp8", _quantize_rows_to_240),
    "FP8 weights scaled per input column": ("swiglu_expert_fp8", _fp8_weights_by_column),
    "FP8 activations scaled per feature": ("swiglu_expert_fp8", _fp8_x_by_column),
    "FP8 h not re-quantised before the down projection": ("swiglu_expert_fp8", _fp8_h_not_requantised),
    "near-tie check ignores the (k+1)-th value": ("near_tie_tokens", _near_tie_ignores_next_value),
    "sampled forward ignores the gates": ("token_forward", _token_forward_ungated),
    "sampled backward omits the shared expert": ("token_backward", _token_backward_without_shared),
    "sampled weight gradients ignore the gates": ("expert_weight_grad_entries", _weight_grad_entries_ungated),
    "sampled FP8 weight gradients from unquantised operands": ("_gemm_operands", _gemm_operands_unquantised),
    "replayed sigmoid gates not renormalised": ("_regate", _regate_unrenormalised),
    "whole expert weight gradients ignore the gates": ("expert_weight_grads", _expert_weight_grads_ungated),
    "shared-unit gradients through the wrong output weights": ("shared_weight_grad_units", _shared_units_dh_from_transposed_weight),
    "token-subset backward normalises the z-loss by the subset": ("layer_backward", _layer_backward_subset_ignores_batch_count),
    "FP8 dgrad: W_d scaled per row instead of per column": ("fp8_dgrad_dh", _dgrad_dh_weights_by_row),
    "FP8 dgrad: dy scaled per column instead of per row": ("fp8_dgrad_dh", _dgrad_dh_dy_by_column),
    "FP8 dgrad: da and du scaled separately": ("fp8_dgrad_dx", _dgrad_dx_separate_scales),
    "FP8 dgrad switch ignored by the expert backward": ("expert_backward", _expert_bwd_fp8_dgrad_ignored),
}


def test_the_unmutated_oracle_passes_every_pin():
    assert len(PINS) > 40
    assert _failing_pins() == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_a_planted_mistake_fails_a_pin(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(O, name, fn)
    assert _failing_pins(), f"no pin catches: {mutant}"
