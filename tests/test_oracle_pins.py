"""The fp64 oracle pinned to facts outside itself: brute force on tiny inputs, closed forms
worked by hand, invariants of the method, finite differences and the pages' own
parameter arithmetic. CPU only."""
import json
import math
import os
import struct

import numpy as np
import pytest

from oracle import moe_oracle as O
from pretraining_sigmoid_softmax_gb300.configs import MoEConfig

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as fh:
        return json.load(fh)


def _tiny_inputs(rng, T, d, E, f, fs=0, b_scale=0.05):
    inp = {
        "x": rng.standard_normal((T, d)),
        "W_r": rng.standard_normal((E, d)) / math.sqrt(d),
        "b": rng.uniform(-b_scale, b_scale, E),
        "W_g": rng.standard_normal((E, f, d)) / math.sqrt(d),
        "W_u": rng.standard_normal((E, f, d)) / math.sqrt(d),
        "W_d": rng.standard_normal((E, d, f)) / math.sqrt(f),
    }
    if fs:
        inp["Ws_g"] = rng.standard_normal((fs, d)) / math.sqrt(d)
        inp["Ws_u"] = rng.standard_normal((fs, d)) / math.sqrt(d)
        inp["Ws_d"] = rng.standard_normal((d, fs)) / math.sqrt(fs)
    return inp


# ------------------------------------------------------------------------- router logits

def test_router_logits_of_basis_tokens_are_columns_of_the_router_weight():
    """Token t = the t-th unit vector picks out column t of W_r: l[t, e] = W_r[e, t]. A square
    shape (T = d = E) lets a transposed operand through the shapes, so the values catch it;
    a scaled basis vector scales its logits exactly (dyadic values)."""
    rng = np.random.default_rng(2)
    n = 5
    W_r = rng.integers(-8, 9, size=(n, n)) / 8.0
    np.testing.assert_array_equal(O.router_logits(np.eye(n), W_r), W_r.T)
    x = np.diag([1.0, -2.0, 0.5, 0.0, 4.0])
    np.testing.assert_array_equal(O.router_logits(x, W_r), np.diag(x)[:, None] * W_r.T)


# ----------------------------------------------------------------------------- selection

@pytest.mark.parametrize("k", [1, 2, 3, 5, 8])
def test_selection_matches_subset_enumeration_with_exact_ties(k):
    """Dyadic logits (exact sums) with many exact ties: the softmax router's choice equals
    the k-subset of largest total, lexicographically smallest among equal totals."""
    rng = np.random.default_rng(10 + k)
    E = 8
    logits = rng.integers(-3, 4, size=(64, E)).astype(np.float64) / 4.0
    r = O.route_softmax(logits, k, 0.0)
    for t in range(64):
        assert tuple(r["idx"][t]) == O.select_brute_force(logits[t], k)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_sigmoid_selection_uses_bias_and_breaks_ties_low(k):
    """Zero logits make every sigmoid score exactly 0.5, so the dyadic bias alone decides
    (with exact ties); the chosen set is the subset enumeration's."""
    rng = np.random.default_rng(20 + k)
    E = 8
    logits = np.zeros((32, E))
    for t in range(32):
        b = rng.integers(-2, 3, size=E).astype(np.float64) / 64.0
        r = O.route_sigmoid(logits[t:t + 1], b, k)
        assert tuple(r["idx"][0]) == O.select_brute_force(0.5 + b, k)
        np.testing.assert_allclose(r["gate"][0], np.full(k, 1.0 / k), rtol=0, atol=1e-15)


def test_sigmoid_selection_random_against_enumeration():
    rng = np.random.default_rng(3)
    E, k = 8, 3
    logits = rng.standard_normal((64, E))
    b = rng.uniform(-0.05, 0.05, E)
    r = O.route_sigmoid(logits, b, k)
    v = 1.0 / (1.0 + np.exp(-logits)) + b
    for t in range(64):
        assert tuple(r["idx"][t]) == O.select_brute_force(v[t], k)
    # invariants: k distinct experts, gates sum to 1 and are proportional to the chosen
    # experts' own sigmoid scores (not to the biased selection values)
    assert all(len(set(row)) == k for row in r["idx"].tolist())
    np.testing.assert_allclose(r["gate"].sum(axis=1), 1.0, rtol=1e-15)
    s = np.take_along_axis(1.0 / (1.0 + np.exp(-logits)), r["idx"], axis=1)
    np.testing.assert_allclose(r["gate"] * s.sum(axis=1, keepdims=True), s, rtol=1e-14)


def test_bias_steers_selection_but_not_gates():
    """A large bias forces an expert in; its gate is still its own renormalised score."""
    logits = np.array([[2.0, 1.0, 0.0, -1.0]])
    b = np.array([0.0, 0.0, 0.0, 10.0])
    r = O.route_sigmoid(logits, b, 2)
    assert list(r["idx"][0]) == [3, 0]
    s = [1 / (1 + math.exp(1.0)), 1 / (1 + math.exp(-2.0))]
    np.testing.assert_allclose(r["gate"][0], [s[0] / (s[0] + s[1]), s[1] / (s[0] + s[1])], rtol=1e-15)


@pytest.mark.parametrize("mode", ["sigmoid", "softmax"])
def test_all_equal_logits(mode):
    E, k = 8, 3
    logits = np.full((5, E), 0.7)
    r = O.route(logits, mode, k, np.zeros(E), 0.0)
    assert (r["idx"] == np.arange(k)).all()
    want = 1.0 / k if mode == "sigmoid" else 1.0 / E
    np.testing.assert_allclose(r["gate"], want, rtol=1e-15)


def test_z_loss_closed_form_at_zero_logits():
    g = _gold("closed_forms.json")["z_loss_uniform"]
    r = O.route_softmax(np.zeros((7, g["E"])), 2, g["coef"])
    assert r["z_loss"] == pytest.approx(g["z"], rel=1e-14)
    np.testing.assert_allclose(r["lse"], math.log(g["E"]), rtol=1e-15)


def test_z_loss_is_the_mean_of_squares_not_the_square_of_the_mean():
    """Worked by hand: logits (0, 0) give lse = ln 2 and (ln 3, 0) give lse = ln 4, so
    mean(lse^2) = 2.5 ln^2 2, while the square of the mean would be 2.25 ln^2 2."""
    r = O.route_softmax(np.array([[0.0, 0.0], [math.log(3.0), 0.0]]), 1, 1.0)
    np.testing.assert_allclose(r["lse"], [math.log(2.0), math.log(4.0)], rtol=1e-15)
    assert r["z_loss"] == pytest.approx(2.5 * math.log(2.0) ** 2, rel=1e-14)


def test_softmax_gates_are_unrenormalised_probabilities():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((16, 6))
    r = O.route_softmax(logits, 2, 0.0)
    np.testing.assert_allclose(r["p"].sum(1), 1.0, rtol=1e-14)
    assert (r["gate"].sum(1) < 1.0).all()
    # the chosen probabilities are the two largest probabilities
    top2 = -np.sort(-r["p"], axis=1)[:, :2]
    np.testing.assert_allclose(r["gate"], top2, rtol=0, atol=0)


def test_k_equals_E_chooses_everything():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((9, 5))
    r = O.route_sigmoid(logits, np.zeros(5), 5)
    assert (np.sort(r["idx"], 1) == np.arange(5)).all()
    s = 1 / (1 + np.exp(-logits))
    np.testing.assert_allclose(np.sort(r["gate"], 1), np.sort(s / s.sum(1, keepdims=True), 1), rtol=1e-14)


def test_near_tie_detector():
    """k = 2: a near tie inside the top k, or between the k-th and the (k+1)-th value, puts
    the choice in doubt; one below the (k+1)-th value does not."""
    v = np.array([[0.9, 0.9 + 5e-7, 0.1, 0.0],
                  [0.9, 0.8, 0.7, 0.6],
                  [0.9, 0.5 + 5e-7, 0.5, 0.0],
                  [0.9, 0.8, 0.7, 0.7 + 1e-9]])
    assert list(O.near_tie_tokens(v, 2)) == [True, False, True, False]


# ------------------------------------------------------------------------------ dispatch

def test_dispatch_invariants_and_round_trip():
    rng = np.random.default_rng(6)
    T, E, k, d = 200, 13, 4, 7
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    D = O.dispatch(idx, E)
    assert D["counts"].sum() == T * k
    assert (np.diff(D["offsets"]) >= 0).all() and D["offsets"][-1] == T * k
    # rows sorted by (expert, token), strictly
    e_of_row = idx[D["perm_token"], D["perm_slot"]]
    key = e_of_row * T + D["perm_token"]
    assert (np.diff(key) > 0).all()
    for e in range(E):
        assert (e_of_row[D["offsets"][e]:D["offsets"][e + 1]] == e).all()
    # slot_to_row is a bijection onto the rows
    assert sorted(D["slot_to_row"].reshape(-1).tolist()) == list(range(T * k))
    x = rng.standard_normal((T, d))
    x_perm = x[D["perm_token"]]
    for i in range(k):
        assert (x_perm[D["slot_to_row"][:, i]] == x).all()


def test_dispatch_empty_experts():
    idx = np.array([[0, 3], [3, 0], [0, 3]])
    D = O.dispatch(idx, 5)
    assert D["counts"].tolist() == [3, 0, 0, 3, 0]
    assert D["offsets"].tolist() == [0, 3, 3, 3, 6, 6]
    assert D["perm_token"].tolist() == [0, 1, 2, 0, 1, 2]


# ------------------------------------------------------------------- experts and combine

def test_swiglu_scalar_closed_form():
    g = _gold("closed_forms.json")["swiglu_scalar"]
    a, u, h, y = O.swiglu_expert(np.array([[g["x"]]]), np.array([[g["w_gate"]]]),
                                 np.array([[g["w_up"]]]), np.array([[g["w_down"]]]))
    assert a[0, 0] == g["a"] and u[0, 0] == g["u"]
    assert h[0, 0] == pytest.approx(g["h"], rel=1e-15)
    assert y[0, 0] == pytest.approx(g["y"], rel=1e-15)


@pytest.mark.parametrize("mode,fs", [("sigmoid", 0), ("sigmoid", 6), ("softmax", 0)])
def test_permuted_layer_equals_dense_masked_brute_force(mode, fs):
    rng = np.random.default_rng(7)
    inp = _tiny_inputs(rng, T=40, d=12, E=6, f=5, fs=fs)
    fwd = O.layer_forward(inp, mode, 3, 1e-3)
    ref = O.layer_forward_dense_masked(inp, mode, 3, 1e-3)
    np.testing.assert_allclose(fwd["out"], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["sigmoid", "softmax"])
def test_single_expert_top1_is_the_dense_ffn(mode):
    """One expert with top-1 routing is the dense SwiGLU FFN it replaces, and the router
    weight gets exactly zero gradient (handbook summary, section 2.5)."""
    rng = np.random.default_rng(8)
    inp = _tiny_inputs(rng, T=11, d=6, E=1, f=4)
    fwd = O.layer_forward(inp, mode, 1, 0.0)
    assert (fwd["gate"] == 1.0).all()
    dense = O.swiglu_expert(inp["x"], inp["W_g"][0], inp["W_u"][0], inp["W_d"][0])[3]
    np.testing.assert_array_equal(fwd["out"], dense)
    dY = rng.standard_normal(fwd["out"].shape)
    bwd = O.layer_backward(inp, fwd, dY)
    assert (bwd["dW_r"] == 0.0).all()
    assert (bwd["dlogits"] == 0.0).all()


def test_gemm_flop_accounting_reproduces_the_pages_parameter_counts():
    """A SwiGLU expert holds 3*d*f parameters, so the eight chosen experts equal the
    dense layer they replace and the printed model totals follow."""
    g = _gold("param_counts.json")
    d, f, E, k, L = g["hidden"], g["expert_width"], g["experts"], g["top_k"], g["layers"]
    cfg = MoEConfig("pin", T=1, d=d, E=E, k=k, f=f, f_shared=0, mode="sigmoid", seed=0,
                    backward=False, bias_update=False)
    per_expert = cfg.gemm_flops() / (2.0 * cfg.N)  # FLOPs per routed row / 2 = params per expert
    assert per_expert == 3 * d * f == 6_291_456
    assert k * per_expert == 3 * d * g["dense_ffn_width"]
    router = E * d
    dense_total = g["dense_total_params_printed_B"] * 1e9
    moe_total = dense_total + L * (E * per_expert - 3 * d * g["dense_ffn_width"] + router)
    moe_active = dense_total + L * router
    assert round(moe_total / 1e9, 2) == g["moe_total_params_printed_B"]
    assert round(moe_active / 1e9, 3) == g["moe_active_params_printed_B"]
    assert L * 1 * d == g["zero_grad_params_single_expert_printed"] - 2


# ---------------------------------------------------------------------------- bias update

def test_bias_update_worked_example():
    g = _gold("closed_forms.json")["bias_update_example"]
    nb = O.bias_update(np.array(g["counts"]), np.array(g["b_before"], np.float32), g["T"], g["k"], g["gamma"])
    got = [hex(struct.unpack("<I", struct.pack("<f", float(v)))[0]) for v in nb]
    assert got == g["b_after_fp32_hex"]


def test_bias_update_invariants():
    rng = np.random.default_rng(9)
    E, T, k = 16, 100, 4
    b = rng.uniform(-0.05, 0.05, E).astype(np.float32)
    counts = rng.multinomial(T * k, np.ones(E) / E)
    nb = O.bias_update(counts, b, T, k, 0.001)
    mean = T * k / E
    delta = nb.astype(np.float64) - b
    for e in range(E):
        if counts[e] == mean:
            assert delta[e] == 0
        else:
            assert np.sign(delta[e]) == np.sign(mean - counts[e])
            assert abs(abs(delta[e]) - 0.001) < 1e-8
    balanced = O.bias_update(np.full(E, T * k // E), b, T, k, 0.001)
    np.testing.assert_array_equal(balanced, b)


# ----------------------------------------------------------------------- finite differences

def _fd_case(mode, seed):
    """Tiny inputs whose selections sit at least 1e-3 away from a tie."""
    rng = np.random.default_rng(seed)
    while True:
        inp = _tiny_inputs(rng, T=6, d=5, E=5, f=3, fs=2)
        lg = O.router_logits(inp["x"], inp["W_r"])
        r = O.route(lg, mode, 2, inp["b"], 0.1)
        if not O.near_tie_tokens(r["select_value"], 2, gap=1e-3).any():
            return inp, rng


@pytest.mark.parametrize("mode,aux", [("sigmoid", None), ("softmax", None),
                                      ("sigmoid", (3, 0.2, 0.3)), ("softmax", (2, 0.4, 0.1))])
def test_backward_matches_central_finite_differences(mode, aux):
    inp, rng = _fd_case(mode, 11 if mode == "sigmoid" else 12)
    z = 0.1 if mode == "softmax" else 0.0
    dY = rng.standard_normal((6, 5))
    fwd = O.layer_forward(inp, mode, 2, z, aux=aux)
    bwd = O.layer_backward(inp, fwd, dY)
    names = {"x": "dx", "W_r": "dW_r", "W_g": "dW_g", "W_u": "dW_u", "W_d": "dW_d",
             "Ws_g": "dWs_g", "Ws_u": "dWs_u", "Ws_d": "dWs_d"}
    h = 1e-6
    for p, gname in names.items():
        arr = inp[p]
        num = np.zeros_like(arr)
        for ix in np.ndindex(arr.shape):
            old = arr[ix]
            arr[ix] = old + h
            lp = O.loss(O.layer_forward(inp, mode, 2, z, aux=aux), dY)
            arr[ix] = old - h
            lm = O.loss(O.layer_forward(inp, mode, 2, z, aux=aux), dY)
            arr[ix] = old
            num[ix] = (lp - lm) / (2 * h)
        ana = bwd[gname]
        scale = max(1.0, np.abs(num).max())
        assert np.abs(ana - num).max() / scale < 1e-6, p


@pytest.mark.parametrize("fs", [0, 4])
def test_router_term_in_the_expert_rows_is_the_same_layer(fs):
    """Sigmoid routing without balancing losses: a token's logit gradient is zero off its
    chosen experts, so adding dl[t, e] W_r[e] to the expert row of each chosen slot (t, e),
    instead of forming dl W_r as a separate summand, gives the same input gradient in exact
    arithmetic, and with bf16 storage the same up to the rounding of the rows; every other
    gradient is untouched. The option is refused where the logit gradient is dense."""
    rng = np.random.default_rng(37)
    inp = _tiny_inputs(rng, T=40, d=8, E=6, f=6, fs=fs)
    dY = rng.standard_normal((40, 8))
    f0 = O.layer_forward(inp, "sigmoid", 3)
    f1 = O.layer_forward(inp, "sigmoid", 3, router_rows=True)
    b0, b1 = O.layer_backward(inp, f0, dY), O.layer_backward(inp, f1, dY)
    np.testing.assert_allclose(b1["dx"], b0["dx"], rtol=1e-12, atol=1e-13)
    for name in ("dg", "dlogits", "dW_r", "dW_g", "dW_u", "dW_d"):
        np.testing.assert_array_equal(b1[name], b0[name], err_msg=name)
    # the rows really carry the term: their difference is the router term of their slots
    s2r, idx = f1["slot_to_row"], f1["idx"]
    for i in range(3):
        diff = b1["dX_perm"][s2r[:, i]] - b0["dX_perm"][s2r[:, i]]
        want = b0["dlogits"][np.arange(40), idx[:, i]][:, None] * inp["W_r"][idx[:, i]]
        np.testing.assert_allclose(diff, want, rtol=1e-10, atol=1e-13)
    assert np.abs(b0["dx_r"]).max() > 1e-3  # the term is not negligible here
    # with bf16 storage: within the rounding of k + 1 rows of the token sum
    s0 = O.layer_forward(inp, "sigmoid", 3, rnd=O.bf16_round, fold_gate=True)
    s1 = O.layer_forward(inp, "sigmoid", 3, rnd=O.bf16_round, fold_gate=True, router_rows=True)
    c0, c1 = O.layer_backward(inp, s0, dY), O.layer_backward(inp, s1, dY)
    bound = 6 * 2.0 ** -8 * (np.abs(b0["dx"]) + 3 * np.abs(b0["dX_perm"]).max())
    assert (np.abs(c1["dx"] - c0["dx"]) <= bound).all()
    with pytest.raises(ValueError):
        O.layer_forward(inp, "softmax", 3, router_rows=True)
    with pytest.raises(ValueError):
        O.layer_forward(inp, "sigmoid", 3, aux=(20, 0.01, 0.01), router_rows=True)


@pytest.mark.parametrize("mode,fs,aux", [("sigmoid", 0, None), ("sigmoid", 4, (5, 0.2, 0.3)),
                                         ("softmax", 0, None)])
def test_gate_folded_into_experts_is_the_same_layer(mode, fs, aux):
    """Applying each slot's gate inside its expert (g * h before the linear down projection)
    and combining without weights is the same layer in exact arithmetic: outputs, every
    gradient and the gate gradient (sum_j (dy W_d)_j h_j) agree with the plain layer."""
    rng = np.random.default_rng(31)
    inp = _tiny_inputs(rng, T=30, d=8, E=5, f=6, fs=fs)
    z = 0.05 if mode == "softmax" else 0.0
    dY = rng.standard_normal((30, 8))
    f0 = O.layer_forward(inp, mode, 2, z, aux=aux)
    f1 = O.layer_forward(inp, mode, 2, z, aux=aux, fold_gate=True)
    np.testing.assert_allclose(f1["out"], f0["out"], rtol=1e-12, atol=1e-13)
    assert not np.allclose(f1["H"], f0["H"])  # the stored h really carries the gate
    b0 = O.layer_backward(inp, f0, dY)
    b1 = O.layer_backward(inp, f1, dY)
    for name in ("dg", "dx", "dW_r", "dW_g", "dW_u", "dW_d", "dlogits"):
        np.testing.assert_allclose(b1[name], b0[name], rtol=1e-11, atol=1e-12, err_msg=name)
    # the per-token and per-entry forms used at large sizes, folded, give the same values
    for t in (0, 17):
        o = O.token_forward(inp, t, f1["idx"][t], f1["gate"][t], fold_gate=True)
        np.testing.assert_allclose(o, f0["out"][t], rtol=1e-12, atol=1e-13)
        if aux is None:
            tb = O.token_backward(inp, t, f1["logits"][t], f1["idx"][t], mode, 2, dY[t], z, 30,
                                  fold_gate=True)
            np.testing.assert_allclose(tb["dx"], b0["dx"][t], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(tb["dg"], b0["dg"][t], rtol=1e-11, atol=1e-12)
    e = int(np.argmax(np.diff(f1["offsets"])))
    rows = np.arange(f1["offsets"][e], f1["offsets"][e + 1])
    tok, sl = f1["perm_token"][rows], f1["perm_slot"][rows]
    ed, eg = [(1, 2), (7, 5)], [(3, 4), (0, 7)]
    w0 = O.expert_weight_grad_entries(inp, e, tok, f1["gate"][tok, sl], dY, ed, eg)
    w1 = O.expert_weight_grad_entries(inp, e, tok, f1["gate"][tok, sl], dY, ed, eg, fold_gate=True)
    for name in ("dW_d", "dW_g", "dW_u"):
        np.testing.assert_allclose(w1[name], w0[name], rtol=1e-11, atol=1e-13)


def test_sampled_rows_equal_full_layer():
    """The per-token and per-entry evaluations used at large sizes agree with the whole
    layer."""
    rng = np.random.default_rng(13)
    for mode, z in (("sigmoid", 0.0), ("softmax", 0.05)):
        inp = _tiny_inputs(rng, T=30, d=8, E=5, f=4, fs=3 if mode == "sigmoid" else 0)
        dY = rng.standard_normal((30, 8))
        fwd = O.layer_forward(inp, mode, 2, z)
        bwd = O.layer_backward(inp, fwd, dY)
        for t in (0, 7, 29):
            o = O.token_forward(inp, t, fwd["idx"][t], fwd["gate"][t])
            np.testing.assert_allclose(o, fwd["out"][t], rtol=1e-12, atol=1e-12)
            tb = O.token_backward(inp, t, fwd["logits"][t], fwd["idx"][t], mode, 2, dY[t], z, 30)
            np.testing.assert_allclose(tb["dx"], bwd["dx"][t], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(tb["dg"], bwd["dg"][t], rtol=1e-12, atol=1e-12)
        for e in range(5):
            rows = np.arange(fwd["offsets"][e], fwd["offsets"][e + 1])
            toks = fwd["perm_token"][rows]
            gates = fwd["gate"][toks, fwd["perm_slot"][rows]]
            ent = O.expert_weight_grad_entries(inp, e, toks, gates, dY, [(0, 1), (7, 3)], [(2, 5), (0, 0)])
            np.testing.assert_allclose(ent["dW_d"], [bwd["dW_d"][e][0, 1], bwd["dW_d"][e][7, 3]], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(ent["dW_g"], [bwd["dW_g"][e][2, 5], bwd["dW_g"][e][0, 0]], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(ent["dW_u"], [bwd["dW_u"][e][2, 5], bwd["dW_u"][e][0, 0]], rtol=1e-11, atol=1e-13)
        if mode == "sigmoid":
            ent = O.shared_weight_grad_entries(inp, dY, [(1, 2)], [(0, 3)])
            np.testing.assert_allclose(ent["dWs_d"], [bwd["dWs_d"][1, 2]], rtol=1e-11)
            np.testing.assert_allclose(ent["dWs_g"], [bwd["dWs_g"][0, 3]], rtol=1e-11)
            np.testing.assert_allclose(ent["dWs_u"], [bwd["dWs_u"][0, 3]], rtol=1e-11)


def test_fp8_sampled_rows_equal_full_layer():
    """The per-token and per-entry evaluations used at large sizes agree with the whole
    layer in FP8 mode too (quantised forward operands, bf16 backward on the stored a, u, h
    and the unquantised x)."""
    rng = np.random.default_rng(25)
    inp = _tiny_inputs(rng, T=30, d=16, E=5, f=8, fs=4)
    dY = rng.standard_normal((30, 16))
    fwd = O.layer_forward(inp, "sigmoid", 2, fp8=True)
    bwd = O.layer_backward(inp, fwd, dY)
    plain = O.layer_forward(inp, "sigmoid", 2)
    assert not np.allclose(fwd["out"], plain["out"], rtol=1e-3)  # FP8 really changes the layer
    for t in (0, 11, 29):
        o = O.token_forward(inp, t, fwd["idx"][t], fwd["gate"][t], fp8=True)
        np.testing.assert_allclose(o, fwd["out"][t], rtol=1e-12, atol=1e-12)
        tb = O.token_backward(inp, t, fwd["logits"][t], fwd["idx"][t], "sigmoid", 2, dY[t], 0.0,
                              30, fp8=True)
        np.testing.assert_allclose(tb["dx"], bwd["dx"][t], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(tb["dg"], bwd["dg"][t], rtol=1e-11, atol=1e-12)
    for e in range(5):
        rows = np.arange(fwd["offsets"][e], fwd["offsets"][e + 1])
        toks = fwd["perm_token"][rows]
        gates = fwd["gate"][toks, fwd["perm_slot"][rows]]
        ent = O.expert_weight_grad_entries(inp, e, toks, gates, dY, [(0, 1), (9, 7)],
                                           [(2, 5), (7, 0)], fp8=True)
        np.testing.assert_allclose(ent["dW_d"], [bwd["dW_d"][e][0, 1], bwd["dW_d"][e][9, 7]], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(ent["dW_g"], [bwd["dW_g"][e][2, 5], bwd["dW_g"][e][7, 0]], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(ent["dW_u"], [bwd["dW_u"][e][2, 5], bwd["dW_u"][e][7, 0]], rtol=1e-11, atol=1e-13)
    ent = O.shared_weight_grad_entries(inp, dY, [(3, 2)], [(1, 6)], fp8=True)
    np.testing.assert_allclose(ent["dWs_d"], [bwd["dWs_d"][3, 2]], rtol=1e-11)
    np.testing.assert_allclose(ent["dWs_g"], [bwd["dWs_g"][1, 6]], rtol=1e-11)
    np.testing.assert_allclose(ent["dWs_u"], [bwd["dWs_u"][1, 6]], rtol=1e-11)


@pytest.mark.parametrize("mode, z, aux, fp8, fold, rnd, f8d", [
    ("sigmoid", 0.0, None, False, False, None, False),
    ("softmax", 0.05, None, False, False, None, False),
    ("softmax", 0.05, (10, 0.3, 0.2), False, False, None, False),
    ("sigmoid", 0.0, (10, 0.3, 0.2), False, True, "bf16", False),
    ("sigmoid", 0.0, None, True, False, "bf16", False),
    ("softmax", 0.05, None, True, False, "bf16", True),
])
def test_token_subset_backward_equals_whole_layer(mode, z, aux, fp8, fold, rnd, f8d):
    """The layer over a subset of a batch's tokens, with the batch's z-loss token count and
    the batch's balancing-loss logit gradient rows passed in, gives the whole layer's out,
    dx and dg rows of those tokens."""
    rng = np.random.default_rng(41)
    r = O.bf16_round if rnd else None
    T = 30
    inp = _tiny_inputs(rng, T=T, d=16, E=5, f=8, fs=4 if mode == "sigmoid" else 0)
    dY = O.bf16_round(rng.standard_normal((T, 16)))
    fwd = O.layer_forward(inp, mode, 2, z, rnd=r, aux=aux, fp8=fp8, fold_gate=fold,
                          fp8_dgrad=f8d)
    bwd = O.layer_backward(inp, fwd, dY)
    sub = np.array([0, 3, 4, 17, 29])
    dl = None if aux is None else O.aux_losses_backward(fwd["logits"], fwd["idx"], mode, *aux)[sub]
    part = dict(inp, x=inp["x"][sub])
    f1 = O.layer_forward(part, mode, 2, z, logits=fwd["logits"][sub], idx=fwd["idx"][sub], rnd=r,
                         fp8=fp8, fold_gate=fold, fp8_dgrad=f8d)
    b1 = O.layer_backward(part, f1, dY[sub], T_norm=T, dl_extra=dl, weight_grads=False)
    np.testing.assert_allclose(f1["out"], fwd["out"][sub], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b1["dx"], bwd["dx"][sub], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(b1["dg"], bwd["dg"][sub], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(b1["dlogits"], bwd["dlogits"][sub], rtol=1e-11, atol=1e-13)
    assert "dW_g" not in b1 and "dWs_g" not in b1


@pytest.mark.parametrize("fp8, fold, rnd, f8d", [(False, False, None, False),
                                                 (False, True, "bf16", False),
                                                 (False, False, "bf16", False),
                                                 (True, False, "bf16", False),
                                                 (True, False, "bf16", True)])
def test_whole_expert_and_shared_unit_weight_grads_equal_whole_layer(fp8, fold, rnd, f8d):
    """One expert's whole weight gradients from its own rows alone, and whole weight rows of
    chosen shared-expert units, equal those of the whole layer."""
    rng = np.random.default_rng(43)
    r = O.bf16_round if rnd else None
    T = 40
    inp = _tiny_inputs(rng, T=T, d=16, E=5, f=8, fs=6)
    dY = O.bf16_round(rng.standard_normal((T, 16)))
    fwd = O.layer_forward(inp, "sigmoid", 2, rnd=r, fp8=fp8, fold_gate=fold, fp8_dgrad=f8d)
    bwd = O.layer_backward(inp, fwd, dY)
    for e in range(5):
        rows = np.arange(fwd["offsets"][e], fwd["offsets"][e + 1])
        toks = fwd["perm_token"][rows]
        gates = fwd["gate"][toks, fwd["perm_slot"][rows]]
        w = O.expert_weight_grads(inp, e, inp["x"][toks], gates, dY[toks], rnd=r, fp8=fp8,
                                  fold_gate=fold, fp8_dgrad=f8d)
        for name in ("dW_g", "dW_u", "dW_d"):
            np.testing.assert_allclose(w[name], bwd[name][e], rtol=1e-11, atol=1e-13)
    units = [0, 2, 5]
    w = O.shared_weight_grad_units(inp, dY, units, rnd=r, fp8=fp8, fp8_dgrad=f8d)
    np.testing.assert_allclose(w["dWs_g"], bwd["dWs_g"][units], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(w["dWs_u"], bwd["dWs_u"][units], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(w["dWs_d"], bwd["dWs_d"][:, units], rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------- bf16 storage precision

def test_bf16_round_matches_library_conversion_including_ties():
    """Round-to-nearest-even to 8 significant bits equals torch's fp32 -> bf16 conversion
    (a library routine) on random values and on exact halfway cases."""
    import torch
    rng = np.random.default_rng(14)
    scale = (10.0 ** rng.integers(-40, 30, 20000)).astype(np.float32)  # includes subnormals
    vals = (rng.standard_normal(20000) * scale).astype(np.float32)
    bits = vals.view(np.uint32)
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)  # exact halfway
    allv = np.concatenate([vals, ties, np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875])])
    want = torch.from_numpy(allv).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.bf16_round(allv.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_mode_sampled_rows_equal_full_layer():
    rng = np.random.default_rng(15)
    for mode, z in (("sigmoid", 0.0), ("softmax", 0.05)):
        inp = _tiny_inputs(rng, T=24, d=8, E=5, f=4, fs=3 if mode == "sigmoid" else 0)
        dY = O.bf16_round(rng.standard_normal((24, 8)))
        fwd = O.layer_forward(inp, mode, 2, z, rnd=O.bf16_round)
        bwd = O.layer_backward(inp, fwd, dY)
        for t in (0, 5, 23):
            o = O.token_forward(inp, t, fwd["idx"][t], fwd["gate"][t], rnd=O.bf16_round)
            np.testing.assert_allclose(o, fwd["out"][t], rtol=1e-12, atol=1e-12)
            tb = O.token_backward(inp, t, fwd["logits"][t], fwd["idx"][t], mode, 2, dY[t], z, 24,
                                  rnd=O.bf16_round)
            np.testing.assert_allclose(tb["dx"], bwd["dx"][t], rtol=1e-11, atol=1e-12)
        for e in range(5):
            rows = np.arange(fwd["offsets"][e], fwd["offsets"][e + 1])
            toks = fwd["perm_token"][rows]
            gates = fwd["gate"][toks, fwd["perm_slot"][rows]]
            ent = O.expert_weight_grad_entries(inp, e, toks, gates, dY, [(3, 1)], [(2, 5)],
                                               rnd=O.bf16_round)
            np.testing.assert_allclose(ent["dW_d"], [bwd["dW_d"][e][3, 1]], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(ent["dW_g"], [bwd["dW_g"][e][2, 5]], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(ent["dW_u"], [bwd["dW_u"][e][2, 5]], rtol=1e-11, atol=1e-13)


def test_bf16_mode_stays_close_to_the_exact_definition():
    """Storing activations in bf16 moves the layer by about the bf16 unit roundoff."""
    rng = np.random.default_rng(16)
    inp = _tiny_inputs(rng, T=64, d=32, E=6, f=16, fs=8)
    dY = O.bf16_round(rng.standard_normal((64, 32)))
    f64 = O.layer_forward(inp, "sigmoid", 2)
    b16 = O.layer_forward(inp, "sigmoid", 2, rnd=O.bf16_round)
    np.testing.assert_allclose(b16["out"], f64["out"], rtol=2e-2, atol=2e-2)
    g64 = O.layer_backward(inp, f64, dY)
    g16 = O.layer_backward(inp, b16, dY)
    for name in ("dx", "dW_g", "dW_d", "dWs_u", "dW_r"):
        np.testing.assert_allclose(g16[name], g64[name], rtol=3e-2, atol=3e-2)
    # the stored tensors are bf16 values
    for name in ("A", "U", "H", "Y_perm", "out"):
        np.testing.assert_array_equal(O.bf16_round(b16[name]), b16[name])


def test_proportional_bias_update_invariants():
    """Reading of the proportional rule: the step is gamma times the relative deviation of
    the load from the mean, toward the mean; a balanced expert does not move."""
    rng = np.random.default_rng(17)
    E, T, k, gamma = 64, 49152, 4, 0.01
    b = rng.uniform(-0.05, 0.05, E).astype(np.float32)
    counts = rng.multinomial(T * k, np.ones(E) / E)
    counts[7] = T * k // E
    nb = O.bias_update_proportional(counts, b, T, k, gamma)
    mean = T * k / E
    exact_step = gamma * (mean - counts) / mean
    delta = nb.astype(np.float64) - b.astype(np.float64)
    assert delta[7] == 0.0
    # one fp32 rounding of the ratio, the product and the sum: within a few fp32 ulps of b
    ulp32 = np.spacing((np.abs(b) + np.abs(exact_step)).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(delta - exact_step) <= 4 * ulp32)
    moved = counts != mean
    assert np.all(np.sign(delta[moved]) == np.sign(mean - counts[moved]))


# ------------------------------------------------------------------- balancing losses

@pytest.mark.parametrize("mode", ["sigmoid", "softmax"])
def test_aux_losses_are_exactly_one_for_a_single_expert(mode):
    """Handbook summary, section 2.5: the one-expert MoE recorded a load-balance loss of
    exactly 1 (before its coefficient)."""
    rng = np.random.default_rng(18)
    logits = rng.standard_normal((64, 1))
    a = O.aux_losses(logits, np.zeros((64, 1), dtype=np.int64), mode, 16, 1e-3, 1e-3)
    assert a["switch_unscaled"] == 1.0 and a["seq_unscaled"] == 1.0
    assert a["switch"] == pytest.approx(1e-3) and a["seq"] == pytest.approx(1e-3)
    assert (O.aux_losses_backward(logits, np.zeros((64, 1), dtype=np.int64), mode, 16, 1e-3, 1e-3) == 0).all()


def test_aux_losses_balanced_closed_form():
    """Uniform probabilities and perfectly balanced choices: f_e = 1/E and P_e = 1/E, so the
    unscaled losses are E * E * (1/E)(1/E) = 1."""
    E, k, T = 8, 2, 32
    logits = np.zeros((T, E))
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    for mode in ("sigmoid", "softmax"):
        a = O.aux_losses(logits, idx, mode, 8, 1.0, 1.0)
        assert a["switch_unscaled"] == pytest.approx(1.0, abs=1e-15)
        assert a["seq_unscaled"] == pytest.approx(1.0, abs=1e-15)


def test_sequence_loss_uses_each_sequences_own_counts():
    """Worked by hand: two sequences of two tokens, E = 2, k = 1, softmax probabilities
    (0.9, 0.1) on sequence 0, whose tokens both choose expert 0, and (0.1, 0.9) on sequence
    1, whose tokens both choose expert 1. Per sequence f = (2, 0) resp. (0, 2) and P = the
    sequence's probabilities, so sum_e f P = 1.8 on each: seq = 1.8. Batch-wide f = P =
    (0.5, 0.5), so switch = 2 (0.25 + 0.25) = 1."""
    l9 = math.log(9.0)
    logits = np.array([[l9, 0.0], [l9, 0.0], [0.0, l9], [0.0, l9]])
    idx = np.array([[0], [0], [1], [1]])
    a = O.aux_losses(logits, idx, "softmax", 2, 1.0, 1.0)
    assert a["seq_unscaled"] == pytest.approx(1.8, rel=1e-14)
    assert a["switch_unscaled"] == pytest.approx(1.0, rel=1e-14)


@pytest.mark.parametrize("mode", ["sigmoid", "softmax"])
def test_aux_losses_gradient_matches_finite_differences(mode):
    rng = np.random.default_rng(19)
    T, E, k, L = 12, 5, 2, 4
    logits = rng.standard_normal((T, E))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    coef = (0.3, 0.7)
    ana = O.aux_losses_backward(logits, idx, mode, L, *coef)
    h = 1e-6
    num = np.zeros_like(logits)
    for ix in np.ndindex(logits.shape):
        lp = logits.copy(); lp[ix] += h
        lm = logits.copy(); lm[ix] -= h
        ap = O.aux_losses(lp, idx, mode, L, *coef)
        am = O.aux_losses(lm, idx, mode, L, *coef)
        num[ix] = ((ap["switch"] + ap["seq"]) - (am["switch"] + am["seq"])) / (2 * h)
    np.testing.assert_allclose(ana, num, rtol=1e-6, atol=1e-9)


# -------------------------------------------------------------------- FP8 quantisation

def test_e4m3_round_matches_library_conversion():
    """Round to nearest even on 4 significant bits with E4M3 subnormals equals torch's
    float8_e4m3fn conversion (a library routine) over the finite range."""
    import torch
    rng = np.random.default_rng(21)
    scale = (2.0 ** rng.integers(-12, 9, 20000)).astype(np.float32)
    vals = (rng.uniform(-1, 1, 20000).astype(np.float32) * scale)
    vals = vals[np.abs(vals) <= 464.0]
    halfway = np.array([0.5625, 1.0625, 1.1875, 3.25 + 0.125, 2.0 ** -9 * 1.5, 440.0, 464.0 - 1e-3],
                       dtype=np.float32)  # exact midpoints and near-max values
    allv = np.concatenate([vals, halfway, -halfway, np.float32([0.0])])
    want = torch.from_numpy(allv).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(O.e4m3_round(allv.astype(np.float64)), want)


def test_rowwise_fp8_quantisation_invariants():
    rng = np.random.default_rng(22)
    X = O.bf16_round(rng.standard_normal((50, 64)) * rng.uniform(0.01, 100, (50, 1)))
    X[3] = 0.0
    q, sc = O.quantize_rows_fp8(X)
    assert np.all(np.abs(q) <= 448.0)
    amax_pos = np.argmax(np.abs(X), axis=1)
    live = np.abs(X).max(axis=1) > 0
    assert np.all(np.abs(q[np.arange(50), amax_pos])[live] == 448.0)  # the row maximum maps to 448
    assert np.all(q[3] == 0.0) and sc[3] == 1.0
    assert np.all(O.e4m3_round(q) == q)  # every code is an E4M3 value
    deq = q * sc[:, None]
    rel = np.abs(deq - X) / np.maximum(np.abs(X), 1e-30)
    assert np.all((rel <= 2.0 ** -4 + 1e-12) | (np.abs(X) < 2.0 ** -6 * sc[:, None]))


def _e4m3_rows(rng, rows, cols):
    """Rows exactly representable under rowwise E4M3 scaling: E4M3 values times a per-row
    power of two, with one element at +-448 so that the row's scale is that power of two."""
    mags = np.array([m * 2.0 ** e for e in range(-6, 9) for m in (1, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875)])
    mags = mags[mags <= 448.0]
    v = rng.choice(mags, size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
    v[np.arange(rows), rng.integers(0, cols, rows)] = 448.0 * rng.choice([-1.0, 1.0], rows)
    return v * 2.0 ** rng.integers(-14, -9, size=(rows, 1))


def test_fp8_expert_reduces_to_the_exact_expert_on_representable_operands():
    """When x and every weight row are exactly representable under rowwise scaling, the FP8
    expert's a, u and h equal the exact expert's; only h's own quantisation before the down
    projection moves y, by at most its rounding (2^-4 relative per element of h)."""
    rng = np.random.default_rng(24)
    d, f = 64, 48
    x = _e4m3_rows(rng, 40, d)
    Wg, Wu = _e4m3_rows(rng, f, d), _e4m3_rows(rng, f, d)
    Wd = _e4m3_rows(rng, d, f)
    q, sc = O.quantize_rows_fp8(x)
    np.testing.assert_array_equal(q * sc[:, None], x)  # the construction is representable
    a8, u8, h8, y8 = O.swiglu_expert_fp8(x, Wg, Wu, Wd)
    a, u, h, y = O.swiglu_expert(x, Wg, Wu, Wd)
    np.testing.assert_array_equal(a8, a)
    np.testing.assert_array_equal(u8, u)
    np.testing.assert_array_equal(h8, h)
    assert not np.array_equal(y8, y)  # h itself is not representable: its codes move y
    bound = (2.0 ** -4 * np.abs(h) + 2.0 ** -9 * np.abs(h).max(axis=1, keepdims=True) / 448) @ np.abs(Wd).T
    assert np.all(np.abs(y8 - y) <= bound * (1 + 1e-12))


def test_fp8_data_gradients_are_exact_on_representable_operands():
    """The FP8 data-gradient products reduce to the exact products when every operand row
    (or column) is an E4M3 code times a scale that fp32 holds exactly.

    dh = dy W_d: dy rows are 1.75 e_i (scale 2^-8, code 448); every row and column of W_d
    holds +-1.75 among 0, +-0.25, +-0.5, +-1 (scale 2^-8 on either axis). dX = [da|du]
    [W_g; W_u]: every da row holds 49/32 among 7/8, 7/16, 7/32 (joint scale 7/2048); du
    rows hold 24 and 16 times 7/2048 (codes 24 and 16 under the joint scale, but 448 and
    298.7 under a scale of their own); every column of W_g holds 1.75 and W_u only 0.75 and
    0.5 (codes 192, 128 under the joint scale 2^-8, but 448 and 298.7 alone). So the joint
    scales give the exact products and separate ones do not."""
    rng = np.random.default_rng(51)
    d, f, n = 8, 4, 3
    vals = np.array([0.0, 0.25, -0.25, 0.5, -0.5, 1.0, -1.0])
    W_d = rng.choice(vals, (d, f))
    for i in range(d):
        W_d[i, i % f] = 1.75 * (1 if i % 2 else -1)
    for j in range(f):
        W_d[j + 4, j] = -1.75  # every column too
    dy = np.zeros((n, d))
    dy[np.arange(n), [1, 4, 6]] = 1.75
    np.testing.assert_array_equal(O.fp8_dgrad_dh(dy, W_d), dy @ W_d)
    c = 7.0 / 2048
    da = c * rng.choice([0.0, 256.0, -256.0, 128.0, 64.0], (n, f))
    da[:, 0] = c * 448.0 * np.array([1, -1, 1])
    du = c * rng.choice([16.0, -16.0], (n, f))
    du[:, 1] = c * 24.0
    W_g = rng.choice(vals, (f, d))
    W_g[0, :] = 1.75
    W_u = rng.choice([0.5, -0.5], (f, d))
    W_u[2, :] = 0.75
    np.testing.assert_array_equal(O.fp8_dgrad_dx(da, du, W_g, W_u), da @ W_g + du @ W_u)


def test_fp8_data_gradient_scaling_axes():
    """Scaling one row of the left operand, or one column of the right, by 4 scales that row
    or column of the FP8 product by exactly 4 and leaves the rest bit for bit: the scales
    run along the contraction axis of each operand (rows of dy and of [da|du]; columns of
    W_d and of [W_g; W_u])."""
    rng = np.random.default_rng(52)
    n, d, f = 5, 16, 8
    dy = O.bf16_round(rng.standard_normal((n, d)))
    W_d = O.bf16_round(rng.standard_normal((d, f)))
    base = O.fp8_dgrad_dh(dy, W_d)
    dy2 = dy.copy(); dy2[2] *= 4
    got = O.fp8_dgrad_dh(dy2, W_d)
    np.testing.assert_array_equal(got[2], 4 * base[2])
    np.testing.assert_array_equal(np.delete(got, 2, 0), np.delete(base, 2, 0))
    W2 = W_d.copy(); W2[:, 5] *= 4
    got = O.fp8_dgrad_dh(dy, W2)
    np.testing.assert_array_equal(got[:, 5], 4 * base[:, 5])
    np.testing.assert_array_equal(np.delete(got, 5, 1), np.delete(base, 5, 1))
    da = O.bf16_round(rng.standard_normal((n, f)))
    du = O.bf16_round(rng.standard_normal((n, f)))
    W_g = O.bf16_round(rng.standard_normal((f, d)))
    W_u = O.bf16_round(rng.standard_normal((f, d)))
    base = O.fp8_dgrad_dx(da, du, W_g, W_u)
    da2, du2 = da.copy(), du.copy(); da2[1] *= 4; du2[1] *= 4
    got = O.fp8_dgrad_dx(da2, du2, W_g, W_u)
    np.testing.assert_array_equal(got[1], 4 * base[1])
    np.testing.assert_array_equal(np.delete(got, 1, 0), np.delete(base, 1, 0))
    Wg2, Wu2 = W_g.copy(), W_u.copy(); Wg2[:, 3] *= 4; Wu2[:, 3] *= 4
    got = O.fp8_dgrad_dx(da, du, Wg2, Wu2)
    np.testing.assert_array_equal(got[:, 3], 4 * base[:, 3])
    np.testing.assert_array_equal(np.delete(got, 3, 1), np.delete(base, 3, 1))


def test_fp8_data_gradients_stay_close_to_the_bf16_backward():
    """E4M3 keeps 4 significant bits: the FP8 data gradients move the expert's backward by a
    few per cent of the gradient's scale, and leave the weight gradients' form alone."""
    rng = np.random.default_rng(53)
    inp = _tiny_inputs(rng, T=64, d=32, E=4, f=16, fs=8)
    dY = O.bf16_round(rng.standard_normal((64, 32)))
    f0 = O.layer_forward(inp, "sigmoid", 2, fp8=True)
    f1 = O.layer_forward(inp, "sigmoid", 2, fp8=True, fp8_dgrad=True)
    b0, b1 = O.layer_backward(inp, f0, dY), O.layer_backward(inp, f1, dY)
    for name in ("dx", "dA", "dU", "dW_g", "dW_u", "dWs_g"):
        rms = np.sqrt(np.mean(b0[name] ** 2))
        err = np.sqrt(np.mean((b1[name] - b0[name]) ** 2))
        assert 0 < err < 0.1 * rms, name
    np.testing.assert_array_equal(b1["dW_d"], b0["dW_d"])  # dy and h do not change
    np.testing.assert_array_equal(b1["dWs_d"], b0["dWs_d"])


def test_fp8_expert_stays_close_to_bf16_expert():
    """FP8 operands (3 mantissa bits, about 2% RMS rounding each) move an expert's output
    by several percent through the two GEMMs and the SwiGLU."""
    rng = np.random.default_rng(23)
    x = O.bf16_round(rng.standard_normal((64, 128)))
    Wg, Wu = (O.bf16_round(rng.standard_normal((96, 128)) / np.sqrt(128)) for _ in range(2))
    Wd = O.bf16_round(rng.standard_normal((128, 96)) / np.sqrt(96))
    y16 = O.swiglu_expert(x, Wg, Wu, Wd)[3]
    y8 = O.swiglu_expert_fp8(x, Wg, Wu, Wd)[3]
    assert np.linalg.norm(y8 - y16) / np.linalg.norm(y16) < 0.10  # measured 0.062
