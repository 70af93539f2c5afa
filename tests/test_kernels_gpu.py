"""Per-kernel parity of the CUDA path against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from pretraining_sigmoid_softmax_gb300 import ops

from gpu_common import (assert_close, assert_gemm_exact, dev, gpu_rows, h64, padded_offsets,
                        randn_bf16, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _ws(T, d, E, k):
    return torch.empty(ops.moe_workspace_bytes(T, d, E, k), dtype=torch.uint8, device="cuda")


def _route(x, W_r, b, k, mode, z):
    T, d = x.shape
    E = W_r.shape[0]
    out = dict(logits=torch.empty(T, E, device="cuda"),
               idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               gate=torch.empty(T, k, device="cuda"), score=torch.empty(T, k, device="cuda"),
               lse=torch.empty(T, device="cuda"), z=torch.zeros(1, device="cuda"))
    softmax = mode == ops.MODE_SOFTMAX
    ops.moe_route(dev(x), dev(W_r), None if softmax else dev(b), k, mode, z, out["logits"],
                  out["idx"], out["gate"], out["score"], out["lse"] if softmax else None,
                  out["z"] if softmax else None, _ws(T, d, E, k))
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------------------------- router

ROUTE_CASES = [
    (512, 256, 8, 2, "sigmoid"),
    (1000, 384, 64, 8, "sigmoid"),
    (777, 256, 32, 4, "softmax"),
    (300, 128, 128, 8, "sigmoid"),
    (129, 256, 256, 32, "softmax"),
    (64, 128, 1, 1, "sigmoid"),
    (200, 128, 5, 5, "softmax"),
    (65, 128, 200, 3, "sigmoid"),
    (400, 256, 64, 12, "sigmoid"),   # tensor-core kernel, choice wider than the network
    (333, 128, 40, 7, "sigmoid"),    # network over a ragged expert tile
    # larger layers: more tiles than CTAs in some, long reductions over d in all
    (8192, 1024, 64, 8, "sigmoid"),
    (2000, 2048, 32, 4, "softmax"),
    (20000, 1024, 128, 8, "sigmoid"),  # a ragged last wave of tiles
    (4000, 1024, 64, 12, "sigmoid"),
]


@pytest.mark.parametrize("T,d,E,k,mode", ROUTE_CASES)
def test_route_matches_oracle(T, d, E, k, mode):
    g = torch.Generator().manual_seed(T * 7 + E)
    x = randn_bf16((T, d), g)
    W_r = torch.randn(E, d, generator=g) * d ** -0.5
    b = torch.rand(E, generator=g) * 0.1 - 0.05
    m = ops.MODE_SIGMOID if mode == "sigmoid" else ops.MODE_SOFTMAX
    z = 1e-3
    r = _route(x, W_r, b, k, m, z)
    x64, W64, b64 = h64(x), h64(W_r), h64(b)
    l64 = O.router_logits(x64, W64)
    lg = h64(r["logits"])
    # fp32 dot product error bound (Higham): gamma_d * sum |x_j w_j|
    u = 2.0 ** -24
    gamma = d * u / (1 - d * u)
    bound = gamma * (np.abs(x64) @ np.abs(W64).T)
    assert (np.abs(lg - l64) <= bound).all(), "router logits outside the fp32 error bound"
    # replay the choice on the GPU's own fp32 logits
    ref = O.route(lg, mode, k, b64, z)
    near = O.near_tie_tokens(ref["select_value"], k) if mode == "sigmoid" else np.zeros(T, bool)
    idx = r["idx"].cpu().numpy()
    assert (idx[~near] == ref["idx"][~near]).all(), "expert choice differs from the oracle"
    assert near.mean() < 0.01
    keep = ~near
    np.testing.assert_allclose(h64(r["gate"])[keep], ref["gate"][keep], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(h64(r["score"])[keep], ref["score"][keep], rtol=1e-5, atol=1e-6)
    for t in range(T):  # k distinct experts per token
        assert len(set(idx[t].tolist())) == k
    if mode == "softmax":
        np.testing.assert_allclose(h64(r["lse"]), ref["lse"], rtol=1e-5, atol=1e-5)
        assert float(r["z"][0]) == pytest.approx(ref["z_loss"], rel=1e-4)


@pytest.mark.parametrize("T,d,E,k,mode", [(1000, 256, 64, 8, "sigmoid"), (500, 128, 64, 5, "sigmoid"),
                                         (777, 256, 32, 5, "softmax"), (400, 128, 24, 3, "sigmoid"),
                                         (300, 128, 128, 7, "sigmoid"), (400, 128, 64, 11, "sigmoid"),
                                         (3000, 1024, 64, 8, "sigmoid")])
def test_route_breaks_exact_ties_by_lower_index(T, d, E, k, mode):
    """Experts 2j and 2j + 1 have identical router rows (and biases), so every selection value
    has an exact twin: the choice must take the lower index first, as the definition's order
    (larger value, then lower index) says, and otherwise agree with the oracle on the GPU's
    own logits wherever the distinct values are not near a tie."""
    g = torch.Generator().manual_seed(T + 31 * E + k)
    x = randn_bf16((T, d), g)
    half = torch.randn((E + 1) // 2, d, generator=g) * d ** -0.5
    W_r = half.repeat_interleave(2, dim=0)[:E].contiguous()
    bh = torch.rand((E + 1) // 2, generator=g) * 0.1 - 0.05
    b = bh.repeat_interleave(2)[:E].contiguous()
    m = ops.MODE_SIGMOID if mode == "sigmoid" else ops.MODE_SOFTMAX
    r = _route(x, W_r, b, k, m, 0.0)
    lg = r["logits"].cpu()
    assert torch.equal(lg[:, 0:E - 1:2], lg[:, 1:E:2]), "twin experts' logits differ"
    ref = O.route(h64(lg), mode, k, h64(b), 0.0)
    if mode == "sigmoid":  # fp32 against fp64 selection values: skip near ties between pairs
        near = O.near_tie_tokens(ref["select_value"][:, 0::2], (k + 1) // 2)
    else:
        near = np.zeros(T, bool)
    assert near.mean() < 0.02
    idx = r["idx"].cpu().numpy()
    assert (idx[~near] == ref["idx"][~near]).all(), "choice differs from the oracle's order"
    for t in range(T):  # an upper twin is never taken before its lower twin
        pos = {e: i for i, e in enumerate(idx[t].tolist())}
        for e, i in pos.items():
            if e % 2 == 1:
                assert e - 1 in pos and pos[e - 1] < i, (t, idx[t])


@pytest.mark.parametrize("E,k", [(64, 8), (128, 8), (64, 12)])
def test_route_saturated_logits(E, k):
    """Logits far outside sigmoid's working range (|l| up to a few hundred): the sigmoid
    saturates at 0 and 1 in fp32, so the bias decides among the saturated experts. The
    choice must match the oracle's on the GPU's own logits wherever the values are not near
    a tie, and the scores the fp32 sigmoid of those logits. The biases are evenly spaced (in
    shuffled order), so experts saturated at the same end never tie on the bias."""
    g = torch.Generator().manual_seed(E + k)
    T, d = 700, 256
    x = randn_bf16((T, d), g)
    W_r = torch.randn(E, d, generator=g) * (60.0 * d ** -0.5)
    b = (torch.arange(E, dtype=torch.float32) * (0.1 / E) - 0.05)[torch.randperm(E, generator=g)]
    r = _route(x, W_r, b, k, ops.MODE_SIGMOID, 0.0)
    lg = h64(r["logits"])
    assert np.abs(lg).max() > 100.0
    ref = O.route(lg, "sigmoid", k, h64(b), 0.0)
    near = O.near_tie_tokens(ref["select_value"], k)
    assert near.mean() < 0.01
    idx = r["idx"].cpu().numpy()
    assert (idx[~near] == ref["idx"][~near]).all(), "expert choice differs from the oracle"
    np.testing.assert_allclose(h64(r["score"])[~near], ref["score"][~near], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(h64(r["gate"])[~near], ref["gate"][~near], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("T,d", [(2000, 512), (8192, 1024), (20000, 1024)])
def test_route_is_bitwise_repeatable(T, d):
    g = torch.Generator().manual_seed(5)
    x = randn_bf16((T, d), g)
    W_r = torch.randn(64, d, generator=g) * d ** -0.5
    b = torch.rand(64, generator=g) * 0.1 - 0.05
    r1 = _route(x, W_r, b, 8, ops.MODE_SIGMOID, 0.0)
    r2 = _route(x, W_r, b, 8, ops.MODE_SIGMOID, 0.0)
    for key in ("logits", "idx", "gate"):
        assert torch.equal(r1[key], r2[key])


# ------------------------------------------------------------------------------ permute

def _random_choice(T, E, k, gen, skew=False):
    w = torch.ones(E)
    if skew:
        w = torch.tensor([1.0 / (i + 1) ** 1.2 for i in range(E)])
        w[E // 2:E // 2 + max(1, E // 8)] = 0.0  # a block of empty experts
    idx = torch.stack([torch.multinomial(w, k, replacement=False, generator=gen) for _ in range(T)])
    return idx.to(torch.int32)


def _permute(idx, x, E, gate=None):
    T, k = idx.shape
    d = x.shape[1]
    R = ops.moe_padded_rows(T, k, E)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int64, device="cuda"),
               row_offsets=torch.empty(E + 1, dtype=torch.int64, device="cuda"),
               perm_token=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               slot_to_row=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               X_perm=torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda"))
    if gate is not None:
        out["row_gate"] = torch.full((R,), float("nan"), device="cuda")
    ops.moe_permute(dev(idx), dev(x), E, out["counts"], out["offsets"], out["row_offsets"],
                    out["perm_token"], out["slot_to_row"], out["X_perm"], _ws(T, d, E, k),
                    topk_gate=None if gate is None else dev(gate), row_gate=out.get("row_gate"))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,d,E,k,skew", [(1000, 128, 8, 2, False), (3000, 256, 64, 8, True),
                                          (2049, 128, 256, 32, False), (5, 128, 16, 4, True),
                                          (1, 128, 1, 1, False),
                                          # 157 chunks of 256 tokens: runs of 4 or 5 per lane
                                          (40100, 128, 64, 8, True)])
def test_permute_is_bit_exact(T, d, E, k, skew):
    g = torch.Generator().manual_seed(T + E)
    idx = _random_choice(T, E, k, g, skew)
    x = randn_bf16((T, d), g)
    gate = torch.rand(T, k, generator=g)
    r = _permute(idx, x, E, gate)
    D = O.dispatch(idx.numpy().astype(np.int64), E)
    counts = r["counts"].cpu().numpy()
    assert (counts == D["counts"]).all()
    assert (r["offsets"].cpu().numpy() == D["offsets"]).all()
    ro = r["row_offsets"].cpu().numpy()
    assert (ro == padded_offsets(D["counts"])).all()
    rows = gpu_rows(D["offsets"], ro)
    pt = r["perm_token"].cpu().numpy()
    assert (pt[rows] == D["perm_token"]).all()
    s2r = r["slot_to_row"].cpu().numpy()
    assert (s2r == rows[D["slot_to_row"]]).all()
    Xp = r["X_perm"].float().cpu()
    assert torch.equal(Xp[torch.from_numpy(rows)], x.float()[torch.from_numpy(D["perm_token"])])
    pad = np.setdiff1d(np.arange(int(ro[-1])), rows)
    assert (pt[pad] == -1).all()
    assert (Xp[torch.from_numpy(pad)] == 0).all()
    # the gate of each row's slot, copied in the same pass; zero on padding rows
    rg = r["row_gate"].cpu().numpy()
    want = gate.numpy()[D["perm_token"], D["perm_slot"]]
    assert np.array_equal(rg[rows].view(np.uint32), want.astype(np.float32).view(np.uint32))
    assert (rg[pad] == 0).all()


def test_permute_reports_bad_index_without_touching_other_rows():
    ops.moe_clear_device_status()
    idx = torch.tensor([[0, 1], [1, 9], [2, 2]], dtype=torch.int32)  # 9 out of range, 2 repeated
    x = randn_bf16((3, 128), torch.Generator().manual_seed(1))
    r = _permute(idx, x, 4)
    code, site = ops.moe_device_status()
    assert code == 5
    s2r = r["slot_to_row"].cpu().numpy()
    assert s2r[1, 1] == -1 and s2r[2, 1] == -1
    assert r["counts"].cpu().tolist() == [1, 2, 1, 0]
    ops.moe_clear_device_status()
    assert ops.moe_device_status()[0] == 0


def test_bounded_wait_that_runs_out_records_timeout_and_returns():
    """Failure detection without a fault: a bounded wait on an mbarrier that nothing arrives
    on runs out after its limit, records MOE_ERR_TIMEOUT (site 90) and the kernel returns;
    the context stays usable (an expert GEMM right after gives the usual result)."""
    import time
    ops.moe_clear_device_status()
    assert ops.moe_device_status()[0] == 0
    t0 = time.perf_counter()
    ops.moe_check_bounded_wait(5_000_000)  # 5 ms
    code, site = ops.moe_device_status()
    elapsed = time.perf_counter() - t0
    assert (code, site) == (6, 90)
    assert elapsed >= 0.005
    ops.moe_clear_device_status()
    assert ops.moe_device_status()[0] == 0
    g = torch.Generator().manual_seed(90)
    X, dY = randn_bf16((200, 256), g), randn_bf16((200, 256), g)
    W_g, W_u, W_d = _weights(1, 256, 128, g)
    B = _run_experts(X, dY, None, W_g, W_u, W_d)
    _check_expert(B, 0, 0, 200, X, dY, W_g, W_u, W_d, "after a timeout")


@pytest.mark.parametrize("offsets", [[0, 256, 128, 384],   # a segment that ends before it starts
                                     [0, 100, 228, 356],   # segments not whole 128-row tiles
                                     [128, 256, 384, 512],  # a layout that does not start at 0
                                     [0, 128, 256, 1024]])  # past the row capacity
def test_expert_gemms_reject_a_malformed_layout(offsets):
    """row_offsets that break the padded layout are reported (MOE_ERR_BAD_INDEX) by every
    CTA's own check before any tile is touched: the outputs stay as they were."""
    rows, d, f, E = 512, 256, 128, 3
    g = torch.Generator().manual_seed(91)
    X = dev(randn_bf16((rows, d), g))
    W_g, W_u, W_d = (dev(w) for w in _weights(E, d, f, g))
    B = _expert_buffers(rows, d, f, E)
    ro = torch.tensor(offsets, dtype=torch.int64, device="cuda")
    ops.moe_clear_device_status()
    ops.moe_expert_fwd(X, ro, W_g, W_u, W_d, B["A"], B["U"], B["H"], B["Y"], _ws(rows, d, E, 1))
    torch.cuda.synchronize()
    code, site = ops.moe_device_status()
    assert (code, site) == (5, 20)
    for name in ("A", "U", "H", "Y"):
        assert torch.isnan(B[name].float()).all(), name
    ops.moe_clear_device_status()


# --------------------------------------------------------------------- expert GEMMs

def _expert_buffers(rows, d, f, E):
    bf = dict(dtype=torch.bfloat16, device="cuda")
    return {k: torch.full(s, float("nan"), **bf) for k, s in
            dict(A=(rows, f), U=(rows, f), H=(rows, f), Y=(rows, d), dX=(rows, d), dA=(rows, f),
                 dU=(rows, f), dW_g=(E, f, d), dW_u=(E, f, d), dW_d=(E, d, f)).items()}


def _run_experts(X, dY, row_offsets, W_g, W_u, W_d):
    rows, d = X.shape
    E, f, _ = W_g.shape
    B = _expert_buffers(rows, d, f, E)
    ws = _ws(rows, d, E, 1)
    ro = None if row_offsets is None else dev(torch.from_numpy(row_offsets))
    ops.moe_expert_fwd(dev(X), ro, dev(W_g), dev(W_u), dev(W_d), B["A"], B["U"], B["H"], B["Y"], ws)
    ops.moe_expert_bwd(dev(dY), dev(X), B["A"], B["U"], B["H"], ro, dev(W_g), dev(W_u), dev(W_d),
                       B["dX"], B["dA"], B["dU"], B["dW_g"], B["dW_u"], B["dW_d"], ws)
    # the backward again with caller-made saved activations (padding rows zero), so that
    # the weight-gradient GEMM can be checked on operands that are all test inputs
    g = torch.Generator().manual_seed(rows + 99)
    live = (X.float().abs().sum(1, keepdim=True) > 0).to(torch.bfloat16)
    B["Hin"] = randn_bf16((rows, f), g) * live
    B2 = _expert_buffers(rows, d, f, E)
    ops.moe_expert_bwd(dev(dY), dev(X), dev(randn_bf16((rows, f), g) * live),
                       dev(randn_bf16((rows, f), g) * live), dev(B["Hin"]), ro, dev(W_g),
                       dev(W_u), dev(W_d), B2["dX"], B2["dA"], B2["dU"], B2["dW_g"], B2["dW_u"],
                       B2["dW_d"], ws)
    B["dW_d_in"] = B2["dW_d"]
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    return B


def _weights(E, d, f, g):
    return (randn_bf16((E, f, d), g, d ** -0.5), randn_bf16((E, f, d), g, d ** -0.5),
            randn_bf16((E, d, f), g, f ** -0.5))


def _check_expert(B, e, lo, hi, X, dY, W_g, W_u, W_d, tag):
    rnd = O.bf16_round
    x = h64(X[lo:hi])
    a, u, h, y = O.swiglu_expert(x, h64(W_g[e]), h64(W_u[e]), h64(W_d[e]), rnd)
    assert_close(B["A"][lo:hi], a, f"{tag} A")
    assert_close(B["U"][lo:hi], u, f"{tag} U")
    assert_close(B["H"][lo:hi], h, f"{tag} H")
    assert_close(B["Y"][lo:hi], y, f"{tag} Y")
    gr = O.expert_backward(h64(dY[lo:hi]), x, a, u, h, h64(W_g[e]), h64(W_u[e]), h64(W_d[e]), rnd)
    assert_close(B["dA"][lo:hi], gr["dA"], f"{tag} dA")
    assert_close(B["dU"][lo:hi], gr["dU"], f"{tag} dU")
    assert_close(B["dX"][lo:hi], gr["dX"], f"{tag} dX")
    assert_close(B["dW_d"][e], gr["dW_d"], f"{tag} dW_d", reduction=True)
    assert_close(B["dW_g"][e], gr["dW_g"], f"{tag} dW_g", reduction=True)
    assert_close(B["dW_u"][e], gr["dW_u"], f"{tag} dW_u", reduction=True)
    # tensor-core results of the caller's own operands: within half a bf16 ulp + fp32 bound
    assert_gemm_exact(B["A"][lo:hi], x, h64(W_g[e]).T, f"{tag} A exact")
    assert_gemm_exact(B["U"][lo:hi], x, h64(W_u[e]).T, f"{tag} U exact")
    assert_gemm_exact(B["dW_d_in"][e], h64(dY[lo:hi]).T, h64(B["Hin"][lo:hi]), f"{tag} dW_d exact")


@pytest.mark.parametrize("rows,d,f", [(200, 256, 128), (128, 384, 256), (77, 128, 128),
                                      (640, 512, 384), (1000, 512, 512)])
def test_dense_expert_gemms(rows, d, f):
    """One expert over all rows (the shared-expert path): ragged M tail, both tile widths."""
    g = torch.Generator().manual_seed(rows + d + f)
    X = randn_bf16((rows, d), g)
    dY = randn_bf16((rows, d), g)
    W_g, W_u, W_d = _weights(1, d, f, g)
    B = _run_experts(X, dY, None, W_g, W_u, W_d)
    _check_expert(B, 0, 0, rows, X, dY, W_g, W_u, W_d, "dense")


@pytest.mark.parametrize("counts,d,f", [([130, 0, 5, 256, 1], 256, 128),
                                        ([0, 300, 0], 256, 256),
                                        ([128, 129, 127, 0, 0, 1], 384, 128),
                                        ([300, 0, 129, 1, 513, 256], 512, 256)])
def test_routed_expert_gemms(counts, d, f):
    """Padded expert segments with empty experts and 1-row / 127 / 128 / 129-row segments."""
    E = len(counts)
    g = torch.Generator().manual_seed(sum(counts) + d)
    ro = padded_offsets(counts)
    rows = int(ro[-1]) + 128  # capacity beyond the last segment is never touched
    X = torch.zeros(rows, d, dtype=torch.bfloat16)
    dY = torch.zeros(rows, d, dtype=torch.bfloat16)
    for e in range(E):
        X[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g)
        dY[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g, 0.25)
    W_g, W_u, W_d = _weights(E, d, f, g)
    B = _run_experts(X, dY, ro, W_g, W_u, W_d)
    for e in range(E):
        lo, c = int(ro[e]), counts[e]
        if c == 0:
            for name in ("dW_g", "dW_u", "dW_d"):
                assert (B[name][e].float() == 0).all(), f"empty expert {e} {name}"
            continue
        _check_expert(B, e, lo, lo + c, X, dY, W_g, W_u, W_d, f"expert {e}")
        # padding rows stay zero through every GEMM
        for name in ("A", "U", "H", "Y", "dA", "dU", "dX"):
            assert (B[name][lo + c:int(ro[e + 1])].float() == 0).all(), f"{name} padding {e}"


@pytest.mark.parametrize("counts,d,f", [([130, 0, 5, 256, 1], 256, 128), ([300, 129], 384, 256)])
def test_router_term_in_the_dx_rows(counts, d, f):
    """moe_expert_bwd in two calls (dh first, then dX and the weight gradients) with the
    router term: each row's dX gains dl_rows[p] * W_r[e] before it is rounded; dA, dU and
    the weight gradients are bit for bit those of the single call without the term."""
    E = len(counts)
    g = torch.Generator().manual_seed(sum(counts) + 3 * d)
    ro = padded_offsets(counts)
    rows = int(ro[-1]) + 128
    X = torch.zeros(rows, d, dtype=torch.bfloat16)
    dY = torch.zeros(rows, d, dtype=torch.bfloat16)
    for e in range(E):
        X[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g)
        dY[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g, 0.25)
    W_g, W_u, W_d = _weights(E, d, f, g)
    W_r = torch.randn(E, d, generator=g) * d ** -0.5
    dl = torch.randn(rows, generator=g) * 0.3
    B0 = _run_experts(X, dY, ro, W_g, W_u, W_d)  # the single call, no term
    B1 = _expert_buffers(rows, d, f, E)
    ws = _ws(rows, d, E, 1)
    rod = dev(torch.from_numpy(ro))
    for k in ("A", "U", "H"):
        B1[k].copy_(B0[k])
    args = (dev(dY), dev(X), B1["A"], B1["U"], B1["H"], rod, dev(W_g), dev(W_u), dev(W_d),
            B1["dX"], B1["dA"], B1["dU"], B1["dW_g"], B1["dW_u"], B1["dW_d"], ws)
    ops.moe_expert_bwd(*args, parts=ops.BWD_DH)
    ops.moe_expert_bwd(*args, parts=ops.BWD_DX | ops.BWD_W, dl_rows=dev(dl), W_r=dev(W_r))
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    for name in ("dA", "dU", "dW_g", "dW_u", "dW_d"):  # bits (rows past the layout hold NaN)
        assert torch.equal(B1[name].view(torch.int16), B0[name].view(torch.int16)), name
    rnd = O.bf16_round
    for e in range(E):
        lo, c = int(ro[e]), counts[e]
        if c == 0:
            continue
        hi = lo + c
        x = h64(X[lo:hi])
        a, u, h, y = O.swiglu_expert(x, h64(W_g[e]), h64(W_u[e]), h64(W_d[e]), rnd)
        gr = O.expert_backward(h64(dY[lo:hi]), x, a, u, h, h64(W_g[e]), h64(W_u[e]),
                               h64(W_d[e]), rnd)
        term = h64(dl[lo:hi])[:, None] * h64(W_r[e])[None, :]
        assert_close(B1["dX"][lo:hi], rnd(gr["dX_exact"] + term), f"expert {e} dX with term")
        # the term really moved the rows
        assert not torch.equal(B1["dX"][lo:hi], B0["dX"][lo:hi])


# -------------------------------------------------- gate folded into the experts

@pytest.mark.parametrize("counts,d,f", [([130, 0, 5, 256, 1], 256, 256), ([77, 300, 0], 384, 128)])
def test_gate_folded_expert_path(counts, d, f):
    """moe_expert_fwd / moe_expert_bwd with row gates: h and y carry the gate, dh = g (dy W_d),
    and the gate-gradient partials sum to <dy, y> (the combine's gate gradient)."""
    E = len(counts)
    g = torch.Generator().manual_seed(sum(counts) + 7 * f)
    ro = padded_offsets(counts)
    rows = int(ro[-1]) + 128
    X = torch.zeros(rows, d, dtype=torch.bfloat16)
    dY = torch.zeros(rows, d, dtype=torch.bfloat16)
    gate = torch.zeros(rows)
    for e in range(E):
        X[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g)
        dY[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g, 0.25)
        gate[ro[e]:ro[e] + counts[e]] = torch.rand(counts[e], generator=g) * 0.9 + 0.05
    W_g, W_u, W_d = _weights(E, d, f, g)
    B = _expert_buffers(rows, d, f, E)
    ws = _ws(rows, d, E, 1)
    rod = dev(torch.from_numpy(ro))
    rg = dev(gate)
    part = torch.full((rows, f // 64), float("nan"), device="cuda")
    ops.moe_expert_fwd(dev(X), rod, dev(W_g), dev(W_u), dev(W_d), B["A"], B["U"], B["H"], B["Y"],
                       ws, row_gate=rg)
    ops.moe_expert_bwd(dev(dY), dev(X), B["A"], B["U"], B["H"], rod, dev(W_g), dev(W_u), dev(W_d),
                       B["dX"], B["dA"], B["dU"], B["dW_g"], B["dW_u"], B["dW_d"], ws,
                       row_gate=rg, gate_part=part)
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    rnd = O.bf16_round
    for e in range(E):
        lo, c = int(ro[e]), counts[e]
        if c == 0:
            for name in ("dW_g", "dW_u", "dW_d"):
                assert (B[name][e].float() == 0).all()
            continue
        hi = lo + c
        x, gv, dy = h64(X[lo:hi]), h64(gate[lo:hi])[:, None], h64(dY[lo:hi])
        a, u, h, y = O.swiglu_expert(x, h64(W_g[e]), h64(W_u[e]), h64(W_d[e]), rnd)
        assert_close(B["A"][lo:hi], a, f"expert {e} A")
        a_acc, u_acc = x @ h64(W_g[e]).T, x @ h64(W_u[e]).T  # before their bf16 rounding
        h_g = rnd(gv * O.silu(a_acc) * u_acc)  # the gated h, rounded where it is stored
        assert_close(B["H"][lo:hi], h_g, f"expert {e} gated h")
        assert_gemm_exact(B["Y"][lo:hi], h64(B["H"][lo:hi]), h64(W_d[e]).T, f"expert {e} gated y")
        assert_close(B["Y"][lo:hi], gv * y, f"expert {e} gated y vs g y")
        # upstream gradient g dy; dW_d = (g dy)^T (h_g / g) = dy^T h_g, the stored operand
        gr = O.expert_backward(gv * dy, x, a, u, h_g / gv, h64(W_g[e]), h64(W_u[e]),
                               h64(W_d[e]), rnd)
        for name in ("dA", "dU", "dX"):
            assert_close(B[name][lo:hi], gr[name], f"expert {e} {name}")
        for name in ("dW_g", "dW_u", "dW_d"):
            assert_close(B[name][e], gr[name], f"expert {e} {name}", reduction=True)
        dg = part[lo:hi].double().sum(1).cpu().numpy()
        # (dy W_d) . silu(a) u over the stored a, u (the kernel's own operands; the oracle's
        # a, u can round to the neighbouring bf16 value): <dy, y> of the ungated y = h W_d^T
        A_s, U_s = h64(B["A"][lo:hi]), h64(B["U"][lo:hi])
        ref = ((dy @ h64(W_d[e])) * O.silu(A_s) * U_s).sum(1)
        assert_close(dg, ref, f"expert {e} gate gradient", atol=1e-3, rtol=1e-3, reduction=True)
        # padding rows of the segment stay zero
        for name in ("A", "U", "H", "Y", "dA", "dU", "dX"):
            assert (B[name][hi:int(ro[e + 1])].float() == 0).all(), f"{name} padding {e}"


def test_row_gates_and_gate_gradient_are_bit_exact():
    g = torch.Generator().manual_seed(61)
    T, d, E, k, f = 900, 128, 12, 3, 384
    idx = _random_choice(T, E, k, g, skew=True)
    P = _permute(idx, randn_bf16((T, d), g), E)
    R = P["X_perm"].shape[0]
    gate = torch.rand(T, k, generator=g)
    row_gate = torch.full((R,), float("nan"), device="cuda")
    ops.moe_row_gates(dev(gate), P["slot_to_row"], row_gate)
    s2r = P["slot_to_row"].cpu().numpy().reshape(-1)
    want = np.zeros(R, np.float32)
    want[s2r] = gate.numpy().reshape(-1)
    assert np.array_equal(row_gate.cpu().numpy().view(np.uint32), want.view(np.uint32))
    part = torch.randn(R, f // 64, generator=g)
    dg = torch.empty(T, k, device="cuda")
    ops.moe_gate_grad(dev(part), P["slot_to_row"], f, dg)
    acc = np.zeros(T * k, np.float32)
    pn = part.numpy()[s2r]
    for j in range(f // 64):  # fp32, in order of j
        acc = (acc + pn[:, j]).astype(np.float32)
    assert np.array_equal(dg.cpu().numpy().reshape(-1).view(np.uint32), acc.view(np.uint32))


# ------------------------------------------------------------- combine and backward

def test_combine_and_backward_kernels():
    g = torch.Generator().manual_seed(21)
    T, d, E, k = 700, 256, 16, 4
    idx = _random_choice(T, E, k, g, skew=True)
    x = randn_bf16((T, d), g)
    P = _permute(idx, x, E)
    D = O.dispatch(idx.numpy().astype(np.int64), E)
    ro = P["row_offsets"].cpu().numpy()
    rows = gpu_rows(D["offsets"], ro)
    R = P["X_perm"].shape[0]
    Y_perm = torch.zeros(R, d, dtype=torch.bfloat16)
    Y_perm[torch.from_numpy(rows)] = randn_bf16((T * k, d), g)
    gate = torch.rand(T, k, generator=g)
    Ys = randn_bf16((T, d), g)
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ops.moe_combine(dev(Y_perm), dev(gate), P["slot_to_row"], dev(Ys), out)
    Yp64 = h64(Y_perm)[rows]
    ref = O.combine(Yp64, h64(gate), D["slot_to_row"], h64(Ys), O.bf16_round)
    assert_close(out, ref, "combine")
    # combine backward
    dY = randn_bf16((T, d), g)
    dY_perm = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dg = torch.empty(T, k, device="cuda")
    ops.moe_combine_bwd(dev(dY), dev(Y_perm), dev(gate), P["slot_to_row"], P["row_offsets"],
                        P["perm_token"], dY_perm, dg)
    rdYp, rdg = O.combine_backward(h64(dY), Yp64, h64(gate), D["slot_to_row"], D["perm_token"],
                                   D["perm_slot"], O.bf16_round)
    assert_close(dY_perm[torch.from_numpy(rows).cuda()], rdYp, "dY_perm")
    assert_close(dg, rdg, "dg", atol=1e-4, rtol=1e-4, reduction=True)
    pad = torch.from_numpy(np.setdiff1d(np.arange(int(ro[-1])), rows)).cuda()
    assert (dY_perm[pad].float() == 0).all()
    # rows that already carry their gates: unweighted sum; backward: plain row copies
    out1 = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ops.moe_combine(dev(Y_perm), None, P["slot_to_row"], dev(Ys), out1)
    assert_close(out1, O.combine(Yp64, np.ones((T, k)), D["slot_to_row"], h64(Ys), O.bf16_round),
                 "combine without gates")
    dY_copy = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops.moe_combine_bwd(dev(dY), None, None, P["slot_to_row"], P["row_offsets"], P["perm_token"],
                        dY_copy, None)
    assert torch.equal(dY_copy[torch.from_numpy(rows).cuda()].cpu(),
                       dY[torch.from_numpy(D["perm_token"])])
    assert (dY_copy[pad].float() == 0).all()
    # input gradient with shared and router terms
    dX_perm = torch.zeros(R, d, dtype=torch.bfloat16)
    dX_perm[torch.from_numpy(rows)] = randn_bf16((T * k, d), g)
    dxs = randn_bf16((T, d), g)
    W_r = torch.randn(E, d, generator=g) * d ** -0.5
    dl = torch.randn(T, E, generator=g) * (torch.rand(T, E, generator=g) < 0.3)
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ops.moe_permute_bwd(dev(dX_perm), P["slot_to_row"], dev(dxs), dev(dl), dev(W_r), dx)
    ref = O.input_gradient(h64(dX_perm)[rows], D["slot_to_row"], h64(dxs), h64(dl) @ h64(W_r),
                           O.bf16_round)
    assert_close(dx, ref, "dx")
    # the same with the router's term formed on the tensor cores first
    dx_r = torch.empty(T, d, device="cuda")
    ops.moe_router_dx(dev(dl), dev(W_r), dx_r, _ws(T, d, E, k))
    dx2 = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ops.moe_permute_bwd(dev(dX_perm), P["slot_to_row"], dev(dxs), None, None, dx2, dx_router=dx_r)
    assert_close(dx2, ref, "dx (router term from moe_router_dx)")


# E = 8 and 100 (expert axis padded to 64 and 128), d = 256 and 384 (256- and 128-column
# tiles), a ragged token count
@pytest.mark.parametrize("T,d,E", [(1000, 256, 8), (777, 384, 100), (64, 128, 64)])
def test_router_dx_is_the_fp32_product(T, d, E):
    g = torch.Generator().manual_seed(T + d + E)
    dl = torch.randn(T, E, generator=g) * 0.1
    W_r = torch.randn(E, d, generator=g) * d ** -0.5
    dx_r = torch.full((T, d), float("nan"), device="cuda")
    ops.moe_router_dx(dev(dl), dev(W_r), dx_r, _ws(T, d, E, 2))
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    dl64, W64 = h64(dl), h64(W_r)
    ref = dl64 @ W64
    # kept pieces d0 w0 + d0 w1 + d1 w0: dropped terms below 3 * 2^-16 of each product, plus
    # the fp32 accumulation of 3E products (Higham gamma_3E) and the pieces' own residue
    scale = np.abs(dl64) @ np.abs(W64)
    bound = (3 * 2.0 ** -16 + (3 * E + 8) * 2.0 ** -24) * scale
    got = h64(dx_r)
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= bound).all(), f"max excess {np.max(np.abs(got - ref) - bound):.3e}"


# E <= 128 runs the tensor-core W_r-gradient kernel (64- and 128-wide expert tiles, ragged
# token splits); E = 200 the SIMT kernel.
@pytest.mark.parametrize("mode,T,d,E,k", [("sigmoid", 3000, 256, 32, 4), ("softmax", 3000, 256, 32, 4),
                                          ("sigmoid", 4100, 512, 64, 8), ("softmax", 1000, 384, 128, 8),
                                          ("sigmoid", 333, 128, 200, 3), ("softmax", 70, 128, 8, 2)])
def test_router_backward(mode, T, d, E, k):
    g = torch.Generator().manual_seed(31 + T + E)
    x = randn_bf16((T, d), g)
    W_r = torch.randn(E, d, generator=g) * d ** -0.5
    b = torch.rand(E, generator=g) * 0.1 - 0.05
    m = ops.MODE_SIGMOID if mode == "sigmoid" else ops.MODE_SOFTMAX
    z = 0.01
    r = _route(x, W_r, b, k, m, z)
    dg = torch.randn(T, k, generator=g)
    dl = torch.empty(T, E, device="cuda")
    dW_r = torch.empty(E, d, device="cuda")
    ops.moe_route_bwd(dev(dg), dev(x), r["idx"], r["gate"], r["score"],
                      r["logits"] if mode == "softmax" else None,
                      r["lse"] if mode == "softmax" else None, E, m, z, dl, dW_r, _ws(T, d, E, k))
    torch.cuda.synchronize()
    lg = h64(r["logits"])
    ref = O.route(lg, mode, k, h64(b), z)
    ref = O._regate(ref, lg, r["idx"].cpu().numpy(), mode, h64(b), z)
    rb = O.router_backward(h64(dg), ref, h64(x), h64(W_r), mode, z)
    assert_close(dl, rb["dlogits"], "dlogits", atol=1e-5, rtol=1e-4)
    assert_close(dW_r, rb["dW_r"], "dW_r", atol=1e-3, rtol=1e-3, reduction=True)
    if mode == "sigmoid":  # each slot's logit gradient at its row as well, the same bits
        s2r = torch.randperm(T * k, generator=g).to(torch.int32).reshape(T, k) + 3
        s2r[0, 0] = -1  # a dropped slot writes nothing
        rows = torch.full((T * k + 3,), float("nan"), device="cuda")
        dl2 = torch.empty(T, E, device="cuda")
        ops.moe_route_bwd(dev(dg), dev(x), r["idx"], r["gate"], r["score"], None, None, E, m, z,
                          dl2, dW_r, _ws(T, d, E, k), slot_to_row=dev(s2r), dl_rows=rows)
        torch.cuda.synchronize()
        assert torch.equal(dl2, dl)
        idx = r["idx"].cpu().long()
        want = dl.cpu().gather(1, idx)
        got = rows.cpu()[s2r.long().clamp(min=0)]
        live = s2r >= 0
        assert torch.equal(got[live], want[live])
        assert torch.isnan(rows.cpu()[:3]).all()  # rows that no slot maps to are left alone


def test_bias_update_is_bit_exact():
    g = torch.Generator().manual_seed(41)
    E, T, k = 64, 4096, 8
    counts = torch.multinomial(torch.ones(E), T * k, replacement=True, generator=g).bincount(minlength=E)
    counts[3] = T * k // E  # exactly balanced expert: no change
    counts = counts.to(torch.int32)
    b = torch.rand(E, generator=g) * 0.1 - 0.05
    bd = dev(b)
    ops.moe_bias_update(dev(counts), T, k, 0.001, bd)
    ref = O.bias_update(counts.numpy(), b.numpy(), T, k, 0.001)
    assert np.array_equal(bd.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_proportional_bias_update_is_bit_exact():
    g = torch.Generator().manual_seed(43)
    E, T, k = 64, 49152, 4
    counts = torch.multinomial(torch.ones(E), T * k, replacement=True, generator=g).bincount(minlength=E)
    counts[5] = T * k // E
    counts = counts.to(torch.int32)
    b = torch.rand(E, generator=g) * 0.1 - 0.05
    bd = dev(b)
    ops.moe_bias_update_proportional(dev(counts), T, k, 0.01, bd)
    ref = O.bias_update_proportional(counts.numpy(), b.numpy(), T, k, 0.01)
    assert np.array_equal(bd.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("mode,T,E,k,L", [("sigmoid", 4096, 64, 8, 1024), ("softmax", 3000, 32, 4, 1000),
                                         ("sigmoid", 512, 1, 1, 256), ("softmax", 777, 200, 3, 777)])
def test_balancing_losses_match_oracle(mode, T, E, k, L):
    g = torch.Generator().manual_seed(T + E)
    logits = torch.randn(T, E, generator=g) * 2
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    m = ops.MODE_SIGMOID if mode == "sigmoid" else ops.MODE_SOFTMAX
    sw, sq = 1e-3, 2e-3
    aux = torch.zeros(2, device="cuda")
    f = torch.empty(E + (T // L) * E, device="cuda")
    dl = torch.empty(T, E, device="cuda")
    ops.moe_aux_loss(dev(logits), dev(idx), m, L, sw, sq, aux, f, _ws(T, 128, E, k))
    ops.moe_aux_loss_bwd(dev(logits), f, m, L, sw, sq, dl)
    torch.cuda.synchronize()
    ref = O.aux_losses(h64(logits), idx.numpy().astype(np.int64), mode, L, sw, sq)
    assert float(aux[0]) == pytest.approx(ref["switch"], rel=1e-5)
    assert float(aux[1]) == pytest.approx(ref["seq"], rel=1e-5)
    np.testing.assert_allclose(h64(f[:E]), ref["f"], rtol=1e-6)
    rdl = O.aux_losses_backward(h64(logits), idx.numpy().astype(np.int64), mode, L, sw, sq)
    scale = np.abs(rdl).max()
    assert_close(dl, rdl, "dlogits_aux", atol=1e-5 * scale, rtol=1e-4)


def test_router_backward_adds_the_extra_logit_gradient():
    g = torch.Generator().manual_seed(33)
    T, d, E, k = 2000, 256, 32, 4
    x = randn_bf16((T, d), g)
    W_r = torch.randn(E, d, generator=g) * d ** -0.5
    b = torch.rand(E, generator=g) * 0.1 - 0.05
    r = _route(x, W_r, b, k, ops.MODE_SIGMOID, 0.0)
    dg = torch.randn(T, k, generator=g)
    extra = torch.randn(T, E, generator=g) * 1e-3
    dl = torch.empty(T, E, device="cuda")
    dW_r = torch.empty(E, d, device="cuda")
    ops.moe_route_bwd(dev(dg), dev(x), r["idx"], r["gate"], r["score"], None, None, E,
                      ops.MODE_SIGMOID, 0.0, dl, dW_r, _ws(T, d, E, k), dlogits_extra=dev(extra))
    torch.cuda.synchronize()
    lg = h64(r["logits"])
    ref = O.route(lg, "sigmoid", k, h64(b))
    ref = O._regate(ref, lg, r["idx"].cpu().numpy(), "sigmoid", h64(b), 0.0)
    rb = O.router_backward(h64(dg), ref, h64(x), h64(W_r), "sigmoid", 0.0, dl_extra=h64(extra))
    assert_close(dl, rb["dlogits"], "dlogits", atol=1e-5, rtol=1e-4)
    assert_close(dW_r, rb["dW_r"], "dW_r", atol=1e-3, rtol=1e-3, reduction=True)


# ------------------------------------------------------------------------------- FP8

def _e4m3_values(codes_u8):
    return h64(codes_u8.cpu().view(torch.float8_e4m3fn).float())


def test_fp8_rowwise_quantisation_is_bit_exact():
    g = torch.Generator().manual_seed(51)
    X = randn_bf16((300, 512), g) * torch.rand(300, 1, generator=g).mul(50).to(torch.bfloat16)
    X[7] = 0
    Q = torch.empty(300, 512, dtype=torch.uint8, device="cuda")
    S = torch.empty(300, device="cuda")
    lim = torch.tensor([250], dtype=torch.int64, device="cuda")  # rows past 250 untouched
    Q.fill_(0x7F)
    ops.moe_quantize_rows_fp8(dev(X), lim, Q, S)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_rows_fp8(h64(X))
    assert np.array_equal(S[:250].cpu().numpy().view(np.uint32), s_ref[:250].astype(np.float32).view(np.uint32))
    assert np.array_equal(_e4m3_values(Q[:250]), q_ref[:250])
    assert (Q[250:] == 0x7F).all()


def test_fp8_quantisation_is_bit_exact_on_ties_and_extremes():
    """Rows built so that x / scale lands exactly on E4M3 rounding midpoints (power-of-two
    scales), rows spanning nine decades (most quotients round to zero or subnormal codes),
    and rows at the saturation edge: the codes and scales must equal the oracle's IEEE
    quotients bit for bit."""
    g = torch.Generator().manual_seed(52)
    cols = 256
    rows = []
    # midpoints between neighbouring E4M3 values in [2^-6, 448), signed, times 2^k
    mids = []
    for e in range(-6, 9):
        for m in range(8):
            lo = (1 + m / 8) * 2.0 ** e
            mids.append(lo + 2.0 ** e / 16)
    mids = torch.tensor([v for v in mids if v < 448.0])
    for k in (-20, -3, 0, 5, 30):
        v = mids[torch.randint(len(mids), (cols,), generator=g)]
        v = v * torch.where(torch.rand(cols, generator=g) < 0.5, -1.0, 1.0)
        v[0] = 448.0  # sets the row's amax, so scale = 2^k exactly
        rows.append(v * 2.0 ** k)
    for _ in range(40):  # nine decades in one row, random row maxima
        mag = 10.0 ** (torch.rand(cols, generator=g) * 9 - 6)
        rows.append(mag * torch.randn(cols, generator=g).sign())
    rows.append(torch.full((cols,), 3.0))  # every element at the row maximum
    X = torch.stack(rows).to(torch.bfloat16)
    n = X.shape[0]
    Q = torch.empty(n, cols, dtype=torch.uint8, device="cuda")
    S = torch.empty(n, device="cuda")
    ops.moe_quantize_rows_fp8(dev(X), None, Q, S)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_rows_fp8(h64(X))
    assert np.array_equal(S.cpu().numpy().view(np.uint32), s_ref.astype(np.float32).view(np.uint32))
    assert np.array_equal(_e4m3_values(Q), q_ref)


@pytest.mark.parametrize("T,d,E,k,skew", [(1000, 256, 8, 2, False), (777, 512, 16, 4, True),
                                          (5, 128, 16, 4, True)])
def test_fp8_permuted_codes_equal_quantised_permuted_rows(T, d, E, k, skew):
    """Codes and scales copied from the token rows to the expert-major rows equal the
    oracle's rowwise quantisation of the permuted bf16 rows bit for bit; padding rows are
    zero codes with scale 1 (a zero row's quantisation), including skewed layouts with empty
    experts."""
    g = torch.Generator().manual_seed(T + 7 * E)
    idx = _random_choice(T, E, k, g, skew)
    x = randn_bf16((T, d), g) * torch.rand(T, 1, generator=g).mul(20).to(torch.bfloat16)
    x[min(3, T - 1)] = 0  # a zero token row: scale 1 on each of its rows
    r = _permute(idx, x, E)
    xq = torch.empty(T, d, dtype=torch.uint8, device="cuda")
    sx = torch.empty(T, device="cuda")
    ops.moe_quantize_rows_fp8(dev(x), None, xq, sx)
    R = r["X_perm"].shape[0]
    Xq = torch.full((R, d), 0x7F, dtype=torch.uint8, device="cuda")
    sX = torch.full((R,), -7.0, device="cuda")
    ops.moe_permute_fp8(xq, sx, r["slot_to_row"], r["perm_token"], r["row_offsets"], Xq, sX)
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    n = int(r["row_offsets"][-1])
    q_ref, s_ref = O.quantize_rows_fp8(h64(r["X_perm"][:n].cpu()))
    assert np.array_equal(sX[:n].cpu().numpy().view(np.uint32), s_ref.astype(np.float32).view(np.uint32))
    assert np.array_equal(_e4m3_values(Xq[:n]), q_ref)
    assert (Xq[n:] == 0x7F).all() and (sX[n:] == -7.0).all()  # past the layout: untouched


def _quantize(t):
    rows = t.reshape(-1, t.shape[-1])
    Q = torch.empty(rows.shape, dtype=torch.uint8, device="cuda")
    S = torch.empty(rows.shape[0], device="cuda")
    ops.moe_quantize_rows_fp8(dev(rows), None, Q, S)
    return Q.view(t.shape), S


@pytest.mark.parametrize("counts,d,f", [(None, 512, 256), ([300, 0, 129, 1, 513], 512, 256),
                                        ([130, 5, 0], 384, 128)])
def test_fp8_expert_forward_matches_oracle(counts, d, f):
    g = torch.Generator().manual_seed(61 + d)
    if counts is None:
        rows, E, ro, segs = 700, 1, None, [(0, 700)]
        X = randn_bf16((rows, d), g)
    else:
        E = len(counts)
        ro = padded_offsets(counts)
        rows = int(ro[-1]) + 128
        X = torch.zeros(rows, d, dtype=torch.bfloat16)
        segs = []
        for e in range(E):
            X[ro[e]:ro[e] + counts[e]] = randn_bf16((counts[e], d), g)
            segs.append((int(ro[e]), int(ro[e]) + counts[e]))
    W_g, W_u, W_d = _weights(E, d, f, g)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    A, U, H = (torch.full((rows, f), float("nan"), **bf) for _ in range(3))
    Y = torch.full((rows, d), float("nan"), **bf)
    Hq = torch.empty(rows, f, dtype=torch.uint8, device="cuda")
    sH = torch.empty(rows, device="cuda")
    ro_d = None if ro is None else dev(torch.from_numpy(ro))
    Xq = torch.empty(rows, d, dtype=torch.uint8, device="cuda")
    sX = torch.empty(rows, device="cuda")
    ops.moe_quantize_rows_fp8(dev(X), None if ro_d is None else ro_d[E:], Xq, sX)
    Wgq, sWg = _quantize(W_g)
    Wuq, sWu = _quantize(W_u)
    Wdq, sWd = _quantize(W_d)
    ops.moe_expert_fwd_fp8(Xq, sX, ro_d, Wgq, sWg, Wuq, sWu, Wdq, sWd, A, U, H, Hq, sH, Y,
                           _ws(rows, d, E, 1))
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    for e, (lo, hi) in enumerate(segs):
        if hi == lo:
            continue
        a, u, h, y = O.swiglu_expert_fp8(h64(X[lo:hi]), h64(W_g[e]), h64(W_u[e]), h64(W_d[e]),
                                         O.bf16_round)
        assert_close(A[lo:hi], a, f"fp8 A e{e}")
        assert_close(U[lo:hi], u, f"fp8 U e{e}")
        assert_close(H[lo:hi], h, f"fp8 H e{e}")
        assert_close(Y[lo:hi], y, f"fp8 Y e{e}")
        # tensor-core result of the oracle's own E4M3 operands, dequantised in the epilogue
        xq = O.fp8_dequant_rows(h64(X[lo:hi]))
        assert_gemm_exact(A[lo:hi], xq, O.fp8_dequant_rows(h64(W_g[e])).T, f"fp8 A exact e{e}")


# ------------------------------------------------------ FP8 data gradients (backward)

def test_fp8_columnwise_and_joint_row_codes_are_bit_exact():
    """moe_quantize_cols_fp8 (one scale per column over the rows, codes transposed), also
    over the stack of two matrices, and moe_quantize_rows2_fp8 (one scale per row over two
    halves) give the oracle's codes and scales bit for bit."""
    g = torch.Generator().manual_seed(71)
    E, K0, N = 3, 256, 320
    X0 = randn_bf16((E, K0, N), g) * torch.rand(1, 1, N, generator=g).mul(40).to(torch.bfloat16)
    X1 = randn_bf16((E, K0, N), g) * 0.25
    X0[1, :, 7] = 0  # an all-zero column: scale 1
    for X1v, K in ((None, K0), (X1, 2 * K0)):
        Qt = torch.full((E, N, K), 0x7F, dtype=torch.uint8, device="cuda")
        S = torch.empty(E * N, device="cuda")
        ops.moe_quantize_cols_fp8(dev(X0), None if X1v is None else dev(X1v), Qt, S)
        torch.cuda.synchronize()
        for e in range(E):
            M = h64(X0[e]) if X1v is None else np.concatenate([h64(X0[e]), h64(X1v[e])], axis=0)
            q_ref, s_ref = O.quantize_rows_fp8(M.T)  # columns of M as rows
            assert np.array_equal(S[e * N:(e + 1) * N].cpu().numpy().view(np.uint32),
                                  s_ref.astype(np.float32).view(np.uint32))
            assert np.array_equal(_e4m3_values(Qt[e]), q_ref)
    rows, cols = 300, 256
    A = randn_bf16((rows, cols), g) * torch.rand(rows, 1, generator=g).mul(8).to(torch.bfloat16)
    B = randn_bf16((rows, cols), g) * 0.1
    B[5] = 30.0  # this row's amax comes from the second half
    Q = torch.full((rows, 2 * cols), 0x7F, dtype=torch.uint8, device="cuda")
    S = torch.empty(rows, device="cuda")
    lim = torch.tensor([280], dtype=torch.int64, device="cuda")
    ops.moe_quantize_rows2_fp8(dev(A), dev(B), lim, Q, S)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_rows_fp8(np.concatenate([h64(A), h64(B)], axis=1))
    assert np.array_equal(S[:280].cpu().numpy().view(np.uint32),
                          s_ref[:280].astype(np.float32).view(np.uint32))
    assert np.array_equal(_e4m3_values(Q[:280]), q_ref[:280])
    assert (Q[280:] == 0x7F).all()


@pytest.mark.parametrize("counts,d,f", [(None, 512, 256), ([300, 0, 129, 1, 513], 512, 256),
                                        ([130, 5, 0], 384, 128)])
def test_fp8_expert_backward_matches_oracle(counts, d, f):
    """moe_expert_bwd_fp8 on caller-made saved activations: dA and dU against the oracle's FP8
    data gradient; dX as the exact tensor-core product of the oracle's own codes of the GPU's
    [dA | dU] and of [W_g; W_u]; the bf16 weight gradients as before; empty experts zero."""
    g = torch.Generator().manual_seed(73 + d)
    if counts is None:
        E, ro, rows, segs = 1, None, 600, [(0, 600)]
    else:
        E = len(counts)
        ro = padded_offsets(counts)
        rows = int(ro[-1]) + 128
        segs = [(int(ro[e]), int(ro[e]) + counts[e]) for e in range(E)]
    z = dict(dtype=torch.bfloat16)
    X, dY = torch.zeros(rows, d, **z), torch.zeros(rows, d, **z)
    A, U, H = (torch.zeros(rows, f, **z) for _ in range(3))
    for lo, hi in segs:
        for t, std in ((X, 1.0), (dY, 0.3), (A, 1.0), (U, 1.0), (H, 0.5)):
            t[lo:hi] = randn_bf16((hi - lo, t.shape[1]), g, std)
    W_g, W_u, W_d = _weights(E, d, f, g)
    ro_d = None if ro is None else dev(torch.from_numpy(ro))
    u8 = dict(dtype=torch.uint8, device="cuda")
    dYq, sdY = torch.empty(rows, d, **u8), torch.empty(rows, device="cuda")
    ops.moe_quantize_rows_fp8(dev(dY), None if ro_d is None else ro_d[E:], dYq, sdY)
    Wdq, sWd = torch.empty(E, f, d, **u8), torch.empty(E * f, device="cuda")
    Wguq, sWgu = torch.empty(E, d, 2 * f, **u8), torch.empty(E * d, device="cuda")
    ops.moe_quantize_cols_fp8(dev(W_d), None, Wdq, sWd)
    ops.moe_quantize_cols_fp8(dev(W_g), dev(W_u), Wguq, sWgu)
    B = _expert_buffers(rows, d, f, E)
    AUq, sAU = torch.empty(rows, 2 * f, **u8), torch.empty(rows, device="cuda")
    ops.moe_expert_bwd_fp8(dYq, sdY, dev(dY), dev(X), dev(A), dev(U), dev(H), ro_d, Wdq, sWd,
                           Wguq, sWgu, B["dX"], B["dA"], B["dU"], AUq, sAU, B["dW_g"], B["dW_u"],
                           B["dW_d"], _ws(rows, d, E, 1))
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    for e, (lo, hi) in enumerate(segs):
        if hi == lo:
            for nm in ("dW_g", "dW_u", "dW_d"):
                assert (B[nm][e] == 0).all(), nm
            continue
        x, dy, a, u, h = (h64(t[lo:hi]) for t in (X, dY, A, U, H))
        wg, wu, wd = h64(W_g[e]), h64(W_u[e]), h64(W_d[e])
        r = O.fp8_dgrad_dh(dy, wd)
        da, du = O.swiglu_backward(r, a, u)
        assert_close(B["dA"][lo:hi], O.bf16_round(da), f"fp8 dA e{e}")
        assert_close(B["dU"][lo:hi], O.bf16_round(du), f"fp8 dU e{e}")
        # dX: the exact product of the codes of the GPU's own bf16 dA, dU and of the weights
        dag, dug = h64(B["dA"][lo:hi]), h64(B["dU"][lo:hi])
        AU = O.fp8_dequant_rows(np.concatenate([dag, dug], axis=1))
        Wgu = O.fp8_dequant_cols(np.concatenate([wg, wu], axis=0))
        assert_gemm_exact(B["dX"][lo:hi], AU, Wgu, f"fp8 dX exact e{e}")
        ref = O.expert_backward(dy, x, a, u, h, wg, wu, wd, O.bf16_round, fp8_dgrad=True)
        assert_close(B["dX"][lo:hi], ref["dX"], f"fp8 dX e{e}")
        assert_gemm_exact(B["dW_d"][e], dy.T, h, f"dW_d exact e{e}")
        assert_gemm_exact(B["dW_g"][e], dag.T, x, f"dW_g exact e{e}")
        assert_gemm_exact(B["dW_u"][e], dug.T, x, f"dW_u exact e{e}")


def test_combine_backward_with_fp8_codes():
    """moe_combine_bwd_fp8 gives moe_combine_bwd's dY_perm and dg bit for bit, and the codes
    and scales of moe_quantize_rows_fp8 of that dY_perm (padding rows: zero codes, scale 1),
    including a token whose gradient row is zero and a gate of zero."""
    g = torch.Generator().manual_seed(75)
    T, d, E, k = 900, 384, 12, 4
    idx = _random_choice(T, E, k, g, skew=True)
    P = _permute(idx, randn_bf16((T, d), g), E)
    R = P["X_perm"].shape[0]
    Y_perm = randn_bf16((R, d), g)
    gate = torch.rand(T, k, generator=g)
    gate[3, 1] = 0.0
    dY = randn_bf16((T, d), g) * torch.rand(T, 1, generator=g).mul(20).to(torch.bfloat16)
    dY[5] = 0
    bf = dict(dtype=torch.bfloat16, device="cuda")
    a_dYp, b_dYp = torch.full((R, d), float("nan"), **bf), torch.full((R, d), float("nan"), **bf)
    a_dg, b_dg = torch.empty(T, k, device="cuda"), torch.empty(T, k, device="cuda")
    ops.moe_combine_bwd(dev(dY), dev(Y_perm), dev(gate), P["slot_to_row"], P["row_offsets"],
                        P["perm_token"], a_dYp, a_dg)
    q = torch.full((R, d), 0x7F, dtype=torch.uint8, device="cuda")
    sq = torch.full((R,), float("nan"), device="cuda")
    ops.moe_combine_bwd_fp8(dev(dY), dev(Y_perm), dev(gate), P["slot_to_row"], P["row_offsets"],
                            P["perm_token"], b_dYp, b_dg, q, sq)
    n = int(P["row_offsets"][-1])
    q_ref = torch.empty(R, d, dtype=torch.uint8, device="cuda")
    s_ref = torch.empty(R, device="cuda")
    ops.moe_quantize_rows_fp8(a_dYp, P["row_offsets"][E:], q_ref, s_ref)
    torch.cuda.synchronize()
    assert torch.equal(a_dYp[:n], b_dYp[:n]) and torch.equal(a_dg, b_dg)
    assert torch.equal(q[:n], q_ref[:n])
    assert torch.equal(sq[:n], s_ref[:n])
