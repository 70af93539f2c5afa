"""Whole-layer parity (forward, backward, bias update) of the CUDA path against the fp64
oracle on the workloads and on small ragged shapes, through the C ABI.

Every value check has two parts. Parity proper compares the GPU with the plain definition
(the oracle's exact fp64 layer, nothing rounded, its own fp64 router logits and the GPU's
choice of experts) at the literal tolerance |gpu - oracle| <= 1e-2 + 1e-2 |oracle|, and
reports the elements outside it per tensor (``check_plain``). A second check holds the
kernels' arithmetic to the oracle's bf16-storage model (the tensors the workloads store in
bf16 rounded where they are stored), which is tighter on everything but the sums over tokens.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from pretraining_sigmoid_softmax_gb300 import ops
from pretraining_sigmoid_softmax_gb300.configs import CONFIGS, MoEConfig
from pretraining_sigmoid_softmax_gb300.inputs import make_inputs, make_upstream_gate_grad
from pretraining_sigmoid_softmax_gb300.layer import MoEPlan, MoEShape

from gpu_common import (assert_close, check_plain, dx_summand_ulps, gpu_rows, h64,
                        padded_offsets, record_near_ties, require_gpu)

# FP8 operands: the fraction of elements the storage-model check lets a bf16 neighbour of h
# move past its bound by rounding to the next E4M3 code (every element of the affected rows)
FP8_CODE_FLIPS = 1e-3

pytestmark = pytest.mark.gpu
RND = O.bf16_round


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def oracle_bias(cfg):
    return O.bias_update_proportional if cfg.bias_rule == "proportional" else O.bias_update


def run_gpu(cfg: MoEConfig, inp: dict):
    plan = MoEPlan(MoEShape.from_config(cfg), "cuda", backward=cfg.backward)
    d = {k: v.cuda() for k, v in inp.items()}
    ops.moe_clear_device_status()
    plan.forward(d["x"], d["W_r"], d["b"], d["W_g"], d["W_u"], d["W_d"], d.get("Ws_g"),
                 d.get("Ws_u"), d.get("Ws_d"))
    b_new = None
    if cfg.backward:
        plan.backward(d["dY"])
        if cfg.bias_update:
            b_new = d["b"].clone()
            plan.bias_update(b_new, cfg.gamma, cfg.bias_rule)
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    return plan, b_new


def check_routing(cfg, inp, plan):
    """Bit-exact choice against the oracle replayed on the GPU's fp32 logits; returns the
    GPU choice and logits (fp64)."""
    lg = h64(plan.logits)
    b64 = h64(inp["b"])
    ref = O.route(lg, cfg.mode, cfg.k, b64, cfg.z_coef)
    near = (O.near_tie_tokens(ref["select_value"], cfg.k) if cfg.mode == "sigmoid"
            else np.zeros(cfg.T, bool))
    idx = plan.topk_idx.cpu().numpy().astype(np.int64)
    assert (idx[~near] == ref["idx"][~near]).all(), "expert choice differs from the oracle"
    assert near.mean() < 0.01, f"near-tie tokens {near.sum()}"
    # dispatch of the GPU's choice: counts, offsets and permutation bit-exact
    D = O.dispatch(idx, cfg.E)
    assert (plan.counts.cpu().numpy() == D["counts"]).all()
    assert (plan.offsets.cpu().numpy() == D["offsets"]).all()
    ro = plan.row_offsets.cpu().numpy()
    assert (ro == padded_offsets(D["counts"])).all()
    rows = gpu_rows(D["offsets"], ro)
    assert (plan.perm_token.cpu().numpy()[rows] == D["perm_token"]).all()
    assert (plan.slot_to_row.cpu().numpy() == rows[D["slot_to_row"]]).all()
    return idx, lg, D, rows, int(near.sum())


def dlogits_atol(bwd):
    """Absolute term of the storage check of the logit gradient. It is linear in the gate
    gradient dg with coefficients of magnitude at most 1 (softmax: p_j (delta_j - p_i);
    sigmoid: s (1 - s) (delta - g) / sum of the chosen s), so it inherits dg's absolute
    error: twice dg's absolute term, 1e-2 max(1, rms(dg))."""
    dg = np.asarray(bwd["dg"])
    return 2.0 * 1e-2 * max(1.0, float(np.sqrt(np.mean(dg * dg)))) if dg.size else 1e-2


def both(plain, storage):
    """The plain-definition and bf16-storage oracle evaluations side by side in two threads
    (numpy's elementwise work releases the GIL); returns their results in that order."""
    with ThreadPoolExecutor(2) as ex:
        a, b = ex.submit(plain), ex.submit(storage)
        return a.result(), b.result()


def _aux(cfg):
    return (cfg.seq_len or cfg.T, cfg.aux_switch, cfg.aux_seq) if cfg.has_aux else None


def _replayed_gates(cfg, lg, idx, b):
    """Gates of the GPU's choice from the given logits."""
    r = O.route(lg, cfg.mode, cfg.k, b, cfg.z_coef)
    return O._regate(r, lg, idx, cfg.mode, b, cfg.z_coef)


def full_parity(cfg, inp):
    plan, b_new = run_gpu(cfg, inp)
    idx, lg, D, rows, near = check_routing(cfg, inp, plan)
    record_near_ties(cfg.name, near, cfg.T)
    i64 = {k: O.to64(v) for k, v in inp.items() if k != "dY"}
    aux = _aux(cfg)
    fp8, f8d = cfg.fp8, cfg.fp8_dgrad
    # gates of the GPU's fp32 logits: fp32-tight
    assert_close(plan.topk_gate, _replayed_gates(cfg, lg, idx, i64["b"])["gate"], "gates",
                 atol=1e-6, rtol=1e-5)
    # the plain definition and the bf16-storage model (the bf16 layer folds each slot's gate
    # into its expert: the stored h and y carry the gate)
    dY = O.to64(inp["dY"]) if cfg.backward else None

    def run(**kw):
        fwd = O.layer_forward(i64, cfg.mode, cfg.k, cfg.z_coef, idx=idx, aux=aux, fp8=fp8,
                              fp8_dgrad=f8d, **kw)
        return fwd, (O.layer_backward(i64, fwd, dY) if cfg.backward else None)

    # the storage model: bf16 rows, the gate folded into the bf16 layer's experts, and the
    # router's input-gradient term in the rows where the plan puts it there
    (P, PB), (S, SB) = both(lambda: run(), lambda: run(rnd=RND, fold_gate=not fp8,
                                                       router_rows=plan.router_rows))
    case = cfg.name
    assert_close(plan.X_perm[torch.from_numpy(rows).cuda()], P["X_perm"], "X_perm", 0, 0)
    check_plain(case, "logits", plan.logits, P["logits"], S["logits"])
    check_plain(case, "gates", plan.topk_gate, P["gate"], S["gate"])
    flips = FP8_CODE_FLIPS if fp8 else 0.0
    check_plain(case, "out", plan.out, P["out"], S["out"])
    assert_close(plan.out, S["out"], "out", allow_frac=flips)
    if aux is not None:
        assert float(plan.aux_loss[0]) == pytest.approx(P["aux_switch"], rel=1e-5)
        assert float(plan.aux_loss[1]) == pytest.approx(P["aux_seq"], rel=1e-5)
    if cfg.mode == "softmax":
        check_plain(case, "lse", plan.lse, P["lse"], S["lse"])
        assert float(plan.z_loss[0]) == pytest.approx(P["z_loss"], rel=1e-4)
    if not cfg.backward:
        return
    names = ["dx", "dg", "dlogits", "dW_r", "dW_g", "dW_u", "dW_d"]
    if cfg.f_shared:
        names += ["dWs_g", "dWs_u", "dWs_d"]
    for name in names:
        got = getattr(plan, name)
        check_plain(case, name, got, PB[name], SB[name])
        if name == "dx":
            assert_close(got, SB[name], name, extra=dx_summand_ulps(S, SB), allow_frac=flips)
        elif name == "dlogits":
            assert_close(got, SB[name], name, atol=dlogits_atol(SB), allow_frac=flips)
        else:  # sums over tokens, or (dg) over the features of bf16 rows
            assert_close(got, SB[name], name, reduction=True, allow_frac=flips)
    if cfg.bias_update:
        ref = oracle_bias(cfg)(D["counts"], inp["b"].numpy(), cfg.T, cfg.k, cfg.gamma)
        assert np.array_equal(b_new.cpu().numpy().view(np.uint32), ref.view(np.uint32))


SMALL = [
    MoEConfig("ragged_sigmoid_shared", T=300, d=256, E=6, k=3, f=128, f_shared=128,
              mode="sigmoid", seed=11, backward=True, bias_update=True),
    MoEConfig("ragged_softmax", T=1000, d=384, E=16, k=4, f=256, f_shared=0, mode="softmax",
              seed=12, backward=True, bias_update=False, z_coef=1e-3),
    MoEConfig("one_expert_top1", T=200, d=128, E=1, k=1, f=128, f_shared=0, mode="sigmoid",
              seed=13, backward=True, bias_update=True),
    MoEConfig("k_equals_E", T=130, d=128, E=4, k=4, f=128, f_shared=128, mode="softmax",
              seed=14, backward=True, bias_update=False, z_coef=1e-2),
    MoEConfig("skewed_small", T=2048, d=256, E=32, k=4, f=128, f_shared=0, mode="sigmoid",
              seed=15, backward=True, bias_update=False, zipf=True),
    MoEConfig("aux_losses_sigmoid", T=1024, d=256, E=16, k=4, f=256, f_shared=128,
              mode="sigmoid", seed=16, backward=True, bias_update=True, aux_switch=1e-2,
              aux_seq=2e-2, seq_len=256),
    MoEConfig("aux_losses_softmax", T=768, d=256, E=8, k=2, f=128, f_shared=0, mode="softmax",
              seed=17, backward=True, bias_update=False, z_coef=1e-3, aux_switch=1e-2,
              aux_seq=1e-2, seq_len=384),
    MoEConfig("fp8_forward_shared", T=1024, d=512, E=8, k=2, f=256, f_shared=256,
              mode="sigmoid", seed=18, backward=True, bias_update=True, precision="fp8"),
    MoEConfig("fp8_forward_softmax_ragged", T=777, d=256, E=5, k=2, f=128, f_shared=0,
              mode="softmax", seed=21, backward=True, bias_update=False, z_coef=1e-3,
              precision="fp8"),
    MoEConfig("fp8_dgrad_shared", T=1024, d=512, E=8, k=2, f=256, f_shared=256,
              mode="sigmoid", seed=24, backward=True, bias_update=True, precision="fp8_dgrad"),
    MoEConfig("fp8_dgrad_softmax_ragged", T=777, d=384, E=5, k=2, f=128, f_shared=0,
              mode="softmax", seed=25, backward=True, bias_update=False, z_coef=1e-3,
              precision="fp8_dgrad"),
    # fewer tokens than one tile row block: 7-row tensors behind 32- and 128-row boxes
    MoEConfig("sub_tile_T7", T=7, d=128, E=4, k=2, f=128, f_shared=128, mode="sigmoid",
              seed=19, backward=True, bias_update=True),
    # experts long enough (d_ff 768) for the router's input-gradient term to ride in their
    # dX rows
    MoEConfig("router_term_in_rows", T=400, d=256, E=5, k=2, f=768, f_shared=256,
              mode="sigmoid", seed=26, backward=True, bias_update=True),
    MoEConfig("fp8_dgrad_router_term_in_rows", T=400, d=256, E=4, k=2, f=768, f_shared=256,
              mode="sigmoid", seed=27, backward=True, bias_update=True, precision="fp8_dgrad"),
    # the widest router (SIMT logits and W_r gradient), most experts with 0-3 rows
    MoEConfig("widest_router_E256", T=300, d=256, E=256, k=8, f=128, f_shared=0,
              mode="softmax", seed=20, backward=True, bias_update=False, z_coef=1e-3),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_small_layers_full_parity(cfg):
    full_parity(cfg, make_inputs(cfg))


def test_single_expert_router_gets_zero_gradient():
    """One expert with top-1: the gate is 1 and the router weight gradient is exactly 0."""
    cfg = SMALL[2]
    plan, _ = run_gpu(cfg, make_inputs(cfg))
    assert (plan.topk_gate == 1).all()
    assert (plan.dW_r == 0).all()


@pytest.mark.parametrize("name", ["C0", "C1", "C2"])
def test_workload_full_parity(name):
    cfg = CONFIGS[name]
    full_parity(cfg, make_inputs(cfg))


def test_layer_is_bitwise_repeatable():
    cfg = CONFIGS["C1"]
    inp = make_inputs(cfg)
    p1, _ = run_gpu(cfg, inp)
    r1 = {k: v.clone() for k, v in p1.grads().items()}
    o1 = p1.out.clone()
    p2, _ = run_gpu(cfg, inp)
    assert torch.equal(o1, p2.out)
    for k, v in p2.grads().items():
        assert torch.equal(r1[k], v), k


SAMPLED_TOKENS = 2048
SHARED_UNITS = 16


@pytest.mark.parametrize("name", ["C3", "C4", "C5", "C6", "C7", "C8"])
def test_workload_sampled_parity(name):
    """Full-size workloads in the benchmark's launch configuration, against a stratified
    subset of the oracle: routing, counts and permutation in full; out, dx, the gate and
    logit gradients on 2,048 fixed-seed tokens plus the first and last; the whole weight
    gradients of the most-loaded expert and of the least-loaded live one (a handful of rows
    in the skewed workload); exactly zero weight gradients for every empty expert; whole
    weight rows of 16 shared-expert units."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    plan, b_new = run_gpu(cfg, inp)
    idx, lg, D, rows, near = check_routing(cfg, inp, plan)
    record_near_ties(cfg.name, near, cfg.T)
    case = cfg.name
    fp8, f8d = cfg.fp8, cfg.fp8_dgrad
    W64 = {k: O.to64(v) for k, v in inp.items() if k not in ("x", "dY")}
    x64, dY64 = O.to64(inp["x"]), O.to64(inp["dY"])
    lg64 = O.router_logits(x64, W64["W_r"])
    R = _replayed_gates(cfg, lg64, idx, W64["b"])
    rng = np.random.default_rng(cfg.seed)
    toks = np.unique(np.concatenate([[0, cfg.T - 1],
                                     rng.choice(cfg.T, SAMPLED_TOKENS, replace=False)]))
    tt = torch.from_numpy(toks).cuda()
    dl_aux = None
    if cfg.has_aux:  # batch-wide losses: compared in full, their gradient rows feed dx
        a = O.aux_losses(lg64, idx, cfg.mode, cfg.seq_len, cfg.aux_switch, cfg.aux_seq)
        assert float(plan.aux_loss[0]) == pytest.approx(a["switch"], rel=1e-5)
        assert float(plan.aux_loss[1]) == pytest.approx(a["seq"], rel=1e-5)
        dl_aux = O.aux_losses_backward(lg64, idx, cfg.mode, cfg.seq_len, cfg.aux_switch,
                                       cfg.aux_seq)[toks]
    # the layer over the sampled tokens: each token's out and dx depend only on its own
    # routing; the z-loss mean and the balancing losses are the whole batch's
    part = dict(W64, x=x64[toks])

    def run(**kw):
        fwd = O.layer_forward(part, cfg.mode, cfg.k, cfg.z_coef, logits=lg64[toks], idx=idx[toks],
                              fp8=fp8, fp8_dgrad=f8d, **kw)
        return fwd, O.layer_backward(part, fwd, dY64[toks], T_norm=cfg.T, dl_extra=dl_aux,
                                     weight_grads=False)

    # the storage model: bf16 rows, the gate folded into the bf16 layer's experts, and the
    # router's input-gradient term in the rows where the plan puts it there
    (P, PB), (S, SB) = both(lambda: run(), lambda: run(rnd=RND, fold_gate=not fp8,
                                                       router_rows=plan.router_rows))
    flips = FP8_CODE_FLIPS if fp8 else 0.0
    check_plain(case, "gates", plan.topk_gate[tt], P["gate"], S["gate"])
    check_plain(case, "out", plan.out[tt], P["out"], S["out"])
    assert_close(plan.out[tt], S["out"], "out", allow_frac=flips)
    for nm in ("dx", "dg", "dlogits"):
        got = getattr(plan, nm)[tt]
        check_plain(case, nm, got, PB[nm], SB[nm])
        if nm == "dx":
            assert_close(got, SB[nm], nm, extra=dx_summand_ulps(S, SB), allow_frac=flips)
        elif nm == "dlogits":
            assert_close(got, SB[nm], nm, atol=dlogits_atol(SB), allow_frac=flips)
        else:
            assert_close(got, SB[nm], nm, reduction=True, allow_frac=flips)
    # whole weight gradients of chosen experts
    counts = D["counts"]
    live = np.nonzero(counts)[0]
    for e in sorted({int(live[np.argmax(counts[live])]), int(live[np.argmin(counts[live])])}):
        lo, hi = int(D["offsets"][e]), int(D["offsets"][e + 1])
        tok_e = D["perm_token"][lo:hi]
        gates = R["gate"][tok_e, D["perm_slot"][lo:hi]]
        Pw, Sw = both(
            lambda: O.expert_weight_grads(W64, e, x64[tok_e], gates, dY64[tok_e], fp8=fp8,
                                          fp8_dgrad=f8d),
            lambda: O.expert_weight_grads(W64, e, x64[tok_e], gates, dY64[tok_e], rnd=RND,
                                          fp8=fp8, fold_gate=not fp8, fp8_dgrad=f8d))
        for nm in ("dW_g", "dW_u", "dW_d"):
            got = getattr(plan, nm)[e]
            check_plain(case, f"{nm}[{e}]", got, Pw[nm], Sw[nm])
            assert_close(got, Sw[nm], f"{nm}[{e}]", reduction=True)
    for e in np.nonzero(counts == 0)[0]:
        for nm in ("dW_g", "dW_u", "dW_d"):
            assert (getattr(plan, nm)[int(e)] == 0).all()
    if cfg.zipf:
        assert (counts == 0).sum() >= 10
    if cfg.f_shared:
        units = np.sort(rng.choice(cfg.f_shared, SHARED_UNITS, replace=False))
        sh = {"x": x64, "Ws_g": W64["Ws_g"], "Ws_u": W64["Ws_u"], "Ws_d": W64["Ws_d"]}
        Pu, Su = both(
            lambda: O.shared_weight_grad_units(sh, dY64, units, fp8=fp8, fp8_dgrad=f8d),
            lambda: O.shared_weight_grad_units(sh, dY64, units, rnd=RND, fp8=fp8, fp8_dgrad=f8d))
        ut = torch.from_numpy(units).cuda()
        for nm, got in (("dWs_g", plan.dWs_g[ut]), ("dWs_u", plan.dWs_u[ut]),
                        ("dWs_d", plan.dWs_d[:, ut])):
            check_plain(case, nm, got, Pu[nm], Su[nm])
            assert_close(got, Su[nm], nm, reduction=True)
    if cfg.bias_update:
        refb = oracle_bias(cfg)(counts, inp["b"].numpy(), cfg.T, cfg.k, cfg.gamma)
        assert np.array_equal(b_new.cpu().numpy().view(np.uint32), refb.view(np.uint32))


def test_router_backward_at_full_size():
    """Router backward of the largest workload with a synthetic gate gradient."""
    cfg = CONFIGS["C4"]
    g = torch.Generator().manual_seed(cfg.seed)
    x = (torch.randn(cfg.T, cfg.d, generator=g)).to(torch.bfloat16)
    W_r = torch.randn(cfg.E, cfg.d, generator=g) * cfg.d ** -0.5
    b = torch.rand(cfg.E, generator=g) * 0.1 - 0.05
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    f32 = dict(device="cuda", dtype=torch.float32)
    logits, gate, score = torch.empty(T, E, **f32), torch.empty(T, k, **f32), torch.empty(T, k, **f32)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    dl, dW_r = torch.empty(T, E, **f32), torch.empty(E, d, **f32)
    ws = torch.empty(ops.moe_workspace_bytes(T, d, E, k), dtype=torch.uint8, device="cuda")
    xd, Wd = x.cuda(), W_r.cuda()
    ops.moe_route(xd, Wd, b.cuda(), k, ops.MODE_SIGMOID, 0.0, logits, idx, gate, score, None,
                  None, ws)
    dg = make_upstream_gate_grad(T, k, cfg.seed)
    ops.moe_route_bwd(dg.cuda(), xd, idx, gate, score, None, None, E, ops.MODE_SIGMOID, 0.0, dl,
                      dW_r, ws)
    torch.cuda.synchronize()

    class _P:
        pass
    plan = _P()
    plan.logits, plan.topk_idx, plan.dlogits, plan.dW_r = logits, idx, dl, dW_r
    lg = h64(plan.logits)
    ref = O.route(lg, "sigmoid", cfg.k, O.to64(b))
    ref = O._regate(ref, lg, plan.topk_idx.cpu().numpy(), "sigmoid", O.to64(b), 0.0)
    rb = O.router_backward(O.to64(dg), ref, O.to64(x), O.to64(W_r), "sigmoid", 0.0)
    assert_close(plan.dlogits, rb["dlogits"], "dlogits", atol=1e-5, rtol=1e-4)
    assert_close(plan.dW_r, rb["dW_r"], "dW_r")  # the literal tolerance
    assert_close(plan.dW_r, rb["dW_r"], "dW_r", atol=1e-3, rtol=1e-3, reduction=True)


def test_cuda_graph_replay_matches_eager_step():
    """A whole step captured as one CUDA graph and replayed gives the eager step's bits."""
    cfg = CONFIGS["C1"]
    inp = make_inputs(cfg)
    p_eager, b_eager = run_gpu(cfg, inp)
    d = {k: v.cuda() for k, v in inp.items()}
    plan = MoEPlan(MoEShape.from_config(cfg), "cuda", backward=True)
    b = d["b"].clone()
    weights = {k: d[k] for k in ("W_r", "W_g", "W_u", "W_d", "Ws_g", "Ws_u", "Ws_d")}
    graph = plan.capture_step(d["x"], weights, d["dY"], b, cfg.gamma, cfg.bias_rule, True,
                              warmup=1)
    b.copy_(d["b"])  # capture ran one warm-up step that moved the bias
    graph.replay()
    torch.cuda.synchronize()
    assert ops.moe_device_status()[0] == 0
    assert torch.equal(plan.out, p_eager.out)
    for k, v in plan.grads().items():
        assert torch.equal(v, p_eager.grads()[k]), k
    assert torch.equal(b, b_eager)


LAUNCH_CASES = [CONFIGS["C1"], CONFIGS["C2"]] + [
    c for c in SMALL if c.name in ("aux_losses_sigmoid", "aux_losses_softmax", "fp8_forward_shared",
                                   "fp8_dgrad_shared", "widest_router_E256", "one_expert_top1",
                                   "router_term_in_rows", "fp8_dgrad_router_term_in_rows")]


@pytest.mark.parametrize("cfg", LAUNCH_CASES, ids=lambda c: c.name)
def test_launch_count_matches_the_plan(cfg):
    """The bench's gpu_launches is launches_per_step times the steps: count the library's
    kernels that one step actually runs (CUDA activity of the profiler, kernels of the moe
    namespace; the profiler's own and torch's kernels are not the library's)."""
    from torch.autograd import DeviceType
    from torch.profiler import ProfilerActivity, profile
    inp = make_inputs(cfg)
    d = {k: v.cuda() for k, v in inp.items()}
    plan = MoEPlan(MoEShape.from_config(cfg), "cuda", backward=cfg.backward)
    b = d["b"].clone()

    def step():
        plan.forward(d["x"], d["W_r"], b, d["W_g"], d["W_u"], d["W_d"], d.get("Ws_g"),
                     d.get("Ws_u"), d.get("Ws_d"))
        if cfg.backward:
            plan.backward(d["dY"])
            if cfg.bias_update:
                plan.bias_update(b, cfg.gamma, cfg.bias_rule)

    step()  # every kernel loaded before the counted step
    torch.cuda.synchronize()
    kernels = []
    for _ in range(2):  # the profiler's first session in a process may record no activity
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            step()
            torch.cuda.synchronize()
        kernels = [e.name for e in prof.events() if e.device_type == DeviceType.CUDA]
        if kernels:
            break
    if not kernels:
        pytest.skip("the profiler recorded no CUDA activity on this machine")
    ours = [n for n in kernels if "moe::" in n]
    want = plan.launches_per_step(cfg.backward, cfg.bias_update)
    counts = {}
    for n in ours:
        key = n.split("(")[0].replace("(anonymous namespace)::", "")
        counts[key] = counts.get(key, 0) + 1
    assert len(ours) == want, (len(ours), want, counts)
