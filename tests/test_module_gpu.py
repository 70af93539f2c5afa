"""The user-facing autograd module ``MoELayer``: out, x.grad and every parameter's .grad after
``loss.backward()`` against the plain definition of the layer (the oracle's exact fp64 layer,
loss = <out, dY> plus the router z-loss with weight 1), the bias left without a gradient and
moved only by ``update_bias()``, and a stale backward refused."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from pretraining_sigmoid_softmax_gb300.configs import CONFIGS, MoEConfig
from pretraining_sigmoid_softmax_gb300.inputs import make_inputs
from pretraining_sigmoid_softmax_gb300.layer import MoELayer

from gpu_common import assert_close, check_plain, dx_summand_ulps, require_gpu

pytestmark = pytest.mark.gpu

SOFTMAX_ZLOSS = MoEConfig("module_softmax_zloss", T=1000, d=384, E=16, k=4, f=256, f_shared=0,
                          mode="softmax", seed=22, backward=True, bias_update=False, z_coef=1e-3)
SIGMOID_AUX = MoEConfig("module_sigmoid_aux_shared", T=1024, d=256, E=16, k=4, f=256,
                        f_shared=128, mode="sigmoid", seed=23, backward=True, bias_update=True,
                        aux_switch=1e-2, aux_seq=2e-2, seq_len=256)
# experts long enough (d_ff 768) for the router's input-gradient term to ride in the dX rows
SIGMOID_ROWS = MoEConfig("module_sigmoid_router_rows", T=512, d=256, E=4, k=2, f=768,
                         f_shared=256, mode="sigmoid", seed=28, backward=True, bias_update=True)


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _module(cfg, inp):
    layer = MoELayer(cfg.d, cfg.E, cfg.k, cfg.f, cfg.f_shared, cfg.mode, cfg.z_coef, cfg.gamma,
                     device="cuda", bias_rule=cfg.bias_rule, aux_switch=cfg.aux_switch,
                     aux_seq=cfg.aux_seq, seq_len=cfg.seq_len)
    with torch.no_grad():
        for name in ("W_r", "b", "W_g", "W_u", "W_d", "Ws_g", "Ws_u", "Ws_d"):
            if name in inp:
                getattr(layer, name).copy_(inp[name])
    return layer


@pytest.mark.parametrize("cfg", [CONFIGS["C1"], SOFTMAX_ZLOSS, SIGMOID_AUX, SIGMOID_ROWS],
                         ids=lambda c: c.name)
def test_module_backward_matches_the_plain_definition(cfg):
    inp = make_inputs(cfg)
    layer = _module(cfg, inp)
    x = inp["x"].cuda().requires_grad_(True)
    dY = inp["dY"].cuda()
    out = layer(x)
    loss = (out.float() * dY.float()).sum()  # d loss / d out = dY exactly
    loss.backward()
    torch.cuda.synchronize()
    plan = layer._last_plan
    assert plan.router_rows == (cfg.name == SIGMOID_ROWS.name)
    idx = plan.topk_idx.cpu().numpy().astype(np.int64)
    i64 = {k: O.to64(v) for k, v in inp.items() if k != "dY"}
    aux = (cfg.seq_len, cfg.aux_switch, cfg.aux_seq) if cfg.has_aux else None
    P = O.layer_forward(i64, cfg.mode, cfg.k, cfg.z_coef, idx=idx, aux=aux)
    S = O.layer_forward(i64, cfg.mode, cfg.k, cfg.z_coef, idx=idx, rnd=O.bf16_round, aux=aux,
                        fold_gate=True, router_rows=plan.router_rows)
    dY64 = O.to64(inp["dY"])
    PB, SB = O.layer_backward(i64, P, dY64), O.layer_backward(i64, S, dY64)
    case = "module " + cfg.name
    check_plain(case, "out", out.detach(), P["out"], S["out"])
    check_plain(case, "dx", x.grad, PB["dx"], SB["dx"])
    assert_close(x.grad, SB["dx"], "dx", extra=dx_summand_ulps(S, SB))
    grads = {"W_r": "dW_r", "W_g": "dW_g", "W_u": "dW_u", "W_d": "dW_d"}
    if cfg.f_shared:
        grads.update(Ws_g="dWs_g", Ws_u="dWs_u", Ws_d="dWs_d")
    for p, g in grads.items():
        got = getattr(layer, p).grad
        assert got is not None and got.dtype == getattr(layer, p).dtype, p
        check_plain(case, g, got, PB[g], SB[g])
        assert_close(got, SB[g], g, reduction=True)
    if cfg.mode == "softmax":
        assert float(layer.z_loss()[0]) == pytest.approx(P["z_loss"], rel=1e-4)
    if aux is not None:
        assert float(layer.aux_loss()[0]) == pytest.approx(P["aux_switch"], rel=1e-5)
        assert float(layer.aux_loss()[1]) == pytest.approx(P["aux_seq"], rel=1e-5)
    # the bias gets no gradient and moves only by the update, with this step's counts
    assert layer.b.grad is None and not layer.b.requires_grad
    assert torch.equal(layer.b.cpu(), inp["b"])
    layer.update_bias()
    if cfg.mode == "sigmoid":
        rule = O.bias_update_proportional if cfg.bias_rule == "proportional" else O.bias_update
        want = rule(P["counts"], inp["b"].numpy(), cfg.T, cfg.k, cfg.gamma)
        assert np.array_equal(layer.b.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:  # softmax routing has no bias
        assert torch.equal(layer.b.cpu(), inp["b"])


def test_module_refuses_a_backward_whose_activations_were_overwritten():
    cfg = SOFTMAX_ZLOSS
    inp = make_inputs(cfg)
    layer = _module(cfg, inp)
    x = inp["x"].cuda()
    out1 = layer(x)
    out2 = layer(x)
    with pytest.raises(RuntimeError, match="overwrote its saved activations"):
        out1.float().sum().backward()
    out2.float().sum().backward()  # the latest forward's backward still runs
    torch.cuda.synchronize()
    assert layer.W_g.grad is not None


def test_module_rejects_a_wrong_input():
    cfg = SOFTMAX_ZLOSS
    layer = _module(cfg, make_inputs(cfg))
    with pytest.raises(ValueError):
        layer(torch.zeros(8, cfg.d, device="cuda"))  # fp32
    with pytest.raises(ValueError):
        layer(torch.zeros(8, cfg.d + 1, dtype=torch.bfloat16, device="cuda"))
