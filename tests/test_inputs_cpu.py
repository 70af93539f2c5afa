"""The seeded synthetic inputs follow their stated recipe: same seed, same bits; the stated
shapes, dtypes and distributions; the skewed workload's dead experts really get no tokens.
CPU only (the oracle's own routing decides the last point)."""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from pretraining_sigmoid_softmax_gb300.configs import CONFIGS, MoEConfig
from pretraining_sigmoid_softmax_gb300.inputs import ZIPF_DEAD, make_inputs

CFG = MoEConfig("recipe", T=4096, d=256, E=16, k=4, f=128, f_shared=64, mode="sigmoid",
                seed=5, backward=True, bias_update=True)


def test_same_seed_gives_the_same_bits_and_another_seed_does_not():
    a, b = make_inputs(CFG), make_inputs(CFG)
    assert a.keys() == b.keys()
    for name in a:
        assert torch.equal(a[name], b[name]), name
    c = make_inputs(CFG.with_(seed=6))
    assert not torch.equal(a["x"], c["x"])


def test_shapes_and_dtypes():
    t = make_inputs(CFG)
    T, d, E, f, fs = CFG.T, CFG.d, CFG.E, CFG.f, CFG.f_shared
    want = {"x": ((T, d), torch.bfloat16), "W_r": ((E, d), torch.float32),
            "b": ((E,), torch.float32), "W_g": ((E, f, d), torch.bfloat16),
            "W_u": ((E, f, d), torch.bfloat16), "W_d": ((E, d, f), torch.bfloat16),
            "Ws_g": ((fs, d), torch.bfloat16), "Ws_u": ((fs, d), torch.bfloat16),
            "Ws_d": ((d, fs), torch.bfloat16), "dY": ((T, d), torch.bfloat16)}
    assert set(t) == set(want)
    for name, (shape, dtype) in want.items():
        assert tuple(t[name].shape) == shape and t[name].dtype == dtype, name
    fwd_only = make_inputs(CFG.with_(backward=False, f_shared=0))
    assert "dY" not in fwd_only and "Ws_g" not in fwd_only


@pytest.mark.parametrize("name,std", [("x", 1.0), ("dY", 1.0), ("W_r", 256 ** -0.5),
                                      ("W_g", 256 ** -0.5), ("W_u", 256 ** -0.5),
                                      ("W_d", 128 ** -0.5), ("Ws_d", 64 ** -0.5)])
def test_normal_draws_have_the_stated_scale(name, std):
    v = make_inputs(CFG)[name].double().flatten()
    n = v.numel()
    # mean within 5 standard errors of 0, standard deviation within 3% (n >= 16k samples)
    assert abs(v.mean().item()) < 5 * std / math.sqrt(n)
    assert abs(v.std().item() / std - 1) < 0.03
    # Gaussian tails: about 4.6% of |v| beyond 2 std
    tail = (v.abs() > 2 * std).double().mean().item()
    assert 0.035 < tail < 0.057


def test_bias_is_uniform_in_its_range():
    b = make_inputs(CFG.with_(E=4096))["b"]
    assert b.min().item() >= -0.05 and b.max().item() <= 0.05
    assert abs(b.mean().item()) < 0.003 and abs(b.std().item() - 0.1 / math.sqrt(12)) < 0.002


def test_bf16_tensors_are_round_to_nearest_of_their_draws():
    """x is drawn in fp32 and rounded once: every value is a bf16 value and the rounding
    error is within half a bf16 ulp of the fp32 draw (re-drawn here with the same seed)."""
    g = torch.Generator().manual_seed(CFG.seed)
    raw = torch.randn((CFG.T, CFG.d), generator=g, dtype=torch.float32)
    x = make_inputs(CFG)["x"].float()
    np.testing.assert_array_equal(O.bf16_round(x.numpy().astype(np.float64)), x.numpy())
    err = (x - raw).abs()
    half_ulp = torch.ldexp(torch.ones_like(raw), torch.frexp(raw)[1] - 9)
    assert (err <= half_ulp).all()


def test_skewed_workload_leaves_its_dead_experts_without_tokens():
    """The skewed recipe zeroes ZIPF_DEAD router rows; under the oracle's own routing those
    experts receive no tokens and the live ones a heavy-tailed share."""
    cfg = CONFIGS["C3"].with_(T=8192)
    t = make_inputs(cfg, with_grad_input=False)
    W_r = t["W_r"].double().numpy()
    dead = np.where(~W_r.any(axis=1))[0]
    assert len(dead) == ZIPF_DEAD
    logits = O.router_logits(O.to64(t["x"]), W_r)
    r = O.route(logits, cfg.mode, cfg.k, O.to64(t["b"]), cfg.z_coef)
    counts = np.bincount(r["idx"].reshape(-1), minlength=cfg.E)
    assert (counts[dead] == 0).all()
    live = np.sort(counts[counts > 0])[::-1]
    assert live[0] > 10 * live[len(live) // 2]  # the top expert far above the median
