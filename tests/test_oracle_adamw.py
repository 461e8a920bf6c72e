"""Pins for the oracle's AdamW step with global gradient-norm clipping
(walkthrough, "Stage 8"), each tying it to something other than itself:

* PyTorch's own optimizer and clipping routines (``torch.optim.AdamW``,
  ``torch.nn.utils.clip_grad_norm_``) run in float64 over several steps, with
  the projection matrices in a decayed group and the rest undecayed;
* closed forms: Adam's first step is lr * g / (|g| + eps); a constant
  gradient keeps the bias-corrected moments at g and g^2, so the weights
  follow a geometric recurrence; a zero gradient leaves only the decay;
  without eps the step is scale-free;
* the clip coefficient on a (3, 4) gradient, and when clipping is off;
* the sharded norm (each rank's FFN slices, replicated parameters counted on
  rank 0 only) equals the dense norm for every t, and counting the
  replicated ones on every rank overshoots by exactly (t - 1) times their
  squared norm.
"""
import math

import numpy as np
import pytest

from oracle import tpmlp_oracle as O

torch = pytest.importorskip("torch")


def _params(seed, H, F, act):
    rng = np.random.default_rng(seed)
    p = {"norm_w": 1.0 + 0.1 * rng.standard_normal(H), "w_down": 0.3 * rng.standard_normal((H, F)),
         "b_down": 0.05 * rng.standard_normal(H)}
    if act == "swiglu":
        p["w_gate_up"] = 0.3 * rng.standard_normal((2, F, H))
    else:
        p["w_1"] = 0.3 * rng.standard_normal((F, H))
        p["b_1"] = 0.05 * rng.standard_normal(F)
    return p, rng


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("max_norm", [0.0, 1e9, 0.05])
def test_adamw_matches_torch_optimizer(act, max_norm):
    p, rng = _params(7, 8, 12, act)
    hp = dict(lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, max_grad_norm=max_norm)
    names = list(p)
    tp = {k: torch.tensor(p[k], dtype=torch.float64, requires_grad=True) for k in names}
    decayed = [tp[k] for k in names if k in O.DECAYED]
    rest = [tp[k] for k in names if k not in O.DECAYED]
    opt = torch.optim.AdamW([{"params": decayed, "weight_decay": hp["weight_decay"]},
                             {"params": rest, "weight_decay": 0.0}],
                            lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"], foreach=False)
    cur = {k: p[k].copy() for k in names}
    m = {k: np.zeros_like(p[k]) for k in names}
    v = {k: np.zeros_like(p[k]) for k in names}
    for step in range(1, 5):
        g = {k: 0.2 * rng.standard_normal(p[k].shape) for k in names}
        for k in names:
            tp[k].grad = torch.tensor(g[k], dtype=torch.float64)
        tnorm = None
        if max_norm > 0:
            tnorm = float(torch.nn.utils.clip_grad_norm_([tp[k] for k in names], max_norm))
        opt.step()
        out = O.adamw(cur, g, m, v, step, **hp)
        cur, m, v = out["params"], out["m"], out["v"]
        if tnorm is not None:
            assert out["grad_norm"] == pytest.approx(tnorm, rel=1e-14)
        for k in names:
            np.testing.assert_allclose(cur[k], tp[k].detach().numpy(), rtol=1e-13, atol=1e-15)
    if max_norm == 0.05:
        assert out["clip"] < 1.0  # the clipped branch ran
    else:
        assert out["clip"] == 1.0


def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((5, 7))
    g = rng.standard_normal((5, 7)) * np.logspace(-9, -3, 7)
    lr, eps = 1e-3, 1e-8
    out = O.adamw({"w_down": w}, {"w_down": g}, {"w_down": np.zeros_like(w)}, {"w_down": np.zeros_like(w)}, 1,
                  lr=lr, beta1=0.9, beta2=0.999, eps=eps, weight_decay=0.0, max_grad_norm=0.0)
    np.testing.assert_allclose(out["params"]["w_down"], w - lr * g / (np.abs(g) + eps), rtol=1e-12, atol=0)
    np.testing.assert_allclose(out["m"]["w_down"], 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(out["v"]["w_down"], 0.001 * g * g, rtol=1e-13)


def test_adamw_constant_gradient_recurrence():
    # With g fixed, m_k = g (1 - b1^k) and v_k = g^2 (1 - b2^k), so the
    # corrected moments are g and g^2 at every step and each update is
    # w <- (1 - lr wd) w - lr s with s = g / (|g| + eps).
    w0 = np.array([0.5, -0.25, 2.0, 0.0])
    g = np.array([1e-4, -3e-6, 0.0, 2.0])
    lr, wd, eps, K = 0.01, 0.1, 1e-8, 6
    p, m, v = {"w_gate_up": w0}, {"w_gate_up": np.zeros(4)}, {"w_gate_up": np.zeros(4)}
    for k in range(1, K + 1):
        out = O.adamw(p, {"w_gate_up": g}, m, v, k, lr=lr, beta1=0.9, beta2=0.999, eps=eps,
                      weight_decay=wd, max_grad_norm=0.0)
        p, m, v = out["params"], out["m"], out["v"]
        np.testing.assert_allclose(m["w_gate_up"], g * (1 - 0.9 ** k), rtol=1e-13)
        np.testing.assert_allclose(v["w_gate_up"], g * g * (1 - 0.999 ** k), rtol=1e-12)
    s = g / (np.abs(g) + eps)
    a = 1.0 - lr * wd
    expect = a ** K * w0 - lr * s * (1 - a ** K) / (1 - a)
    np.testing.assert_allclose(p["w_gate_up"], expect, rtol=1e-12, atol=1e-15)


def test_adamw_zero_gradient_is_pure_decay():
    w = np.array([[1.0, -2.0], [0.5, 3.0]])
    b = np.array([0.25, -0.75])
    z = {"w_down": np.zeros_like(w), "b_down": np.zeros_like(b)}
    out = O.adamw({"w_down": w, "b_down": b}, z, dict(z), dict(z), 1, lr=0.1, beta1=0.9, beta2=0.999,
                  eps=1e-8, weight_decay=0.2, max_grad_norm=1.0)
    np.testing.assert_array_equal(out["params"]["w_down"], w - 0.1 * 0.2 * w)
    np.testing.assert_array_equal(out["params"]["b_down"], b)  # vectors are not decayed
    assert out["grad_norm"] == 0.0 and out["clip"] == 1.0


def test_adamw_attention_parameters_decay_like_the_mlp_ones():
    # the attention sublayer's projection matrices (W_qkv, W_out) decay, its
    # norm weight and output bias do not: zero gradient and moments leave
    # exactly w (1 - lr wd) or w
    rng = np.random.default_rng(5)
    p = {"norm_w": rng.standard_normal(4), "w_qkv": rng.standard_normal((6, 4)),
         "w_o": rng.standard_normal((4, 2)), "b_o": rng.standard_normal(4)}
    z = {k: np.zeros_like(v) for k, v in p.items()}
    out = O.adamw(p, z, dict(z), dict(z), 3, lr=0.05, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.4,
                  max_grad_norm=1.0)
    for k in ("w_qkv", "w_o"):
        np.testing.assert_array_equal(out["params"][k], p[k] - 0.05 * 0.4 * p[k])
    for k in ("norm_w", "b_o"):
        np.testing.assert_array_equal(out["params"][k], p[k])


def test_adam_step_is_scale_free_without_eps():
    rng = np.random.default_rng(11)
    w = rng.standard_normal(9)
    g1, g2 = rng.standard_normal(9), rng.standard_normal(9)
    z = np.zeros(9)
    outs = []
    for scale in (1.0, 1e-6):
        o1 = O.adamw({"norm_w": w}, {"norm_w": scale * g1}, {"norm_w": z}, {"norm_w": z}, 1, lr=0.1, beta1=0.9,
                     beta2=0.999, eps=0.0, weight_decay=0.0, max_grad_norm=0.0)
        o2 = O.adamw(o1["params"], {"norm_w": scale * g2}, o1["m"], o1["v"], 2, lr=0.1, beta1=0.9, beta2=0.999,
                     eps=0.0, weight_decay=0.0, max_grad_norm=0.0)
        outs.append(o2["params"]["norm_w"])
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-12)
    # first step without eps is lr * sign(g)
    o = O.adamw({"norm_w": w}, {"norm_w": g1}, {"norm_w": z}, {"norm_w": z}, 1, lr=0.1, beta1=0.9, beta2=0.999,
                eps=0.0, weight_decay=0.0, max_grad_norm=0.0)
    np.testing.assert_allclose(o["params"]["norm_w"], w - 0.1 * np.sign(g1), rtol=1e-14)


def test_clip_coefficient_closed_form():
    g = {"b_down": np.array([3.0]), "norm_w": np.array([4.0])}
    assert O.global_grad_norm(g) == 5.0
    assert O.clip_coefficient(5.0, 1.0) == pytest.approx(1.0 / (5.0 + 1e-6), rel=1e-15)
    assert O.clip_coefficient(5.0, 10.0) == 1.0
    assert O.clip_coefficient(5.0, 0.0) == 1.0
    assert O.clip_coefficient(5.0, -1.0) == 1.0
    # the clipped gradient has norm max_norm * norm / (norm + 1e-6)
    c = O.clip_coefficient(5.0, 2.0)
    assert math.hypot(3.0 * c, 4.0 * c) == pytest.approx(2.0 * 5.0 / (5.0 + 1e-6), rel=1e-15)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sharded_norm_equals_dense(act, t):
    p, rng = _params(5, 16, 32, act)
    x = rng.standard_normal((6, 16))
    tgt = rng.standard_normal((6, 16))
    d = O.dense_step(p, x, tgt, 1e-6, 0.1, act)
    dense = O.global_grad_norm({k: d["grads"][k] for k in p})
    s = O.sharded_step(p, x, tgt, 1e-6, 0.1, t, act)
    assert O.sharded_grad_norm(s["ranks"]) == pytest.approx(dense, rel=1e-13)
    over = O.sharded_grad_norm(s["ranks"], count_replicated_once=False)
    rep = sum(float(np.sum(d["grads"][k] ** 2)) for k in O.REPLICATED)
    assert over ** 2 == pytest.approx(dense ** 2 + (t - 1) * rep, rel=1e-12)
    if t > 1:
        assert over > dense


def test_dense_step_adamw_composes():
    p, rng = _params(9, 8, 12, "swiglu")
    x, tgt = rng.standard_normal((4, 8)), rng.standard_normal((4, 8))
    hp = dict(O.ADAMW_DEFAULTS, lr=0.01, max_grad_norm=1e-3)
    z = {k: np.zeros_like(p[k]) for k in p}
    out = O.dense_step_adamw(p, x, tgt, 1e-6, z, dict(z), 1, hp)
    d = O.dense_step(p, x, tgt, 1e-6, 0.0)
    g = {k: d["grads"][k] for k in p}
    ref = O.adamw(p, g, z, dict(z), 1, **hp)
    for k in p:
        np.testing.assert_array_equal(out["new_params"][k], ref["params"][k])
    assert out["clip"] < 1.0
