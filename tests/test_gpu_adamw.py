"""Parity of the clipped AdamW step ("Megatron-LM walkthrough", "Stage 8")
against the oracle, through the C ABI.

* The update in isolation: after one backward, the gradient buffers are
  overwritten with seeded synthetic gradients and seeded moments are bound,
  so the GPU's grad_sqnorm + adamw_update and the oracle's ``adamw`` see the
  same inputs.  Masters (or fp32 parameters), both moments and the norm are
  compared at the fp32 tolerance, for clipping off, inactive and active, at
  a bias-correction step > 1, for both activations and dtypes.  The bf16
  parameter copy must be the round-to-nearest-even of the new master.
* A whole step (forward, loss, backward, AdamW at step 1 with clipping
  active) against the oracle's ``dense_step_adamw``.  At step 1 every update
  is lr * u(c g) with u(z) = z / (|z| + eps), so the gradient tolerance
  carries into the update through u's slope: within the gradient bound the
  update moves by at most lr * dg * eps / (min|c g| + eps)^2, and never by
  more than 2 lr.  That allowance is computed from the oracle's gradient and
  the stated gradient tolerance only.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import TOL, compare, device_inputs, to_np

pytestmark = pytest.mark.gpu

LIB_KEY = {"w_1": "w_gate_up"}


def _cfg(dtype, act, N, H, F):
    base = synth.CONFIGS["fp32_small" if dtype == "f32" else "bf16_h2048"]
    c = dataclasses.replace(base.with_shape(N, H, F), act=act)
    if act == "gelu":
        c = dataclasses.replace(c, b_1_std=0.01)
    return c


def _run_backward(cfg, t, inp):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    m = TPMLP(max(cfg.tokens, 1), cfg.hidden, cfg.ffn, max_t=max(8, t), dtype=cfg.dtype, act=cfg.act)
    d = device_inputs(cfg, inp)
    names = synth.param_names(cfg.act)
    params = {LIB_KEY.get(k, k): d[k] for k in names}
    masters = None
    if cfg.dtype == "bf16":
        masters = {LIB_KEY.get(k, k): torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda() for k in names}
        m.bind_master(masters)
    y = m.forward(d["x"], params["norm_w"], params["w_gate_up"], params["w_down"], params["b_down"], cfg.eps, t,
                  b_1=params.get("b_1"))
    loss, dy = m.mse_loss_grad(y, d["target"])
    dx, g = m.backward(dy)
    return m, params, masters, g


@pytest.mark.parametrize("dtype,act,N,H,F", [("f32", "swiglu", 16, 64, 256), ("f32", "gelu", 24, 64, 200),
                                             ("bf16", "swiglu", 64, 512, 1536), ("bf16", "gelu", 40, 384, 1280),
                                             ("bf16", "swiglu", 8, 2048, 5632)])
@pytest.mark.parametrize("clip", ["off", "inactive", "active"])
def test_adamw_update_matches_oracle(dtype, act, N, H, F, clip):
    cfg = _cfg(dtype, act, N, H, F)
    inp = synth.make_inputs(cfg, seed=5)
    m, params, masters, g = _run_backward(cfg, 2, inp)
    names = synth.param_names(cfg.act)
    st = synth.make_optimizer_state(cfg, seed=77)
    for k in names:
        g[LIB_KEY.get(k, k)].copy_(torch.from_numpy(np.asarray(st["grad"][k], dtype=np.float32)))
    mom = {LIB_KEY.get(k, k): torch.from_numpy(np.asarray(st["m"][k], dtype=np.float32)).cuda() for k in names}
    vel = {LIB_KEY.get(k, k): torch.from_numpy(np.asarray(st["v"][k], dtype=np.float32)).cuda() for k in names}
    m.bind_adam_state(mom, vel)
    norm_o = O.global_grad_norm(st["grad"])
    max_norm = {"off": 0.0, "inactive": 1e9, "active": 0.3 * norm_o}[clip]
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, max_grad_norm=max_norm)
    step = 3
    gn = m.adamw_step(step=step, **hp)
    m.sync()
    p0 = {k: np.asarray(inp[k], dtype=np.float64) for k in names}
    ref = O.adamw(p0, st["grad"], st["m"], st["v"], step, **hp)
    assert (ref["clip"] < 1.0) == (clip == "active")
    assert abs(float(gn.item()) - norm_o) <= 1e-6 * norm_o
    for k in names:
        lk = LIB_KEY.get(k, k)
        new = to_np(masters[lk]) if masters is not None else to_np(params[lk])
        compare("m_" + k, to_np(mom[lk]), ref["m"][k], "f32")
        compare("v_" + k, to_np(vel[lk]), ref["v"][k], "f32")
        compare("w_" + k, new, ref["params"][k], "f32")
        if masters is not None:
            # the bf16 copy is the round-to-nearest-even of the new master
            np.testing.assert_array_equal(synth.bf16_bits(to_np(params[lk])),
                                          synth.bf16_bits(synth.round_to_bf16(new)))


def _step1_allowance(g_o, c_o, lr, eps, dtype):
    """Bound on |lr u(c g_gpu) - lr u(c g_o)| for every g_gpu inside the
    gradient tolerance of ``dtype`` (the clip factor's own error folded in)."""
    tol = TOL[dtype]
    ag = np.abs(g_o)
    dg = c_o * (tol["rtol"] * ag + tol["atol_max"] * float(np.max(ag)) + tol["norm"] * ag)
    lo = np.maximum(c_o * ag - dg, 0.0)
    return np.minimum(lr * dg * eps / (lo + eps) ** 2, 2.0 * lr)


@pytest.mark.parametrize("dtype,act,N,H,F,t", [("f32", "swiglu", 16, 64, 256, 2), ("f32", "gelu", 16, 64, 256, 4),
                                               ("bf16", "swiglu", 300, 512, 1536, 4),
                                               ("bf16", "gelu", 333, 384, 1280, 8)])
def test_adamw_full_step_matches_oracle(dtype, act, N, H, F, t):
    cfg = _cfg(dtype, act, N, H, F)
    inp = synth.make_inputs(cfg, seed=9)
    names = synth.param_names(cfg.act)
    p = {k: inp[k] for k in names}
    z = {k: np.zeros_like(p[k]) for k in names}
    d = O.dense_step(p, inp["x"], inp["target"], cfg.eps, 0.0, cfg.act)
    norm_o = O.global_grad_norm({k: d["grads"][k] for k in names})
    hp = dict(O.ADAMW_DEFAULTS, lr=1e-2, max_grad_norm=0.5 * norm_o)
    ref = O.dense_step_adamw(p, inp["x"], inp["target"], cfg.eps, z, dict(z), 1, hp, cfg.act)
    assert ref["clip"] < 1.0
    m, params, masters, g = _run_backward(cfg, t, inp)
    mom, vel = m.new_adam_state()
    gn = m.adamw_step(step=1, **hp)
    m.sync()
    tol = TOL[dtype]
    assert abs(float(gn.item()) - norm_o) <= tol["norm"] * norm_o
    for k in names:
        lk = LIB_KEY.get(k, k)
        new = to_np(masters[lk]) if masters is not None else to_np(params[lk])
        extra = _step1_allowance(ref["grads"][k], ref["clip"], hp["lr"], hp["eps"], dtype) + \
            0.5 * np.spacing(np.abs(new).astype(np.float32)).astype(np.float64)
        compare("w_" + k, new, ref["new_params"][k], dtype, extra=extra)
        # first moment after one step is (1 - b1) c g: the gradient tolerance, scaled
        compare("m_" + k, to_np(mom[lk]), ref["m"][k], dtype)


def test_adamw_errors():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_ARG, ERR_ORDER, TPMLP, TPMLPError
    m = TPMLP(16, 64, 256, max_t=8, dtype="f32", act="swiglu")
    with pytest.raises(TPMLPError) as e:
        m.adamw_step(lr=1e-3, step=1)
    assert e.value.status == ERR_ORDER
    cfg = synth.CONFIGS["fp32_small"]
    inp = synth.make_inputs(cfg)
    m, params, masters, g = _run_backward(cfg, 2, inp)
    with pytest.raises(TPMLPError) as e:
        m.adamw_step(lr=1e-3, step=1)  # moments not bound
    assert e.value.status == ERR_ARG
    m.new_adam_state()
    for bad in (dict(step=0), dict(step=1, beta1=1.0), dict(step=1, beta2=-0.1), dict(step=1, eps=-1.0),
                dict(step=1, lr=float("nan"))):
        kw = dict(lr=1e-3)
        kw.update(bad)
        with pytest.raises(TPMLPError) as e:
            m.adamw_step(**kw)
        assert e.value.status == ERR_ARG
    m.adamw_step(lr=1e-3, step=1)
    m.sync()
