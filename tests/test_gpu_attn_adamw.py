"""Clipped AdamW on the attention sublayer's parameters, on the GPU against
the oracle, through the C ABI (tpattn_bind_adam_state, tpattn_adamw_step).

The update itself is checked on seeded gradients and moments written into
the context's gradient tensors after a backward (every element against the
oracle's AdamW at the fp32 tolerance, with and without an active clip); a
second test runs forward, loss, backward and AdamW on the fused path and
checks the update against the oracle's AdamW applied to the gradients the
backward produced, and the gradient norm against the oracle's own backward.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, to_np

pytestmark = pytest.mark.gpu

NAMES = ("norm_w", "w_qkv", "w_o", "b_o")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _setup(B, S, H, nq, nkv, d, t, seed):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPAttn
    from tensor_transformer_mlp_rmsnorm_gb300.tpmlp import tpmlp_mse_loss_grad_noalloc
    cfg = dataclasses.replace(synth.ATTN_CONFIGS["attn_small"], name="case", batch=B, seq=S, hidden=H, n_q=nq,
                              n_kv=nkv, d=d, w_std=0.05)
    inp = synth.make_attn_inputs(cfg, seed=seed)
    m = TPAttn(cfg.tokens, H, nq, nkv, d, S, max_t=t)
    p = {k: _dev(inp[k]) for k in NAMES}
    masters = {k: _f32(inp[k]) for k in NAMES}
    m.bind_master(masters)
    y = m.forward(_dev(inp["x"]), p["norm_w"], p["w_qkv"], p["w_o"], p["b_o"], cfg.eps, t, B, S)
    dy = torch.empty_like(y)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    tpmlp_mse_loss_grad_noalloc(y, _dev(inp["target"]), dy, loss)
    _, g = m.backward(dy)
    return cfg, inp, m, p, masters, g


def _check_bf16_copies(p, masters):
    for k in NAMES:
        np.testing.assert_array_equal(synth.bf16_bits(to_np(p[k])),
                                      synth.bf16_bits(synth.round_to_bf16(to_np(masters[k]))))


@pytest.mark.parametrize("clip", ["off", "inactive", "active"])
@pytest.mark.parametrize("B,S,H,nq,nkv,d,t", [(2, 128, 256, 4, 2, 64, 2), (1, 256, 512, 8, 2, 128, 2)])
def test_attention_adamw_update_matches_oracle(B, S, H, nq, nkv, d, t, clip):
    cfg, inp, m, p, masters, g = _setup(B, S, H, nq, nkv, d, t, seed=7)
    st = synth.make_attn_optimizer_state(cfg, seed=91)
    for k in NAMES:
        g[k].copy_(_f32(st["grad"][k]))
    mom = {k: _f32(st["m"][k]) for k in NAMES}
    vel = {k: _f32(st["v"][k]) for k in NAMES}
    m.bind_adam_state(mom, vel)
    norm_o = O.global_grad_norm(st["grad"])
    max_norm = {"off": 0.0, "inactive": 1e9, "active": 0.3 * norm_o}[clip]
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, max_grad_norm=max_norm)
    gn = m.adamw_step(step=4, **hp)
    m.sync()
    p0 = {k: np.asarray(inp[k], dtype=np.float64) for k in NAMES}
    ref = O.adamw(p0, st["grad"], st["m"], st["v"], 4, **hp)
    assert (ref["clip"] < 1.0) == (clip == "active")
    assert abs(float(gn.item()) - norm_o) <= 1e-6 * norm_o
    for k in NAMES:
        compare("m_" + k, to_np(mom[k]), ref["m"][k], "f32")
        compare("v_" + k, to_np(vel[k]), ref["v"][k], "f32")
        compare("w_" + k, to_np(masters[k]), ref["params"][k], "f32")
    _check_bf16_copies(p, masters)


def test_attention_adamw_after_backward():
    B, S, H, nq, nkv, d, t = 2, 256, 512, 4, 2, 128, 2
    cfg, inp, m, p, masters, g = _setup(B, S, H, nq, nkv, d, t, seed=8)
    assert m.fused_active()
    g_gpu = {k: to_np(g[k]).astype(np.float64) for k in NAMES}
    m.new_adam_state()
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_grad_norm=0.5)
    gn = m.adamw_step(step=1, **hp)
    m.sync()
    # the update is AdamW of the gradients the backward wrote
    p0 = {k: np.asarray(inp[k], dtype=np.float64) for k in NAMES}
    z = {k: np.zeros_like(v) for k, v in p0.items()}
    ref = O.adamw(p0, g_gpu, z, dict(z), 1, **hp)
    assert abs(float(gn.item()) - ref["grad_norm"]) <= 1e-5 * ref["grad_norm"]
    for k in NAMES:
        compare("w_" + k, to_np(masters[k]), ref["params"][k], "f32")
    _check_bf16_copies(p, masters)
    # and its norm is the norm of the oracle's own gradients, within the bf16 gradient tolerance
    pa = {k: inp[k] for k in NAMES}
    ora = O.attn_sharded_step(pa, inp["x"], inp["target"], cfg.eps, 0.0, t, B, nq, nkv)
    norm_o = O.global_grad_norm({k: ora["grads"][k] for k in NAMES})
    assert abs(float(gn.item()) - norm_o) <= 2e-2 * norm_o


def test_attention_adamw_errors():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_ARG, ERR_ORDER, TPAttn, TPMLPError
    m = TPAttn(256, 128, 2, 2, 64, 128, max_t=2)
    m.new_adam_state()
    with pytest.raises(TPMLPError) as e:  # no backward yet
        m.adamw_step(lr=1e-3, step=1)
    assert e.value.status == ERR_ORDER
    x = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    wqkv = torch.zeros(6 * 64, 128, dtype=torch.bfloat16, device="cuda")
    wo = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    m.forward(x, w, wqkv, wo, w, 1e-6, 2, 2, 128)
    m.backward(torch.zeros_like(x))
    for bad in (dict(step=0), dict(step=1, beta1=1.0), dict(step=1, eps=-1.0), dict(step=1, lr=float("nan"))):
        with pytest.raises(TPMLPError) as e:
            m.adamw_step(**dict(dict(lr=1e-3), **bad))
        assert e.value.status == ERR_ARG
    m.bind_adam_state(None, None)
    with pytest.raises(TPMLPError) as e:
        m.adamw_step(lr=1e-3, step=1)
    assert e.value.status == ERR_ARG
    m.sync()
