"""The Python binding keeps alive what the library still points to, through
the C ABI.

The library remembers the pointers of the last forward's x and parameters
(backward reads x; the updates write the parameters), of the bound fp32
masters, and of the last backward's gradients (the updates read them).  A
caller that passes temporaries, drops the returned gradients, and then
allocates and fills new tensors of the same sizes must still get the step it
would get holding every tensor itself: bit-identical for the MLP, and for the
attention sublayer on its unfused path (the fused backward's atomic dQ sum is
not reproducible bit for bit).
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from tests._util import to_np

pytestmark = pytest.mark.gpu

LR = 0.1


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _churn(like):
    """Allocate and fill tensors of the given sizes, as a caller's next work would."""
    return [torch.full(t.shape, float("nan"), dtype=t.dtype, device=t.device) for t in like for _ in range(2)]


def _mlp_run(cfg, inp, t, temporaries):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    names = synth.param_names(cfg.act)
    key = {"w_1": "w_gate_up"}
    m = TPMLP(cfg.tokens, cfg.hidden, cfg.ffn, max_t=t, dtype="bf16", act=cfg.act)
    params = {key.get(k, k): _bf16(inp[k]) for k in names}
    if temporaries:
        m.bind_master({key.get(k, k): _f32(inp[k]) for k in names})
        y = m.forward(_bf16(inp["x"]), params["norm_w"], params["w_gate_up"], params["w_down"], params["b_down"],
                      cfg.eps, t, b_1=params.get("b_1"))
        junk = _churn([y, y, params["w_gate_up"].float()])
        _, dy = m.mse_loss_grad(y, _bf16(inp["target"]))
        dx, g = m.backward(dy)
        grads = {k: to_np(v) for k, v in g.items()}
        del g
        junk += _churn([v.float() for v in params.values()])
        m.sgd_step(LR)
        masters = {k: to_np(v) for k, v in m._masters.items()}
    else:
        ms = {key.get(k, k): _f32(inp[k]) for k in names}
        m.bind_master(ms)
        x, tg = _bf16(inp["x"]), _bf16(inp["target"])
        y = m.forward(x, params["norm_w"], params["w_gate_up"], params["w_down"], params["b_down"], cfg.eps, t,
                      b_1=params.get("b_1"))
        _, dy = m.mse_loss_grad(y, tg)
        dx, g = m.backward(dy)
        grads = {k: to_np(v) for k, v in g.items()}
        m.sgd_step(LR)
        masters = {k: to_np(v) for k, v in ms.items()}
    m.sync()
    return {"y": to_np(y), "dx": to_np(dx), "grads": grads, "masters": masters,
            "params": {k: to_np(v) for k, v in params.items()}}


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_mlp_with_temporaries(act):
    cfg = dataclasses.replace(synth.CONFIGS["bf16_h2048"].with_shape(300, 512, 1536), act=act)
    inp = synth.make_inputs(cfg, seed=71)
    held = _mlp_run(cfg, inp, 4, False)
    tmp = _mlp_run(cfg, inp, 4, True)
    for k in ("y", "dx"):
        np.testing.assert_array_equal(tmp[k], held[k], err_msg=k)
    for group in ("grads", "masters", "params"):
        for k in held[group]:
            np.testing.assert_array_equal(tmp[group][k], held[group][k], err_msg=(group, k))


def test_attention_with_temporaries():
    from tensor_transformer_mlp_rmsnorm_gb300 import TPAttn
    from tensor_transformer_mlp_rmsnorm_gb300.tpmlp import tpmlp_mse_loss_grad_noalloc
    names = ("norm_w", "w_qkv", "w_o", "b_o")
    B, S, H, nq, nkv, d, t = 3, 128, 256, 4, 2, 64, 2
    cfg = dataclasses.replace(synth.ATTN_CONFIGS["attn_small"], name="case", batch=B, seq=S, hidden=H, n_q=nq,
                              n_kv=nkv, d=d, w_std=0.05)
    inp = synth.make_attn_inputs(cfg, seed=72)

    def run(temporaries):
        m = TPAttn(cfg.tokens, H, nq, nkv, d, S, max_t=t)
        p = {k: _bf16(inp[k]) for k in names}
        held = None if temporaries else {k: _f32(inp[k]) for k in names}
        m.bind_master({k: _f32(inp[k]) for k in names} if temporaries else held)
        x = None if temporaries else _bf16(inp["x"])
        y = m.forward(_bf16(inp["x"]) if temporaries else x, p["norm_w"], p["w_qkv"], p["w_o"], p["b_o"], cfg.eps,
                      t, B, S)
        junk = _churn([y, y]) if temporaries else []
        dy = torch.empty_like(y)
        loss = torch.zeros(1, dtype=torch.float32, device="cuda")
        tpmlp_mse_loss_grad_noalloc(y, _bf16(inp["target"]), dy, loss)
        dx, g = m.backward(dy)
        grads = {k: to_np(v) for k, v in g.items()}
        if temporaries:
            del g
            junk += _churn([v.float() for v in p.values()])
        m.sgd_step(LR)
        m.sync()
        assert not m.fused_active()
        ms = m._masters
        return {"y": to_np(y), "dx": to_np(dx), "grads": grads, "masters": {k: to_np(v) for k, v in ms.items()},
                "params": {k: to_np(v) for k, v in p.items()}}

    held, tmp = run(False), run(True)
    for k in ("y", "dx"):
        np.testing.assert_array_equal(tmp[k], held[k], err_msg=k)
    for group in ("grads", "masters", "params"):
        for k in names:
            np.testing.assert_array_equal(tmp[group][k], held[group][k], err_msg=(group, k))
