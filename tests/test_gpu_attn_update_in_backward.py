"""The SGD update applied by the attention sublayer's backward
(``tpattn_set_update_in_backward``; "Megatron-LM walkthrough", "Stage 8: the
optimizer step"), through the C ABI.

* Every new fp32 master equals fmaf(-lr, g, w) of its old value w and the
  gradient g that the same backward wrote, bit for bit, and every bf16 copy
  is its round-to-nearest-even, on the fused and the unfused attention path,
  with W_qkv and W_o updated in their weight-gradient epilogues (8192 tokens
  and more; hidden 328 ends in an 8-column chunk) and by the update kernel
  (fewer tokens).
* On the unfused path, which has no atomics, the whole step is also
  bit-identical to backward followed by ``tpattn_sgd_step``: y, dx, every
  gradient, the masters and the copies.  The fused backward accumulates dQ
  with atomic adds in arrival order, so there only y is compared run to run.
* The whole step against the oracle at 8192 tokens.
* Order and argument errors: a backward without bound masters, a non-finite
  lr, and sgd_step / adamw_step after a backward that already applied the
  update.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, fma_f32, to_np

pytestmark = pytest.mark.gpu

LR = 0.1
NAMES = ("norm_w", "w_qkv", "w_o", "b_o")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def _cfg(B, S, H, nq, nkv, d):
    return dataclasses.replace(synth.ATTN_CONFIGS["attn_small"], name="case", batch=B, seq=S, hidden=H, n_q=nq,
                               n_kv=nkv, d=d, w_std=0.05)


def _step(cfg, inp, t, in_backward):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPAttn
    from tensor_transformer_mlp_rmsnorm_gb300.tpmlp import tpmlp_mse_loss_grad_noalloc
    m = TPAttn(cfg.tokens, cfg.hidden, cfg.n_q, cfg.n_kv, cfg.d, cfg.seq, max_t=max(t, 1))
    p = {k: _dev(inp[k]) for k in NAMES}
    masters = {k: torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda() for k in NAMES}
    m.bind_master(masters)
    if in_backward:
        m.set_update_in_backward(True, LR)
    y = m.forward(_dev(inp["x"]), p["norm_w"], p["w_qkv"], p["w_o"], p["b_o"], cfg.eps, t, cfg.batch, cfg.seq)
    dy = torch.empty_like(y)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    tpmlp_mse_loss_grad_noalloc(y, _dev(inp["target"]), dy, loss)
    dx, g = m.backward(dy)
    if not in_backward:
        m.sgd_step(LR)
    m.sync()
    return m, {"y": to_np(y), "loss": float(loss.item()), "dx": to_np(dx), "deterministic": not m.fused_active(),
               "grads": {k: to_np(v) for k, v in g.items()}, "master": {k: to_np(v) for k, v in masters.items()},
               "params": {k: synth.bf16_bits(to_np(v)) for k, v in p.items()}}


CASES = [  # batch, seq, hidden, n_q, n_kv, d, t
    (4, 2048, 512, 4, 2, 128, 2),  # fused attention, 8192 tokens
    (9, 960, 328, 4, 2, 64, 2),  # unfused, 8640 tokens, hidden ending in an 8-column chunk
    (2, 256, 512, 4, 1, 128, 1),  # fewer tokens: the update kernel
    (1, 64, 128, 2, 2, 64, 2),
]


def _check_update(run, inp):
    """New masters are fmaf(-lr, g, w) of the gradients written; copies their bf16 rounding."""
    for k in NAMES:  # the float64 copies hold the float32 values exactly
        want = fma_f32(np.float32(-LR), run["grads"][k].astype(np.float32), np.asarray(inp[k], dtype=np.float32))
        got = run["master"][k].astype(np.float32)
        np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32), err_msg=k)
        np.testing.assert_array_equal(run["params"][k], synth.bf16_bits(synth.round_to_bf16(want)), err_msg=k)


@pytest.mark.parametrize("B,S,H,nq,nkv,d,t", CASES)
def test_update_in_backward(B, S, H, nq, nkv, d, t):
    cfg = _cfg(B, S, H, nq, nkv, d)
    inp = synth.make_attn_inputs(cfg, seed=61)
    _, sep = _step(cfg, inp, t, False)
    m, fused = _step(cfg, inp, t, True)
    assert m.update_in_epilogue() == (B * S >= 8192)
    assert m.fused_active() == (d == 128 and S % 128 == 0)
    _check_update(fused, inp)
    _check_update(sep, inp)
    np.testing.assert_array_equal(fused["y"], sep["y"])
    if fused["deterministic"]:
        np.testing.assert_array_equal(fused["dx"], sep["dx"])
        assert fused["loss"] == sep["loss"]
        for group in ("grads", "master", "params"):
            for k in NAMES:
                np.testing.assert_array_equal(fused[group][k], sep[group][k], err_msg=(group, k))


def test_step_matches_oracle():
    B, S, H, nq, nkv, d, t = 64, 128, 256, 2, 2, 128, 2
    cfg = _cfg(B, S, H, nq, nkv, d)
    inp = synth.make_attn_inputs(cfg, seed=62)
    m, gpu = _step(cfg, inp, t, True)
    assert m.update_in_epilogue()
    ora = O.attn_sharded_step({k: inp[k] for k in NAMES}, inp["x"], inp["target"], cfg.eps, LR, t, B, nq, nkv)
    compare("y", gpu["y"], ora["y"], "bf16")
    compare("dx", gpu["dx"], ora["grads"]["x"], "bf16")
    for k in NAMES:
        compare("d" + k, gpu["grads"][k], ora["grads"][k], "bf16")
        new = gpu["master"][k]
        w0 = np.asarray(inp[k], dtype=np.float32).astype(np.float64)
        compare("post_step_" + k, new, w0 - LR * ora["grads"][k], "bf16",
                extra=0.5 * np.spacing(np.abs(new).astype(np.float32)).astype(np.float64))
        np.testing.assert_array_equal(gpu["params"][k], synth.bf16_bits(synth.round_to_bf16(new)))


def test_errors():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_ARG, ERR_ORDER, TPAttn, TPMLPError
    m = TPAttn(256, 128, 2, 2, 64, 128, max_t=2)
    with pytest.raises(TPMLPError) as e:
        m.set_update_in_backward(True, float("inf"))
    assert e.value.status == ERR_ARG
    m.set_update_in_backward(True, LR)
    x = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    wqkv = torch.zeros(6 * 64, 128, dtype=torch.bfloat16, device="cuda")
    wo = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")

    def fwd_bwd():
        m.forward(x, w, wqkv, wo, w, 1e-6, 2, 2, 128)
        return m.backward(torch.zeros_like(x))

    with pytest.raises(TPMLPError) as e:  # no masters bound
        fwd_bwd()
    assert e.value.status == ERR_ORDER
    m.bind_master({"norm_w": w.float(), "w_qkv": wqkv.float(), "w_o": wo.float(), "b_o": w.float()})
    fwd_bwd()
    for call in (lambda: m.sgd_step(LR), lambda: (m.new_adam_state(), m.adamw_step(lr=1e-3, step=1))):
        with pytest.raises(TPMLPError) as e:
            call()
        assert e.value.status == ERR_ORDER
    # the next step runs normally, with or without the update in backward
    fwd_bwd()
    m.set_update_in_backward(False)
    fwd_bwd()
    m.sgd_step(LR)
    m.sync()
