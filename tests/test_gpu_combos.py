"""The MLP step's options combined, through the C ABI, on bf16 shapes that
span several tiles and a ragged tail ("Megatron tensor-parallel MLP";
walkthrough, "Deep dive: sequence parallelism, memory for free" and "Stage 8:
the optimizer step").

* E4M3 GEMM operands with the sequence-parallel form.  The casts take one
  scale per tensor over all tokens either way, so y, dy, dx and the
  projection gradients are bit-identical to the E4M3 step without sequence
  parallelism; the whole step matches the oracle's E4M3 step at the FP8
  tolerance.
* E4M3 operands, or the sequence-parallel form, followed by the clipped AdamW
  update (clipping active).  The update must equal the oracle's AdamW applied
  to the gradients that backward wrote (fp32 tolerance, norm to 1e-6), and the
  bf16 copies must be the round-to-nearest-even of the new masters: the
  optimizer reads exactly what the preceding backward produced.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, compare_step, device_inputs, gpu_step, to_np

pytestmark = pytest.mark.gpu

LR = 0.1
LIB_KEY = {"w_1": "w_gate_up"}
CASES = [("swiglu", 300, 512, 1536, 4), ("gelu", 336, 384, 1280, 8)]


def _cfg(act, N, H, F):
    c = dataclasses.replace(synth.CONFIGS["bf16_h2048"].with_shape(N, H, F), act=act)
    return dataclasses.replace(c, b_1_std=0.01) if act == "gelu" else c


def _module(cfg, t, fp8=False, sp=False):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    m = TPMLP(cfg.tokens, cfg.hidden, cfg.ffn, max_t=max(8, t), dtype="bf16", act=cfg.act)
    if fp8:
        m.set_precision("fp8")
    m.set_sequence_parallel(sp)
    return m


@pytest.mark.parametrize("act,N,H,F,t", CASES)
def test_fp8_with_sequence_parallel(act, N, H, F, t):
    cfg = _cfg(act, N, H, F)
    inp = synth.make_inputs(cfg, seed=31)
    both = gpu_step(cfg, inp, t, LR, mod=_module(cfg, t, fp8=True, sp=True))
    fp8 = gpu_step(cfg, inp, t, LR, mod=_module(cfg, t, fp8=True, sp=False))
    for k in ("y", "dy", "dx"):
        np.testing.assert_array_equal(both[k], fp8[k], err_msg=k)
    for k in synth.param_names(cfg.act):
        if k not in ("norm_w", "b_down"):
            np.testing.assert_array_equal(both["grads"][k], fp8["grads"][k], err_msg=k)
    p = {k: inp[k] for k in synth.param_names(cfg.act)}
    ora = O.dense_step_fp8(p, inp["x"], inp["target"], cfg.eps, LR, cfg.act, store=synth.round_to_bf16)
    compare_step(cfg, both, ora, inp, LR, tol="fp8")


def _backward_then_adamw(cfg, t, inp, fp8, sp):
    m = _module(cfg, t, fp8=fp8, sp=sp)
    d = device_inputs(cfg, inp)
    names = synth.param_names(cfg.act)
    params = {LIB_KEY.get(k, k): d[k] for k in names}
    masters = {LIB_KEY.get(k, k): torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda() for k in names}
    m.bind_master(masters)
    y = m.forward(d["x"], params["norm_w"], params["w_gate_up"], params["w_down"], params["b_down"], cfg.eps, t,
                  b_1=params.get("b_1"))
    _, dy = m.mse_loss_grad(y, d["target"])
    _, g = m.backward(dy)
    m.sync()
    grads = {k: to_np(g[LIB_KEY.get(k, k)]).astype(np.float64) for k in names}
    norm = O.global_grad_norm(grads)
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, max_grad_norm=0.5 * norm)
    m.new_adam_state()
    gn = m.adamw_step(step=1, **hp)
    m.sync()
    p0 = {k: np.asarray(inp[k], dtype=np.float64) for k in names}
    z = {k: np.zeros_like(p0[k]) for k in names}
    ref = O.adamw(p0, grads, z, dict(z), 1, **hp)
    assert ref["clip"] < 1.0
    assert abs(float(gn.item()) - norm) <= 1e-6 * norm
    for k in names:
        lk = LIB_KEY.get(k, k)
        new = to_np(masters[lk])
        compare("w_" + k, new, ref["params"][k], "f32")
        np.testing.assert_array_equal(synth.bf16_bits(to_np(params[lk])), synth.bf16_bits(synth.round_to_bf16(new)))


@pytest.mark.parametrize("act,N,H,F,t", CASES)
def test_fp8_then_adamw(act, N, H, F, t):
    cfg = _cfg(act, N, H, F)
    _backward_then_adamw(cfg, t, synth.make_inputs(cfg, seed=32), fp8=True, sp=False)


@pytest.mark.parametrize("act,N,H,F,t", CASES)
def test_sequence_parallel_then_adamw(act, N, H, F, t):
    cfg = _cfg(act, N, H, F)
    _backward_then_adamw(cfg, t, synth.make_inputs(cfg, seed=33), fp8=False, sp=True)
