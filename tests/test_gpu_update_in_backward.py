"""The SGD update applied by backward (``tpmlp_set_update_in_backward``;
"Megatron-LM walkthrough", "Stage 8: the optimizer step"), through the C ABI.

* Bit-identical to backward followed by ``tpmlp_sgd_step``: y, dy, dx, every
  gradient, the fp32 masters and the bf16 parameter copies, for both
  activations, several t, E4M3 operands and the sequence-parallel form, with
  the matrices updated in their weight-gradient epilogues (8192 tokens and
  more, ragged chunks and a K-split tile among them: the update is then
  applied by the tile's first part after it adds the later parts) and by the
  update kernel (fewer tokens, and the H = 2048 workload).
* The whole step against the oracle, as for the separate update.
* Order and argument errors: the fp32 dtype, a backward without bound masters,
  and sgd_step / adamw_step after a backward that already applied the update.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare_step, device_inputs, gpu_step

pytestmark = pytest.mark.gpu

LR = 0.1


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


def _same(a, b):
    for k in ("y", "dy", "dx"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    assert a["loss"] == b["loss"]
    for group in ("grads", "new_master", "new_params"):
        for k in a[group]:
            np.testing.assert_array_equal(a[group][k], b[group][k], err_msg=(group, k))


# 8192 tokens and more: the matrices are updated in their weight-gradient epilogues (H = 328 and
# F = 1000 end in 8-column chunks; 8200 tokens leave a ragged k-block; the gate/up gradient's 16
# tiles split along K).  Fewer: by the update kernel at the end of backward.
@pytest.mark.parametrize("act,N,H,F,t,fp8,sp", [("swiglu", 8192, 256, 512, 4, False, False),
                                                ("swiglu", 8200, 328, 1000, 4, False, False),
                                                ("gelu", 8192, 384, 640, 8, False, False),
                                                ("swiglu", 8192, 256, 512, 4, True, False),
                                                ("gelu", 8192, 384, 640, 8, False, True),
                                                ("swiglu", 300, 512, 1536, 4, False, False),
                                                ("gelu", 336, 384, 1280, 8, False, True)])
def test_bit_identical_to_separate_update(act, N, H, F, t, fp8, sp):
    cfg = _cfg(act, N, H, F)
    inp = synth.make_inputs(cfg, seed=51)
    sep = gpu_step(cfg, inp, t, LR, mod=_module(cfg, t, fp8, sp))
    m = _module(cfg, t, fp8, sp)
    fused = gpu_step(cfg, inp, t, LR, mod=m, update_in_backward=True)
    assert m.update_in_epilogue() == (N >= 8192)
    _same(fused, sep)


def test_h2048_workload_with_split_weight_gradient():
    cfg = synth.CONFIGS["bf16_h2048"]
    inp = synth.make_inputs(cfg, seed=52)
    sep = gpu_step(cfg, inp, 4, LR, mod=_module(cfg, 4))
    fused = gpu_step(cfg, inp, 4, LR, mod=_module(cfg, 4), update_in_backward=True)
    _same(fused, sep)


@pytest.mark.parametrize("N,H,F", [(300, 512, 1536), (8192, 256, 512)])
def test_step_matches_oracle(N, H, F):
    cfg = _cfg("swiglu", N, H, F)
    inp = synth.make_inputs(cfg, seed=53)
    gpu = gpu_step(cfg, inp, 4, LR, mod=_module(cfg, 4), update_in_backward=True)
    ora = O.sharded_step({k: inp[k] for k in synth.param_names(cfg.act)}, inp["x"], inp["target"], cfg.eps, LR, 4,
                         cfg.act)
    compare_step(cfg, gpu, ora, inp, LR)


def test_errors():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_ORDER, ERR_UNSUPPORTED, TPMLP, TPMLPError
    with pytest.raises(TPMLPError) as e:
        TPMLP(16, 64, 256, max_t=8, dtype="f32", act="swiglu").set_update_in_backward(True, 0.1)
    assert e.value.status == ERR_UNSUPPORTED
    cfg = _cfg("swiglu", 64, 256, 512)
    inp = synth.make_inputs(cfg, seed=54)
    d = device_inputs(cfg, inp)
    m = TPMLP(cfg.tokens, cfg.hidden, cfg.ffn, max_t=8, dtype="bf16", act="swiglu")
    m.set_update_in_backward(True, LR)

    def fwd_bwd():
        y = m.forward(d["x"], d["norm_w"], d["w_gate_up"], d["w_down"], d["b_down"], cfg.eps, 2)
        _, dy = m.mse_loss_grad(y, d["target"])
        return m.backward(dy)

    with pytest.raises(TPMLPError) as e:  # no masters bound
        fwd_bwd()
    assert e.value.status == ERR_ORDER
    masters = {k: torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda() for k in synth.param_names("swiglu")}
    m.bind_master(masters)
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
