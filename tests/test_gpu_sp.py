"""Sequence-parallel form on the GPU against the oracle's ``sp_step``
(walkthrough, "Deep dive: sequence parallelism, memory for free"; "Stage 7:
finalize_model_grads"), through the C ABI.

* The whole step with sequence parallelism equals the oracle's decomposition
  within the stated tolerances (fp32 and bf16, both activations, several t).
* Only the norm-weight and output-bias gradients depend on the mode: y, the
  loss, dx and the projection gradients are bit-identical to the plain form.
* Without the gradient all-reduce (SKIP_SP_GRAD_SYNC), dnorm_w and db_down
  are the viewing shard's own sums (oracle with ``skip_sp_grad_sync``),
  everything else unchanged bit for bit.
* Shape and mode errors.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, compare_step, gpu_step

pytestmark = pytest.mark.gpu

LR = 0.1


def _cfg(dtype, act, N, H, F):
    base = synth.CONFIGS["fp32_small" if dtype == "f32" else "bf16_h2048"]
    c = dataclasses.replace(base.with_shape(N, H, F), act=act)
    if act == "gelu":
        c = dataclasses.replace(c, b_1_std=0.01)
    return c


def _module(cfg, t, sp):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    m = TPMLP(max(cfg.tokens, 1), cfg.hidden, cfg.ffn, max_t=max(8, t), dtype=cfg.dtype, act=cfg.act)
    m.set_sequence_parallel(sp)
    return m


CASES = [("f32", "swiglu", 16, 64, 256, 2), ("f32", "swiglu", 16, 64, 256, 8), ("f32", "gelu", 24, 64, 200, 4),
         ("bf16", "swiglu", 300, 512, 1536, 4), ("bf16", "gelu", 336, 384, 1280, 8),
         ("bf16", "swiglu", 1024, 256, 2048, 4)]


@pytest.mark.parametrize("dtype,act,N,H,F,t", CASES)
def test_sp_step_matches_oracle(dtype, act, N, H, F, t):
    cfg = _cfg(dtype, act, N, H, F)
    inp = synth.make_inputs(cfg, seed=21)
    gpu = gpu_step(cfg, inp, t, LR, mod=_module(cfg, t, True))
    ora = O.sp_step({k: inp[k] for k in synth.param_names(cfg.act)}, inp["x"], inp["target"], cfg.eps, LR, t,
                    cfg.act)
    compare_step(cfg, gpu, ora, inp, LR)
    plain = gpu_step(cfg, inp, t, LR, mod=_module(cfg, t, False))
    for k in ("y", "dy", "dx"):
        np.testing.assert_array_equal(gpu[k], plain[k], err_msg=k)
    for k in synth.param_names(cfg.act):
        if k not in ("norm_w", "b_down"):
            np.testing.assert_array_equal(gpu["grads"][k], plain["grads"][k], err_msg=k)


@pytest.mark.parametrize("dtype,act,N,H,F,t", [CASES[1], CASES[3], CASES[4]])
def test_sp_without_grad_sync(dtype, act, N, H, F, t):
    from tensor_transformer_mlp_rmsnorm_gb300 import DBG_SKIP_SP_GRAD_SYNC
    cfg = _cfg(dtype, act, N, H, F)
    inp = synth.make_inputs(cfg, seed=22)
    p = {k: inp[k] for k in synth.param_names(cfg.act)}
    synced = gpu_step(cfg, inp, t, LR, mod=_module(cfg, t, True))
    for shard in (0, t - 1):
        gpu = gpu_step(cfg, inp, t, LR, flags=DBG_SKIP_SP_GRAD_SYNC, shard=shard, mod=_module(cfg, t, True))
        ora = O.sp_step(p, inp["x"], inp["target"], cfg.eps, LR, t, cfg.act, skip_sp_grad_sync=True,
                        view_rank=shard)
        compare("dnorm_w", gpu["grads"]["norm_w"], ora["grads"]["norm_w"], cfg.dtype)
        compare("db_down", gpu["grads"]["b_down"], ora["grads"]["b_down"], cfg.dtype)
        for k in ("y", "dx"):
            np.testing.assert_array_equal(gpu[k], synced[k], err_msg=k)
        for k in synth.param_names(cfg.act):
            if k not in ("norm_w", "b_down"):
                np.testing.assert_array_equal(gpu["grads"][k], synced["grads"][k], err_msg=k)
        assert not np.array_equal(gpu["grads"]["norm_w"], synced["grads"]["norm_w"])


def test_sp_errors():
    import torch
    from tensor_transformer_mlp_rmsnorm_gb300 import (DBG_SKIP_FWD_REDUCE, DBG_SKIP_SP_GRAD_SYNC, ERR_ARG, ERR_SHAPE,
                                                      ERR_UNSUPPORTED, TPMLPError)
    cfg = _cfg("f32", "swiglu", 16, 64, 256)
    inp = synth.make_inputs(cfg)
    m = _module(cfg, 8, True)
    with pytest.raises(TPMLPError) as e:
        gpu_step(cfg.with_tokens(12), synth.make_inputs(cfg.with_tokens(12)), 8, LR, mod=m)
    assert e.value.status == ERR_SHAPE
    with pytest.raises(TPMLPError) as e:
        gpu_step(cfg, inp, 2, LR, flags=DBG_SKIP_FWD_REDUCE, mod=m)
    assert e.value.status == ERR_UNSUPPORTED
    m2 = _module(cfg, 2, False)
    with pytest.raises(TPMLPError) as e:
        gpu_step(cfg, inp, 2, LR, flags=DBG_SKIP_SP_GRAD_SYNC, mod=m2)
    assert e.value.status == ERR_ARG
    torch.cuda.synchronize()
