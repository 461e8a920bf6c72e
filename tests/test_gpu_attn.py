"""The tensor-parallel attention sublayer on the GPU against the oracle,
through the C ABI (tpattn_*; the loss through tpmlp_mse_loss_grad_noalloc).

Cases cover grouped-query (n_q = 4 x n_kv), multi-head (n_q = n_kv) and
multi-query (n_kv = 1) attention, head dimensions 64 and 128, several
sequences per batch, and each logical degree t against the oracle's t-rank
decomposition.  Tolerances are the bf16 ones of tests/_util.py; the SGD
update is checked on the fp32 masters as in the MLP tests.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, to_np

pytestmark = pytest.mark.gpu

LR = 0.1
NAMES = ("norm_w", "w_qkv", "w_o", "b_o")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def _run(cfg, t, inp, fused=True, fused_only=False):
    from tensor_transformer_mlp_rmsnorm_gb300 import TPAttn, tpmlp_create  # noqa: F401
    from tensor_transformer_mlp_rmsnorm_gb300.tpmlp import tpmlp_mse_loss_grad_noalloc
    m = TPAttn(cfg.tokens, cfg.hidden, cfg.n_q, cfg.n_kv, cfg.d, cfg.seq, max_t=max(t, 1), fused_only=fused_only)
    if not fused_only:
        m.set_fused(fused)
    p = {k: _dev(inp[k]) for k in NAMES}
    masters = {k: torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda() for k in NAMES}
    m.bind_master(masters)
    x, tgt = _dev(inp["x"]), _dev(inp["target"])
    y = m.forward(x, p["norm_w"], p["w_qkv"], p["w_o"], p["b_o"], cfg.eps, t, cfg.batch, cfg.seq)
    dy = torch.empty_like(y)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    tpmlp_mse_loss_grad_noalloc(y, tgt, dy, loss)
    dx, g = m.backward(dy)
    m.sgd_step(LR)
    m.sync()
    assert m.fused_active() == (fused and cfg.d == 128 and cfg.seq % 128 == 0)
    return {"y": to_np(y), "loss": float(loss.item()), "dx": to_np(dx), "grads": {k: to_np(v) for k, v in g.items()},
            "master": {k: to_np(v) for k, v in masters.items()}}


CASES = [  # batch, seq, hidden, n_q, n_kv, d, t
    (2, 128, 256, 4, 2, 64, 2),
    (1, 256, 512, 8, 8, 64, 4),
    (3, 192, 384, 6, 1, 128, 1),
    (2, 512, 1024, 8, 2, 128, 2),
    (1, 64, 128, 2, 2, 64, 2),
    # shapes the fused kernels take (head_dim 128, seq % 128 == 0): one key
    # block, an odd number of key blocks, multi-query, multi-head
    (3, 128, 256, 2, 2, 128, 2),
    (1, 384, 1024, 8, 4, 128, 4),
    (2, 256, 512, 4, 1, 128, 1),
    # an odd number of query heads: a token row of dZ holds 3 x 16 chunks of 8
    (1, 256, 384, 3, 1, 128, 1),
]
FUSABLE = [c for c in CASES if c[5] == 128 and c[1] % 128 == 0]


def _case(B, S, H, nq, nkv, d, t, fused, fused_only=False):
    cfg = dataclasses.replace(synth.ATTN_CONFIGS["attn_small"], name="case", batch=B, seq=S, hidden=H, n_q=nq,
                              n_kv=nkv, d=d, w_std=0.05)
    inp = synth.make_attn_inputs(cfg, seed=B * 1000 + S)
    return cfg, inp, _run(cfg, t, inp, fused, fused_only)


@pytest.mark.parametrize("B,S,H,nq,nkv,d,t", CASES)
def test_attention_step_matches_oracle(B, S, H, nq, nkv, d, t):
    _check(B, S, H, nq, nkv, d, t, True)


@pytest.mark.parametrize("B,S,H,nq,nkv,d,t", FUSABLE)
def test_attention_step_unfused_matches_oracle(B, S, H, nq, nkv, d, t):
    """The materialised-score path on the shapes the fused kernels otherwise take."""
    _check(B, S, H, nq, nkv, d, t, False)


def _check(B, S, H, nq, nkv, d, t, fused, fused_only=False):
    cfg, inp, gpu = _case(B, S, H, nq, nkv, d, t, fused, fused_only)
    p = {k: inp[k] for k in NAMES}
    ora = O.attn_sharded_step(p, inp["x"], inp["target"], cfg.eps, LR, t, B, nq, nkv)
    compare("y", gpu["y"], ora["y"], "bf16")
    assert abs(gpu["loss"] - ora["loss"]) <= 2e-2 * abs(ora["loss"])
    compare("dx", gpu["dx"], ora["grads"]["x"], "bf16")
    for k in NAMES:
        compare("d" + k, gpu["grads"][k], ora["grads"][k], "bf16")
        new = gpu["master"][k]
        w0 = np.asarray(inp[k], dtype=np.float32).astype(np.float64)
        compare("post_step_" + k, new, w0 - LR * ora["grads"][k], "bf16",
                extra=0.5 * np.spacing(np.abs(new).astype(np.float32)).astype(np.float64))


def test_attention_fused_only_long_sequence():
    """A fused-only context (no score square in its workspace) on a sequence
    longer than the unfused path admits: 4608 tokens, 36 key blocks."""
    _check(1, 4608, 256, 2, 1, 128, 1, True, fused_only=True)


def test_attention_fused_only_refuses_the_unfused_path():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_SHAPE, ERR_UNSUPPORTED, TPAttn, TPMLPError
    m = TPAttn(512, 128, 2, 2, 128, 512, max_t=2, fused_only=True)
    with pytest.raises(TPMLPError) as e:
        m.set_fused(False)
    assert e.value.status == ERR_UNSUPPORTED
    z = torch.zeros(384, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    wqkv = torch.zeros(6 * 128, 128, dtype=torch.bfloat16, device="cuda")
    wo = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TPMLPError) as e:  # seq 192: a multiple of 64 but not of 128
        m.forward(z, w, wqkv, wo, w, 1e-6, 1, 2, 192)
    assert e.value.status == ERR_SHAPE


def test_attention_errors():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_ORDER, ERR_SHAPE, TPAttn, TPMLPError
    m = TPAttn(256, 128, 2, 2, 64, 128, max_t=2)
    x = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    wqkv = torch.zeros(6 * 64, 128, dtype=torch.bfloat16, device="cuda")
    wo = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TPMLPError) as e:
        m.backward(x)
    assert e.value.status == ERR_ORDER
    for batch, seq, t in ((2, 100, 1), (4, 128, 1), (2, 128, 3)):  # seq % 64, tokens > max, t | n_kv
        with pytest.raises(TPMLPError) as e:
            m.forward(torch.zeros(batch * seq, 128, dtype=torch.bfloat16, device="cuda"), w, wqkv, wo, w, 1e-6, t,
                      batch, seq)
        assert e.value.status == ERR_SHAPE
    m.forward(x, w, wqkv, wo, w, 1e-6, 2, 2, 128)
    m.sync()
