"""Repeat determinism of the whole training step on the GPU.

Every reduction of the CUDA path runs in a fixed order (the shard sums in the
GEMM K loops, per-block partials of the token sums added in block order), so
the same step on the same inputs must give bit-identical results every time,
whatever the logical t and whatever the workspace held before.  A difference
between two runs is a race or a read of memory that the step did not write.

The step of the H=2048 workload (4096 tokens, F=5632; page "Megatron
tensor-parallel MLP", "Reproduce one dense training step") runs many times in
one process, cycling t over 1, 2, 4 and refilling the workspace with NaN bytes
before some runs; y, loss, dy, dx, every parameter gradient and the post-step
fp32 masters must equal the first run's bit for bit.  On a mismatch the
message names the tensor, the first differing element and its 32x32 block.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import device_inputs

pytestmark = pytest.mark.gpu

RUNS = 400


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_transformer_mlp_rmsnorm_gb300 import build
    build.build()


def _first_diff(name, a, b):
    bits = {torch.bfloat16: torch.int16, torch.float32: torch.int32}[a.dtype]
    idx = (a.view(bits) != b.view(bits)).nonzero()
    n = int(idx.shape[0])
    first = idx[0].tolist()
    where = f"first at {tuple(first)}"
    if len(first) >= 2:
        where += f", 32x32 block ({first[-2] // 32}, {first[-1] // 32})"
    return f"{name}: {n} elements differ from the first run; {where}"


def test_step_is_bitwise_deterministic():
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    cfg = synth.CONFIGS["bf16_h2048"]
    inp = synth.make_inputs(cfg)
    d = device_inputs(cfg, inp)
    names = synth.param_names(cfg.act)
    w0 = {k: d[k].clone() for k in names}
    m0 = {k: torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda() for k in names}
    m = TPMLP(cfg.tokens, cfg.hidden, cfg.ffn, max_t=8, dtype=cfg.dtype, act=cfg.act)
    params = {k: v.clone() for k, v in w0.items()}
    masters = {k: v.clone() for k, v in m0.items()}
    m.bind_master(masters)
    y = torch.empty_like(d["x"])
    dy, dx = torch.empty_like(y), torch.empty_like(y)
    grads = m.new_grads()
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")

    def run(t, nan_fill):
        for k in names:  # every run starts from the same parameters
            params[k].copy_(w0[k])
            masters[k].copy_(m0[k])
        if nan_fill:
            m.workspace[256:].fill_(0xFF)  # bytes past the status word: NaN in bf16 and f32
        m.forward(d["x"], params["norm_w"], params["w_gate_up"], params["w_down"], params["b_down"], cfg.eps, t,
                  y=y)
        m.mse_loss_grad(y, d["target"], dy=dy, loss=loss)
        m.backward(dy, dx=dx, grads=grads)
        m.sgd_step(0.1)
        out = {"y": y, "loss": loss, "dy": dy, "dx": dx}
        out.update({"d" + k: grads[k] for k in names})
        out.update({"master_" + k: masters[k] for k in names})
        return out

    ref = {k: v.clone() for k, v in run(4, False).items()}
    m.sync()
    for i in range(RUNS):
        cur = run((1, 2, 4)[i % 3], nan_fill=(i % 4 == 3))
        for k in ref:
            if not torch.equal(ref[k], cur[k]):
                m.sync()
                pytest.fail(f"run {i + 1} (t={(1, 2, 4)[i % 3]}): " + _first_diff(k, ref[k], cur[k]))
    m.sync()
