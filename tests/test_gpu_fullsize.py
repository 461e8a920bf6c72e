"""Parity at the full workload sizes, in the launch configuration the
benchmark times (same library calls, same t, same dtypes).

* Element by element against the oracle's whole dense step in float64 (page
  "Megatron tensor-parallel MLP", "Reproduce one dense training step": the
  output, the loss, the input gradient, every parameter gradient and the
  weights after one update), at the GeLU workload (8192 tokens, H 4096,
  F 16384, t = 8), the Llama-3-8B-shaped benchmark workload (16384 tokens,
  H 4096, F 14336, t = 8) and the 70B shape (H 8192, F 28672, t = 8) at 512,
  2048 and 8192 tokens.  The oracle takes tens of seconds of host time for
  each of these.
* At the 70B shape's 32768 tokens the oracle cannot afford the whole step, so
  sampled token rows are checked element by element (a token's output y and
  input gradient dx depend only on that token's row and the weights), and the
  reductions over tokens by identities that hold at any size, evaluated in
  float64 on the GPU's outputs:
    sum(db_down)                    = sum over tokens of dy
    sum(dW_down * W_down)           = sum(dy * (y - x - b_down))
    sum(dW_gate_up * W_gate_up)     = sum(dnorm_w * norm_w)
                                      (G, U are linear in W_gate_up and n = xhat * norm_w)
    (dx - dy) . x = 0 for every row  (RMSNorm is scale invariant, up to eps)
    loss = 0.5 mean((y - target)^2)
  The identities are also checked at the other sizes, as extra checks.
* The logical degree t only fixes where shard boundaries fall inside the
  accumulation order, which runs over the FFN axis in shard order either way,
  so t = 4 and t = 8 give bit-identical results.
"""
import numpy as np
import pytest

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, compare_step, gpu_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_transformer_mlp_rmsnorm_gb300 import build
    build.build()


def sampled_rows(N, k=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, N - 1, N // 2, (N // 128) * 128 - 1 if N >= 128 else 0}
    rows |= set(int(r) for r in rng.integers(0, N, size=k))
    return np.array(sorted(rows))


def oracle_rows(cfg, inp, rows):
    """y, dy and dx of the sampled token rows (each row is independent)."""
    p = {k: inp[k] for k in synth.param_names(cfg.act)}
    x = inp["x"][rows]
    y, c = O.dense_forward(p, x, cfg.eps, cfg.act)
    dy = (y - inp["target"][rows]) / (cfg.tokens * cfg.hidden)
    g = O.dense_backward(p, c, dy)
    return y, dy, g["x"]


def check_identities(cfg, inp, gpu, rel=2e-2):
    x = inp["x"]
    wkey = "w_gate_up" if cfg.act == "swiglu" else "w_1"
    g = gpu["grads"]
    dy = gpu["dy"]

    def close(a, b, what):
        assert abs(a - b) <= rel * max(abs(a), abs(b)), (what, a, b)

    close(float(np.sum(g["b_down"])), float(np.sum(dy)), "sum db_down")
    mlp_out = gpu["y"] - x - inp["b_down"]
    close(float(np.sum(g["w_down"] * inp["w_down"])), float(np.sum(dy * mlp_out)), "dW_down . W_down")
    close(float(np.sum(g[wkey] * inp[wkey])), float(np.sum(g["norm_w"] * inp["norm_w"])),
          "dW_gate_up . W_gate_up")
    dxn = gpu["dx"] - dy
    num = np.abs(np.sum(dxn * x, axis=1))
    den = np.sum(np.abs(dxn) * np.abs(x), axis=1) + 1e-300
    assert np.max(num / den) < 1e-2, float(np.max(num / den))
    loss = 0.5 * float(np.mean((gpu["y"] - inp["target"]) ** 2))
    close(gpu["loss"], loss, "loss")


def run_case(cfg, t, lr):
    """Sampled rows element by element plus the identities (sizes the oracle cannot do whole)."""
    inp = synth.make_inputs(cfg)
    gpu = gpu_step(cfg, inp, t, lr, with_params=False)
    rows = sampled_rows(cfg.tokens)
    y, dy, dx = oracle_rows(cfg, inp, rows)
    compare("y_rows", gpu["y"][rows], y, cfg.dtype)
    compare("dy_rows", gpu["dy"][rows], dy, cfg.dtype)
    compare("dx_rows", gpu["dx"][rows], dx, cfg.dtype)
    check_identities(cfg, inp, gpu)
    return inp, gpu


def full_case(cfg, t, lr):
    """The whole step element by element against the oracle's dense step in float64."""
    inp = synth.make_inputs(cfg)
    gpu = gpu_step(cfg, inp, t, lr)
    del gpu["new_params"]  # the post-step check reads the fp32 masters
    p = {k: inp[k] for k in synth.param_names(cfg.act)}
    ora = O.dense_step(p, inp["x"], inp["target"], cfg.eps, lr, cfg.act)
    del ora["cache"], ora["new_params"]  # the post-step check forms w - lr * g itself
    report = {}
    compare_step(cfg, gpu, ora, inp, lr, report=report)
    compare("dy", gpu["dy"], ora["dy"], cfg.dtype)
    check_identities(cfg, inp, gpu)
    return inp, gpu


def test_llama8b_shape_bench_configuration():
    """The benchmark's workload: 16384 tokens, H 4096, F 14336, t = 8 (and t = 4), whole step."""
    cfg = synth.CONFIGS["bf16_llama8b"]
    inp, g8 = full_case(cfg, 8, cfg.lr)
    g4 = gpu_step(cfg, inp, 4, cfg.lr, with_params=False)
    for k in ("y", "dx"):
        np.testing.assert_array_equal(g8[k], g4[k])
    for k in g8["grads"]:
        np.testing.assert_array_equal(g8["grads"][k], g4["grads"][k])


def test_gelu_h4096_full():
    cfg = synth.CONFIGS["bf16_gelu_h4096"]
    full_case(cfg, 8, cfg.lr)


@pytest.mark.parametrize("tokens", [512, 2048, 8192])
def test_70b_shape_full(tokens):
    cfg = synth.CONFIGS["bf16_70b_n2048"].with_tokens(tokens)
    full_case(cfg, 8, cfg.lr)


def test_70b_shape_32768_sampled():
    cfg = synth.CONFIGS["bf16_70b_n2048"].with_tokens(32768)
    run_case(cfg, 8, cfg.lr)
