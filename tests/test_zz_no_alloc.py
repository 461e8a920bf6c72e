"""The loss entry point that allocates nothing.

Some callers cannot call cudaMalloc: their device memory belongs to a host
framework's pool and budget, or they run a latency-bound loop where an
allocation (which may synchronise the device) is not acceptable.
tpmlp_mse_loss_grad_noalloc serves them: it needs no context and no
workspace, keeping its partial sums in a fixed array inside the library (one
per block of a grid capped at the array's size, so no n is refused for its
sake).  These tests call it through the C ABI and check it against the context
entry point tpmlp_mse_loss_grad and against the oracle's mse_loss on two calls
in a row: the first large enough that the grid is capped, the second smaller,
so stale partials left in the shared array would show.  Invalid arguments are
refused on the host before any GPU work.

This file is collected last on purpose and is self-contained, so it passes
run alone in a fresh process or after every other test.
"""
import ctypes
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402


@pytest.fixture(scope="module")
def T():
    from tensor_transformer_mlp_rmsnorm_gb300 import build
    build.build()
    import tensor_transformer_mlp_rmsnorm_gb300 as T
    return T


def test_noalloc_refuses_invalid_arguments_on_the_host(T):
    L = T.lib()
    max_blocks = T.tpmlp.NOALLOC_LOSS_MAX_BLOCKS
    # refused on the host, before any CUDA call: no device needed
    assert L.tpmlp_mse_loss_grad_noalloc(T.F32, 12, None, None, None, None, None) == T.ERR_SHAPE
    assert L.tpmlp_mse_loss_grad_noalloc(T.BF16, -8, None, None, None, None, None) == T.ERR_SHAPE
    assert L.tpmlp_mse_loss_grad_noalloc(9, 16, None, None, None, None, None) == T.ERR_UNSUPPORTED
    # an n far beyond one partial sum per block of the fixed array is not a shape error: the
    # capped grid strides over it (here the NULL tensors are what is refused)
    big = 64 * max_blocks * 2048
    assert L.tpmlp_mse_loss_grad_noalloc(T.BF16, big, None, None, None, None, None) == T.ERR_ARG
    assert b"NULL" in L.tpmlp_last_error(None)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_context_entry_point_twice(T, dtype):
    import torch
    from tests._util import compare, to_dev
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from oracle import tpmlp_oracle as O
    H, F = 1024, 1024
    # tokens of the two calls: 3000 x 1024 elements need more blocks than the fixed array holds
    # (the grid is capped), 1001 x 1024 fewer, so partial sums left over from the first call
    # would be read by the second if it did not write every one it reads
    sizes = (3000, 1001)
    per_block = 256 * (8 if dtype == "bf16" else 4)
    assert sizes[0] * H > T.tpmlp.NOALLOC_LOSS_MAX_BLOCKS * per_block > sizes[1] * H
    # The context entry point needs a forward first (it takes the token count from it).
    m = T.TPMLP(max(sizes), H, F, max_t=1, dtype=dtype)
    cfg = synth.CONFIGS["bf16_h2048"].with_shape(max(sizes), H, F)
    inp = synth.make_inputs(cfg, seed=77)
    p = {k: to_dev(v, dtype) for k, v in inp.items()}
    L = T.lib()
    stream = torch.cuda.current_stream(dev)
    for call, n_tok in enumerate(sizes):
        m.forward(p["x"][:n_tok], p["norm_w"], p["w_gate_up"], p["w_down"], p["b_down"], 1e-6, 1)
        y = to_dev(synth.normal(100 + call, 1, (n_tok, H)), dtype)
        tgt = to_dev(synth.normal(200 + call, 1, (n_tok, H)), dtype)
        ref_loss, ref_dy = m.mse_loss_grad(y, tgt)
        dy = torch.full_like(y, float("nan"))
        loss = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
        st = L.tpmlp_mse_loss_grad_noalloc(T.BF16 if dtype == "bf16" else T.F32, y.numel(),
                                           ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(tgt.data_ptr()),
                                           ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                           ctypes.c_void_p(stream.cuda_stream))
        assert st == T.tpmlp.OK, L.tpmlp_last_error(None)
        torch.cuda.synchronize()
        got = dy.float().cpu().numpy().astype(np.float64)
        ref = ref_dy.float().cpu().numpy().astype(np.float64)
        compare("noalloc_dy", got, ref, dtype)
        a, b = float(loss.item()), float(ref_loss.item())
        rtol = 1e-5 if dtype == "f32" else 2e-2
        assert abs(a - b) <= rtol * abs(b), (call, a, b)
        # and against the oracle on the same stored values
        o_loss, o_dy = O.mse_loss(y.float().cpu().numpy().astype(np.float64),
                                  tgt.float().cpu().numpy().astype(np.float64))
        compare("noalloc_dy_vs_oracle", got, o_dy, dtype)
        assert abs(a - o_loss) <= rtol * abs(o_loss), (call, a, o_loss)
    m.sync()
