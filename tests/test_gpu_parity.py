"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs, element by element, for every logical t, both
activations, ragged shapes, the broken variants and the edge cases."""
import dataclasses

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


def oracle_step(cfg, inp, t, lr, **kw):
    p = {k: inp[k] for k in synth.param_names(cfg.act)}
    if t == 1 and not kw:
        return O.dense_step(p, inp["x"], inp["target"], cfg.eps, lr, cfg.act)
    return O.sharded_step(p, inp["x"], inp["target"], cfg.eps, lr, t, cfg.act, **kw)


# ------------------------------------------------------------ fp32 configuration
@pytest.mark.parametrize("t", [2, 1, 4, 8])
def test_fp32_small_every_t(t):
    cfg = synth.CONFIGS["fp32_small"]
    inp = synth.make_inputs(cfg)
    gpu = gpu_step(cfg, inp, t, cfg.lr)
    compare_step(cfg, gpu, oracle_step(cfg, inp, t, cfg.lr), inp, cfg.lr)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_fp32_ragged_shapes(act):
    base = synth.CONFIGS["fp32_small"]
    import dataclasses
    cfg = dataclasses.replace(base.with_shape(77, 40, 104), act=act, b_1_std=0.01 if act == "gelu" else 0.0,
                              b_down_std=0.01)
    inp = synth.make_inputs(cfg, seed=7)
    for t in (1, 13):
        gpu = gpu_step(cfg, inp, t, 0.1)
        compare_step(cfg, gpu, oracle_step(cfg, inp, t, 0.1), inp, 0.1)


# ------------------------------------------------------------ bf16, several tiles + ragged tails
BF16_SHAPES = [
    # tokens, hidden, ffn, t values
    (300, 512, 1536, (1, 2, 4, 8)),   # 3 m-tiles (ragged), 2 n-tiles, shards of 192 channels
    (77, 328, 1000, (1, 5)),          # everything ragged, F not a multiple of 64
    (1029, 256, 2048, (4,)),          # 9 m-tiles, K=tokens ragged in the weight gradients
    (600, 320, 1344, (1, 3)),         # H, F multiples of 64 but not of 256: partial 3-D boxes, skipped chunks
]


@pytest.mark.parametrize("N,H,F,ts", BF16_SHAPES)
def test_bf16_swiglu_tiles_and_tails(N, H, F, ts):
    cfg = synth.CONFIGS["bf16_h2048"].with_shape(N, H, F)
    inp = synth.make_inputs(cfg, seed=11)
    ora = O.dense_step({k: inp[k] for k in synth.param_names("swiglu")}, inp["x"], inp["target"], cfg.eps, 0.1)
    for t in ts:
        gpu = gpu_step(cfg, inp, t, 0.1)
        compare_step(cfg, gpu, ora, inp, 0.1)


@pytest.mark.parametrize("N,H,F,t", [(300, 512, 1536, 4), (77, 328, 1000, 1), (1029, 256, 2048, 2)])
def test_bf16_single_cta_tiles(N, H, F, t):
    """The single-CTA 128x256 tile shape (the default is CTA pairs with 256x256 tiles)."""
    from tensor_transformer_mlp_rmsnorm_gb300 import DBG_GEMM_SINGLE_CTA
    cfg = synth.CONFIGS["bf16_h2048"].with_shape(N, H, F)
    inp = synth.make_inputs(cfg, seed=13)
    ora = oracle_step(cfg, inp, t, 0.1)
    gpu = gpu_step(cfg, inp, t, 0.1, flags=DBG_GEMM_SINGLE_CTA)
    compare_step(cfg, gpu, ora, inp, 0.1)


def test_bf16_gelu_tiles_and_tails():
    cfg = synth.CONFIGS["bf16_gelu_h4096"].with_shape(333, 384, 1280)
    inp = synth.make_inputs(cfg, seed=12)
    for t in (1, 8):
        gpu = gpu_step(cfg, inp, t, 0.1)
        compare_step(cfg, gpu, oracle_step(cfg, inp, t, 0.1), inp, 0.1)


def test_bf16_config_h2048_full_every_t():
    """The whole bf16 H=2048 workload (4096 tokens, F=5632), element by element."""
    cfg = synth.CONFIGS["bf16_h2048"]
    inp = synth.make_inputs(cfg)
    ora = O.dense_step({k: inp[k] for k in synth.param_names("swiglu")}, inp["x"], inp["target"], cfg.eps, 0.1)
    for t in cfg.t_list:
        gpu = gpu_step(cfg, inp, t, 0.1)
        compare_step(cfg, gpu, ora, inp, 0.1)


@pytest.mark.parametrize("dtype,act", [("bf16", "swiglu"), ("bf16", "gelu"), ("f32", "swiglu")])
def test_uncommon_t(dtype, act):
    """Degrees other than the powers of two: t = 3, 12 and 48 on F = 1536 (shards of 512, 128
    and 32 channels; 32 is below one 64-wide k-block, so shard boundaries fall inside k-blocks).
    The step must match the oracle's t-rank decomposition, and, since the on-chip sum runs over
    the FFN axis in one order whatever t is, be bit-identical to t = 1."""
    base = synth.CONFIGS["bf16_h2048" if dtype == "bf16" else "fp32_small"]
    N, H = (300, 512) if dtype == "bf16" else (40, 128)
    cfg = dataclasses.replace(base.with_shape(N, H, 1536), act=act)
    if act == "gelu":
        cfg = dataclasses.replace(cfg, b_1_std=0.01)
    inp = synth.make_inputs(cfg, seed=41)
    one = gpu_step(cfg, inp, 1, 0.1)
    for t in (3, 12, 48):
        gpu = gpu_step(cfg, inp, t, 0.1)
        compare_step(cfg, gpu, oracle_step(cfg, inp, t, 0.1), inp, 0.1)
        for k in ("y", "dx"):
            np.testing.assert_array_equal(gpu[k], one[k], err_msg=(t, k))
        for k in gpu["grads"]:
            np.testing.assert_array_equal(gpu["grads"][k], one["grads"][k], err_msg=(t, k))


@pytest.mark.parametrize("N,H,ts", [(512, 256, ((1, 0), (4, 0), (4, 8))), (300, 328, ((3, 0), (3, 8)))])
def test_bf16_tail_split_long_contraction(N, H, ts):
    """Contractions long enough for the tail split along K (F = 12288, 2F = 24576) on a few
    tiles: the down and dN GEMMs run each tile in four K parts whose partial sums the first
    part adds, for CTA pairs and single-CTA tiles (flag 8), on whole and on ragged tiles
    (300 tokens, H = 328), against the oracle, and bit-identical on a repeat."""
    from tensor_transformer_mlp_rmsnorm_gb300 import DBG_GEMM_SINGLE_CTA
    assert DBG_GEMM_SINGLE_CTA == 8
    cfg = synth.CONFIGS["bf16_h2048"].with_shape(N, H, 12288)
    inp = synth.make_inputs(cfg, seed=21)
    for t, flags in ts:
        ora = oracle_step(cfg, inp, t, 0.1)
        gpu = gpu_step(cfg, inp, t, 0.1, flags=flags)
        compare_step(cfg, gpu, ora, inp, 0.1)
        again = gpu_step(cfg, inp, t, 0.1, flags=flags)
        for k in ("y", "dx"):
            assert np.array_equal(gpu[k], again[k]), (t, flags, k)
        for k in gpu["grads"]:
            assert np.array_equal(gpu["grads"][k], again["grads"][k]), (t, flags, k)


# ------------------------------------------------------------ broken variants ("Remove each collective")
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_skip_reductions_match_oracle(dtype):
    from tensor_transformer_mlp_rmsnorm_gb300 import DBG_SKIP_BWD_REDUCE, DBG_SKIP_FWD_REDUCE
    if dtype == "f32":
        cfg = synth.CONFIGS["fp32_small"]
    else:
        cfg = synth.CONFIGS["bf16_h2048"].with_shape(200, 256, 1024)
    inp = synth.make_inputs(cfg, seed=3)
    t = 4
    good = gpu_step(cfg, inp, t, 0.1)
    for flag, kw in ((DBG_SKIP_FWD_REDUCE, {"skip_forward_reduce": True}),
                     (DBG_SKIP_BWD_REDUCE, {"skip_backward_reduce": True})):
        for shard in (0, t - 1):
            ora = oracle_step(cfg, inp, t, 0.1, view_rank=shard, backward_dy="view", **kw)
            gpu = gpu_step(cfg, inp, t, 0.1, flags=flag, shard=shard)
            compare_step(cfg, gpu, ora, inp, 0.1)
            # The page's pattern through the GPU path, which is deterministic:
            # what a removed reduction cannot reach is bit-identical to the
            # good run, everything downstream of it differs.
            same = lambda a, b: np.array_equal(a, b)
            if flag == DBG_SKIP_FWD_REDUCE:
                assert not same(gpu["y"], good["y"]) and gpu["loss"] != good["loss"]
                for k in ("w_gate_up", "w_down", "norm_w", "b_down"):
                    assert not same(gpu["grads"][k], good["grads"][k]), k
            else:
                assert same(gpu["y"], good["y"]) and gpu["loss"] == good["loss"]
                for k in ("w_gate_up", "w_down", "b_down"):
                    assert same(gpu["grads"][k], good["grads"][k]), k
                assert not same(gpu["grads"]["norm_w"], good["grads"]["norm_w"])
            assert not same(gpu["dx"], good["dx"])


# ------------------------------------------------------------ edge cases
@pytest.mark.parametrize("dtype,act,N", [("bf16", "swiglu", 1), ("bf16", "gelu", 2), ("f32", "swiglu", 1)])
def test_one_or_two_tokens(dtype, act, N):
    """A one- or two-token batch: one ragged row tile in every GEMM, and weight-gradient
    contractions of one or two tokens."""
    base = synth.CONFIGS["bf16_h2048" if dtype == "bf16" else "fp32_small"]
    cfg = dataclasses.replace(base.with_shape(N, 256, 512), act=act)
    if act == "gelu":
        cfg = dataclasses.replace(cfg, b_1_std=0.01)
    inp = synth.make_inputs(cfg, seed=43)
    for t in (1, 2):
        compare_step(cfg, gpu_step(cfg, inp, t, 0.1), oracle_step(cfg, inp, t, 0.1), inp, 0.1)


def test_zero_tokens():
    import torch
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    cfg = synth.CONFIGS["bf16_h2048"].with_shape(0, 256, 512)
    m = TPMLP(16, 256, 512, max_t=2, dtype="bf16")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    x = torch.empty(0, 256, **bf)
    p = (torch.ones(256, **bf), torch.randn(2, 512, 256, **bf), torch.randn(256, 512, **bf), torch.zeros(256, **bf))
    y = m.forward(x, *p, cfg.eps, 2)
    loss, dy = m.mse_loss_grad(y, torch.empty(0, 256, **bf))
    dx, g = m.backward(dy)
    m.sync()
    assert y.shape == (0, 256) and float(loss.item()) == 0.0
    for v in g.values():
        assert float(v.abs().max()) == 0.0


def test_output_guard_bands():
    """Outputs written through the ABI stay inside their buffers."""
    import torch
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    cfg = synth.CONFIGS["bf16_h2048"].with_shape(77, 328, 1000)
    inp = synth.make_inputs(cfg, seed=5)
    from tests._util import device_inputs
    d = device_inputs(cfg, inp)
    m = TPMLP(cfg.tokens, cfg.hidden, cfg.ffn, max_t=1, dtype="bf16")
    G = 4096  # guard elements on each side

    def guarded(n, dtype):
        buf = torch.full((n + 2 * G,), float("nan"), dtype=dtype, device="cuda")
        return buf, buf[G:G + n]

    ybuf, y = guarded(cfg.tokens * cfg.hidden, torch.bfloat16)
    y = y.view(cfg.tokens, cfg.hidden)
    m.forward(d["x"], d["norm_w"], d["w_gate_up"], d["w_down"], d["b_down"], cfg.eps, 1, y=y)
    dybuf, dy = guarded(cfg.tokens * cfg.hidden, torch.bfloat16)
    dy = dy.view(cfg.tokens, cfg.hidden)
    m.mse_loss_grad(y, d["target"], dy=dy)
    dxbuf, dx = guarded(cfg.tokens * cfg.hidden, torch.bfloat16)
    dx = dx.view(cfg.tokens, cfg.hidden)
    grads, bufs = {}, []
    for k, shp in (("norm_w", (cfg.hidden,)), ("w_gate_up", (2, cfg.ffn, cfg.hidden)),
                   ("w_down", (cfg.hidden, cfg.ffn)), ("b_down", (cfg.hidden,))):
        b, v = guarded(int(np.prod(shp)), torch.float32)
        grads[k] = v.view(shp)
        bufs.append(b)
    m.backward(dy, dx=dx, grads=grads)
    m.sync()
    for b in [ybuf, dybuf, dxbuf] + bufs:
        assert torch.isnan(b[:G].float()).all() and torch.isnan(b[-G:].float()).all()
        assert not torch.isnan(b[G:-G].float()).any()


def test_forced_timeout_reports_and_recovers():
    from tensor_transformer_mlp_rmsnorm_gb300 import DBG_FORCE_TIMEOUT, ERR_TIMEOUT, TPMLP, TPMLPError
    for dtype in ("bf16", "f32"):
        cfg = (synth.CONFIGS["bf16_h2048"].with_shape(256, 256, 512) if dtype == "bf16"
               else synth.CONFIGS["fp32_small"])
        inp = synth.make_inputs(cfg, seed=9)
        m = TPMLP(cfg.tokens, cfg.hidden, cfg.ffn, max_t=2, dtype=dtype)
        from tests._util import device_inputs
        d = device_inputs(cfg, inp)
        m.set_debug(DBG_FORCE_TIMEOUT, 0)
        m.forward(d["x"], d["norm_w"], d["w_gate_up"], d["w_down"], d["b_down"], cfg.eps, 2)
        with pytest.raises(TPMLPError) as ei:
            m.sync()
        assert ei.value.status == ERR_TIMEOUT
        # the context and the device stay usable
        gpu = gpu_step(cfg, inp, 2, 0.1, mod=m)
        ora = oracle_step(cfg, inp, 2, 0.1)
        compare_step(cfg, gpu, ora, inp, 0.1)


def test_abi_errors_on_device():
    import torch
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_ARG, ERR_ORDER, ERR_SHAPE, TPMLP, TPMLPError, tpmlp
    m = TPMLP(64, 128, 384, max_t=8, dtype="bf16")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    x = torch.randn(64, 128, **bf)
    p = [torch.ones(128, **bf), torch.randn(2, 384, 128, **bf), torch.randn(128, 384, **bf), torch.zeros(128, **bf)]
    import ctypes
    dummy = torch.empty(64 * 384 * 2, dtype=torch.float32, device="cuda")
    dp = ctypes.c_void_p(dummy.data_ptr())
    assert tpmlp.lib().tpmlp_backward(m.ctx, dp, dp, dp, dp, None, dp, dp) == ERR_ORDER
    assert tpmlp.lib().tpmlp_mse_loss_grad(m.ctx, dp, dp, dp, dp) == ERR_ORDER
    with pytest.raises(TPMLPError) as e:
        m.backward(torch.randn(64, 128, **bf))
    assert e.value.status == ERR_ORDER
    with pytest.raises(TPMLPError) as e:
        m.sgd_step(0.1)
    assert e.value.status == ERR_ORDER
    with pytest.raises(TPMLPError) as e:
        m.forward(x, *p, 1e-6, 5)  # 384 % 5 != 0
    assert e.value.status == ERR_SHAPE
    with pytest.raises(TPMLPError) as e:
        m.forward(torch.randn(65, 128, **bf), *p, 1e-6, 2)  # tokens > max_tokens
    assert e.value.status == ERR_SHAPE
    # misaligned pointer straight through the C ABI
    y = torch.empty(64, 128, **bf)
    base = torch.empty(64 * 128 + 8, **bf)
    st = tpmlp.lib().tpmlp_forward(m.ctx, 64, ctypes.c_void_p(base.data_ptr() + 2), *[ctypes.c_void_p(t.data_ptr())
                                   for t in p[:2]], None, ctypes.c_void_p(p[2].data_ptr()),
                                   ctypes.c_void_p(p[3].data_ptr()), 1e-6, 2, ctypes.c_void_p(y.data_ptr()))
    assert st == ERR_ARG
