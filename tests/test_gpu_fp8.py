"""FP8 (E4M3) building blocks on the GPU against the oracle, through the C ABI.

* ``tpmlp_fp8_quantize``: the codes (row-major and transposed) are
  bit-identical to the oracle's ``quantize_e4m3`` of the same bf16 values --
  both sides form x * s in float32 from the same float32 scale, so the
  rounding decision is taken in the same precision -- and 1 / s matches.
  The sign of a zero code is not compared.  Shapes cover several 64x64
  tiles, ragged rows and columns, a single row, zero rows, an all-zero
  tensor and magnitudes from 1e-30 to 1e30.
* ``tpmlp_fp8_gemm``: the tensor-core product of GPU-quantised operands
  against the oracle's ``fp8_linear`` of the same bf16 inputs (which
  quantises them itself).  Products of two codes are exact in float32, so
  the only differences are the order and precision of the float32 sums and
  the final scaling; the bound is the fp32 tolerance of the other parity
  tests.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import tpmlp_oracle as O
from tests._util import compare, to_np

pytestmark = pytest.mark.gpu


def _bf16_input(seed, rows, cols, scale):
    x = synth.round_to_bf16(synth.normal(seed, 31, (rows, cols), 0.0, 1.0) * scale)
    return x, torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).cuda()


def _codes_equal(gpu_codes, ora_codes):
    g = np.asarray(gpu_codes, dtype=np.uint8).copy()
    o = np.asarray(ora_codes, dtype=np.uint8).copy()
    g[g == 0x80] = 0
    o[o == 0x80] = 0
    np.testing.assert_array_equal(g, o)


@pytest.mark.parametrize("rows,cols,scale", [(300, 512, 1.0), (77, 328, 1e-6), (1029, 2048, 30.0), (1, 8, 1.0),
                                             (64, 64, 1e-30), (130, 136, 1e30), (0, 64, 1.0)])
def test_quantize_bit_exact(rows, cols, scale):
    from tensor_transformer_mlp_rmsnorm_gb300 import fp8_quantize
    x, xd = _bf16_input(rows + cols, rows, cols, scale)
    if rows > 2:
        x[1, :] = 0.0  # a zero row
        xd[1, :] = 0
    q, qt, inv = fp8_quantize(xd)
    torch.cuda.synchronize()
    codes, s = O.quantize_e4m3(x)
    _codes_equal(q[:, :cols].cpu().numpy(), codes)
    _codes_equal(qt[:, :rows].cpu().numpy(), codes.T)
    assert float(inv.item()) == float(np.float32(1.0) / s)


def test_quantize_all_zero_and_one_sided_outputs():
    from tensor_transformer_mlp_rmsnorm_gb300 import fp8_quantize
    xd = torch.zeros(100, 96, dtype=torch.bfloat16, device="cuda")
    q, qt, inv = fp8_quantize(xd)
    assert float(inv.item()) == 1.0
    assert int(q[:, :96].max().item()) == 0 and int(qt[:, :100].max().item()) == 0
    x, xd = _bf16_input(5, 200, 256, 2.0)
    q1, none_t, inv1 = fp8_quantize(xd, transposed=False)
    none, qt1, inv2 = fp8_quantize(xd, rows_major=False)
    assert none_t is None and none is None
    codes, _ = O.quantize_e4m3(x)
    _codes_equal(q1[:, :256].cpu().numpy(), codes)
    _codes_equal(qt1[:, :200].cpu().numpy(), codes.T)
    assert float(inv1.item()) == float(inv2.item())


@pytest.mark.parametrize("M,N,K", [(300, 512, 1024), (77, 328, 200), (1029, 2048, 4096), (128, 256, 128),
                                   (4096, 1024, 768)])
def test_fp8_gemm_matches_oracle(M, N, K):
    from tensor_transformer_mlp_rmsnorm_gb300 import fp8_gemm, fp8_quantize
    a, ad = _bf16_input(M * 7 + K, M, K, 1.0)
    b, bd = _bf16_input(N * 5 + K, N, K, 0.02)
    qa, _, inva = fp8_quantize(ad, transposed=False)
    qb, _, invb = fp8_quantize(bd, transposed=False)
    c, status = fp8_gemm(qa, qb, K, inva, invb)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.fp8_linear(a, b)
    report = {}
    compare("fp8_gemm", to_np(c), ref, "f32", report)
    # and the quantisation really happened: FP8 differs from the exact product
    exact = a @ b.T
    assert np.linalg.norm(to_np(c) - exact) / np.linalg.norm(exact) > 1e-3


# ------------------------------------------------------------------ the FP8 training step

LR = 0.1


def _cfg(act, N, H, F):
    import dataclasses
    c = dataclasses.replace(synth.CONFIGS["bf16_h2048"].with_shape(N, H, F), act=act)
    return dataclasses.replace(c, b_1_std=0.01) if act == "gelu" else c


@pytest.mark.parametrize("act,N,H,F,t", [("swiglu", 300, 512, 1536, 4), ("gelu", 333, 384, 1280, 8),
                                         ("swiglu", 1024, 256, 2048, 1), ("swiglu", 77, 328, 1024, 8),
                                         ("swiglu", 600, 320, 1000, 1)])
def test_fp8_step_matches_fp8_oracle(act, N, H, F, t):
    """The step with every GEMM in FP8 against the oracle's FP8 step, which
    quantises the same stored (bf16) operands with the same per-tensor rule:
    the FP8 tolerance of tests/_util.py.  Against the exact step the FP8
    error must be present and inside the FP8 band."""
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    from tests._util import compare_step, gpu_step
    cfg = _cfg(act, N, H, F)
    inp = synth.make_inputs(cfg, seed=31)
    m = TPMLP(N, H, F, max_t=8, dtype="bf16", act=act)
    m.set_precision("fp8")
    gpu = gpu_step(cfg, inp, t, LR, mod=m)
    p = {k: inp[k] for k in synth.param_names(act)}
    ora = O.dense_step_fp8(p, inp["x"], inp["target"], cfg.eps, LR, act, store=synth.round_to_bf16)
    compare_step(cfg, gpu, ora, inp, LR, tol="fp8")
    exact = O.dense_step(p, inp["x"], inp["target"], cfg.eps, LR, act)
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    assert 1e-3 < rel(gpu["y"] - inp["x"], exact["y"] - inp["x"]) < 0.1
    gk = "w_gate_up" if act == "swiglu" else "w_1"
    assert 1e-3 < rel(gpu["grads"][gk], exact["grads"][gk]) < 0.15


def test_fp8_precision_errors():
    from tensor_transformer_mlp_rmsnorm_gb300 import ERR_UNSUPPORTED, TPMLP, TPMLPError
    m = TPMLP(16, 64, 256, max_t=8, dtype="f32", act="swiglu")
    with pytest.raises(TPMLPError) as e:
        m.set_precision("fp8")
    assert e.value.status == ERR_UNSUPPORTED
