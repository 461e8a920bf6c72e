"""Pins for the oracle's FP8 (E4M3) pieces:

* the code table against the format's definition (127 finite non-negative
  values, strictly increasing, subnormals m/8 * 2^-6, largest 448) and every
  finite code round-trips;
* rounding against PyTorch's own ``float8_e4m3fn`` cast (an independent
  implementation) on random values and on every midpoint between adjacent
  codes, where ties go to the even code;
* saturation to +-448 and NaN;
* the per-tensor scale and quantization closed forms (the absolute maximum
  lands on 448);
* ``fp8_linear`` is exact when the operands are already representable with
  scale 1, and otherwise within the E4M3 rounding bound;
* the FP8 step stays within the FP8 error band of the exact dense step.
"""
import numpy as np
import pytest

from oracle import tpmlp_oracle as O

torch = pytest.importorskip("torch")


def _torch_codes(x):
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_table_definition():
    t = O.E4M3_TABLE
    assert len(t) == 127 and t[0] == 0.0 and t[-1] == 448.0
    assert np.all(np.diff(t) > 0)
    assert t[1] == 2.0 ** -9 and t[7] == 7 * 2.0 ** -9 and t[8] == 2.0 ** -6  # subnormals, then 1.0 * 2^-6
    assert t[0x38] == 1.0 and t[0x39] == 1.125 and t[0x7D] == 416.0
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = O.e4m3_encode(O.e4m3_decode(codes))
    np.testing.assert_array_equal(back, codes)
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_rounding_matches_torch_random():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-4, 2.5, 20000),
                        rng.uniform(-448, 448, 5000)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = O.e4m3_encode(x)
    theirs = _torch_codes(x)
    zero = (ours & 0x7F) == 0
    np.testing.assert_array_equal(ours[~zero], theirs[~zero])
    np.testing.assert_array_equal(theirs[zero] & 0x7F, 0)  # zero codes: the sign of zero is not compared


def test_ties_go_to_even_code():
    t = O.E4M3_TABLE
    mids = (t[:-1] + t[1:]) / 2.0  # exactly representable in float32
    codes = O.e4m3_encode(mids)
    lo = np.arange(len(mids))
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    np.testing.assert_array_equal(codes, expect)
    np.testing.assert_array_equal(_torch_codes(mids), expect)
    np.testing.assert_array_equal(O.e4m3_encode(-mids), expect | 0x80)


def test_saturation_and_nan():
    np.testing.assert_array_equal(O.e4m3_encode([448.0, 460.0, 1e30, -500.0]), [0x7E, 0x7E, 0x7E, 0xFE])
    assert O.e4m3_encode([np.nan])[0] == 0x7F


def test_scale_and_quantize_closed_forms():
    assert O.fp8_scale(448.0) == 1.0
    assert O.fp8_scale(2.0) == 224.0
    assert O.fp8_scale(0.0) == 1.0 and O.fp8_scale(np.inf) == 1.0
    rng = np.random.default_rng(1)
    for scale in (1e-7, 1e-3, 1.0, 300.0):
        x = rng.standard_normal((33, 17)) * scale
        q, s = O.quantize_e4m3(x)
        assert s == np.float32(448.0) / np.float32(np.max(np.abs(x.astype(np.float32))))
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert (q[i] & 0x7F) == 0x7E  # the largest magnitude lands on 448
        rel = np.abs(O.e4m3_decode(q) / s - x) / np.maximum(np.abs(x), 1e-300)
        normal = np.abs(x) * s >= 2.0 ** -6
        assert np.max(rel[normal]) <= 2.0 ** -4 * (1 + 1e-6)  # half a unit of the 3-bit mantissa


def test_fp8_linear_exact_when_representable():
    rng = np.random.default_rng(2)
    a = O.e4m3_decode(rng.integers(0, 0x7E, (24, 40)).astype(np.uint8) | (rng.integers(0, 2, (24, 40)) * 0x80).astype(np.uint8))
    b = O.e4m3_decode(rng.integers(0, 0x7E, (16, 40)).astype(np.uint8))
    a[0, 0], b[0, 0] = 448.0, -448.0  # amax 448 -> scale 1
    np.testing.assert_array_equal(O.fp8_linear(a, b), a @ b.T)


def test_fp8_linear_error_bound():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((64, 256))
    b = rng.standard_normal((48, 256)) * 1e-3
    exact = a @ b.T
    got = O.fp8_linear(a, b)
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    # independent relative rounding errors of at most 2^-4 per operand
    assert 1e-3 < rel < 2 * 2.0 ** -4


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_fp8_step_within_fp8_band(act):
    rng = np.random.default_rng(4)
    N, H, F = 32, 64, 128
    p = {"norm_w": 1.0 + 0.1 * rng.standard_normal(H), "w_down": 0.05 * rng.standard_normal((H, F)),
         "b_down": 0.01 * rng.standard_normal(H)}
    if act == "swiglu":
        p["w_gate_up"] = 0.05 * rng.standard_normal((2, F, H))
    else:
        p["w_1"] = 0.05 * rng.standard_normal((F, H))
        p["b_1"] = 0.01 * rng.standard_normal(F)
    x, tgt = rng.standard_normal((N, H)), rng.standard_normal((N, H))
    d = O.dense_step(p, x, tgt, 1e-6, 0.1, act)
    f = O.dense_step_fp8(p, x, tgt, 1e-6, 0.1, act)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 0 < rel(f["y"] - x, d["y"] - x) < 0.1  # the MLP output itself, not the residual
    for k in list(p) + ["x"]:
        assert 0 < rel(f["grads"][k], d["grads"][k]) < 0.15, k
