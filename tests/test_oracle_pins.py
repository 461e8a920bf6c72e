"""Pins for the CPU oracle: each check ties it to something other than itself.

* closed forms and textbook values (RMSNorm of a known row, SiLU/GeLU values
  from the standard normal table),
* a brute-force pure-Python evaluation of the dense block on the page's tiny
  fixture (catches a transposed weight or a wrong index),
* central finite differences of the loss for every parameter and the input
  (pins the hand-derived backward),
* the page's invariants: the t-rank decomposition equals the dense block for
  every t, F % t != 0 is rejected, the inspect-mode shapes, and the two
  fault patterns of "Remove each collective",
* SGD is a descent step; the seeded generator's known answers.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import tpmlp_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _params(seed, N, H, F, act, w_std=0.3, b_std=0.05, nw="rand"):
    rng = np.random.default_rng(seed)
    p = {"norm_w": (1.0 + 0.1 * rng.standard_normal(H)) if nw == "rand" else np.ones(H),
         "w_down": w_std * rng.standard_normal((H, F)),
         "b_down": b_std * rng.standard_normal(H)}
    if act == "swiglu":
        p["w_gate_up"] = w_std * rng.standard_normal((2, F, H))
    else:
        p["w_1"] = w_std * rng.standard_normal((F, H))
        p["b_1"] = b_std * rng.standard_normal(F)
    x = rng.standard_normal((N, H))
    tgt = rng.standard_normal((N, H))
    return p, x, tgt


def _maxrel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b)), 1e-30))


# --------------------------------------------------------------------------- closed forms


def test_rms_norm_known_row():
    # Row (3, 4): mean square 12.5, so the normed row is (3, 4) / sqrt(12.5).
    n, rstd, xhat = O.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 1.0]), 0.0)
    assert n[0, 0] == pytest.approx(0.848528137423857, rel=1e-14)
    assert n[0, 1] == pytest.approx(1.131370849898476, rel=1e-14)
    assert rstd[0] == pytest.approx(1.0 / math.sqrt(12.5), rel=1e-15)
    # Weight scales the output column-wise; eps sits inside the root.
    n2, _, _ = O.rms_norm(np.array([[3.0, 4.0]]), np.array([2.0, -1.0]), 0.0)
    np.testing.assert_allclose(n2, n * np.array([2.0, -1.0]), rtol=1e-15)
    c, eps = 0.5, 1e-6
    nc, _, _ = O.rms_norm(np.full((1, 16), c), np.ones(16), eps)
    np.testing.assert_allclose(nc, c / math.sqrt(c * c + eps), rtol=1e-15)
    nz, rz, _ = O.rms_norm(np.zeros((1, 4)), np.ones(4), 1e-6)
    assert np.all(nz == 0) and rz[0] == pytest.approx(1e3, rel=1e-12)


def test_activation_values():
    # Phi(1) = 0.8413447460685429, phi(1) = 0.24197072451914337 (standard normal table).
    assert O.gelu(np.array(1.0)) == pytest.approx(0.8413447460685429, rel=1e-14)
    assert O.gelu(np.array(-1.0)) == pytest.approx(-(1 - 0.8413447460685429), rel=1e-13)
    assert O.gelu_grad(np.array(1.0)) == pytest.approx(0.8413447460685429 + 0.24197072451914337, rel=1e-14)
    assert O.gelu_grad(np.array(0.0)) == 0.5 and O.gelu(np.array(0.0)) == 0.0
    assert O.silu(np.array(0.0)) == 0.0 and O.silu_grad(np.array(0.0)) == 0.5
    # sigmoid(ln 3) = 3/4 -> silu(ln 3) = 0.75 ln 3
    z = math.log(3.0)
    assert O.silu(np.array(z)) == pytest.approx(0.75 * z, rel=1e-15)
    assert O.silu_grad(np.array(z)) == pytest.approx(0.75 * (1 + z * 0.25), rel=1e-15)
    # asymptotes
    assert O.silu(np.array(40.0)) == pytest.approx(40.0, rel=1e-15)
    assert O.gelu(np.array(-40.0)) == pytest.approx(0.0, abs=1e-300)
    # derivative agrees with a central difference at several points
    for f, df in ((O.silu, O.silu_grad), (O.gelu, O.gelu_grad)):
        zz = np.linspace(-6, 6, 25)
        h = 1e-6
        np.testing.assert_allclose(df(zz), (f(zz + h) - f(zz - h)) / (2 * h), rtol=1e-8, atol=1e-9)


def _brute_forward(p, x, eps, act):
    """The dense block evaluated element by element with Python loops."""
    N, H = x.shape
    F = p["w_down"].shape[1]
    y = [[0.0] * H for _ in range(N)]
    for n in range(N):
        ss = sum(float(x[n, h]) ** 2 for h in range(H))
        r = 1.0 / math.sqrt(ss / H + eps)
        nr = [float(x[n, h]) * r * float(p["norm_w"][h]) for h in range(H)]
        a = []
        for f in range(F):
            if act == "swiglu":
                g = sum(nr[h] * float(p["w_gate_up"][0, f, h]) for h in range(H))
                u = sum(nr[h] * float(p["w_gate_up"][1, f, h]) for h in range(H))
                a.append(g / (1.0 + math.exp(-g)) * u)
            else:
                z = sum(nr[h] * float(p["w_1"][f, h]) for h in range(H)) + float(p["b_1"][f])
                a.append(0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0))))
        for h in range(H):
            y[n][h] = float(x[n, h]) + sum(a[f] * float(p["w_down"][h, f]) for f in range(F)) + float(p["b_down"][h])
    return np.array(y)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_dense_forward_brute_force(act):
    p, x, _ = _params(1, 6, 8, 12, act)
    y, _ = O.dense_forward(p, x, 1e-6, act)
    np.testing.assert_allclose(y, _brute_forward(p, x, 1e-6, act), rtol=1e-12, atol=1e-12)


def test_loss_and_dy_closed_form():
    y = np.array([[1.0, 2.0], [3.0, 4.0]])
    t = np.array([[0.0, 2.0], [1.0, 4.0]])
    loss, dy = O.mse_loss(y, t)
    assert loss == 0.5 * (1 + 0 + 4 + 0) / 4
    np.testing.assert_array_equal(dy, np.array([[0.25, 0.0], [0.5, 0.0]]))


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_backward_finite_differences(act):
    """Central differences of the loss for every element of every parameter and x."""
    eps = 1e-6
    p, x, tgt = _params(2, 6, 8, 12, act)
    step = O.dense_step(p, x, tgt, eps, 0.1, act)
    g = step["grads"]

    def loss_of(pp, xx):
        y, _ = O.dense_forward(pp, xx, eps, act)
        return O.mse_loss(y, tgt)[0]

    h = 1e-5
    for name in list(p) + ["x"]:
        base = x if name == "x" else p[name]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            for sgn in (1, -1):
                pert = base.copy()
                pert[idx] += sgn * h
                if name == "x":
                    val = loss_of(p, pert)
                else:
                    pp = dict(p)
                    pp[name] = pert
                    val = loss_of(pp, x)
                fd[idx] += sgn * val / (2 * h)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-9, err_msg=name)


def test_closed_form_zero_down_weight():
    p, x, tgt = _params(3, 5, 8, 12, "swiglu")
    p["w_down"] = np.zeros_like(p["w_down"])
    s = O.dense_step(p, x, tgt, 1e-6, 0.1)
    np.testing.assert_allclose(s["y"], x + p["b_down"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(s["grads"]["x"], s["dy"], rtol=0, atol=1e-18)
    assert np.all(s["grads"]["w_gate_up"] == 0) and np.all(s["grads"]["norm_w"] == 0)
    np.testing.assert_allclose(s["grads"]["b_down"], s["dy"].sum(0), rtol=1e-15)


def test_closed_form_zero_gate_up():
    p, x, tgt = _params(4, 5, 8, 12, "swiglu")
    p["w_gate_up"] = np.zeros_like(p["w_gate_up"])
    s = O.dense_step(p, x, tgt, 1e-6, 0.1)
    np.testing.assert_allclose(s["y"], x + p["b_down"], rtol=0, atol=1e-15)
    for k in ("w_down", "w_gate_up", "norm_w"):
        assert np.all(s["grads"][k] == 0), k
    np.testing.assert_allclose(s["grads"]["x"], s["dy"], rtol=0, atol=1e-18)


def test_sgd_is_descent_and_exact_identities():
    p, x, tgt = _params(5, 6, 8, 12, "swiglu")
    s = O.dense_step(p, x, tgt, 1e-6, 1e-3)
    y1, _ = O.dense_forward(s["new_params"], x, 1e-6)
    assert O.mse_loss(y1, tgt)[0] < s["loss"]
    q = O.sgd({"w": np.array([1.5, -2.0])}, {"w": np.array([1.5, -2.0])}, 1.0)
    assert np.all(q["w"] == 0.0)
    q0 = O.sgd({"w": np.array([1.5, -2.0])}, {"w": np.array([3.0, 4.0])}, 0.0)
    np.testing.assert_array_equal(q0["w"], [1.5, -2.0])


# --------------------------------------------------------------------------- page invariants


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sharded_equals_dense(act, t):
    """Central claim of "What this reconstruction proves": the t-rank step
    reproduces dense forward, loss, every gradient and the updated weights."""
    cfg = synth.CONFIGS["fp32_small"]
    p, x, tgt = _params(6, cfg.tokens, cfg.hidden, cfg.ffn, act, w_std=0.05)
    d = O.dense_step(p, x, tgt, 1e-6, 0.1, act)
    s = O.sharded_step(p, x, tgt, 1e-6, 0.1, t, act)
    assert _maxrel(s["y"], d["y"]) < 1e-13
    assert abs(s["loss"] - d["loss"]) <= 1e-13 * d["loss"]
    for k in d["grads"]:
        assert _maxrel(s["grads"][k], d["grads"][k]) < 1e-12, k
    for k in d["new_params"]:
        assert _maxrel(s["new_params"][k], d["new_params"][k]) < 1e-13, k
    # replicated parameters get identical gradients on every rank
    for r in s["ranks"]:
        np.testing.assert_array_equal(r["grads"]["norm_w"], s["ranks"][0]["grads"]["norm_w"])
        np.testing.assert_array_equal(r["grads"]["b_down"], s["ranks"][0]["grads"]["b_down"])


def test_ffn_not_divisible_rejected():
    p, x, tgt = _params(7, 6, 8, 12, "swiglu")
    with pytest.raises(O.ShapeError):
        O.sharded_step(p, x, tgt, 1e-6, 0.1, 8)
    with pytest.raises(O.ShapeError):
        O.shard_interval(12, 5, 0)
    assert O.shard_interval(12, 2, 1) == (6, 12)


def test_inspect_shapes_golden():
    gold = json.load(open(os.path.join(GOLDEN, "p2_inspect_shapes.json")))
    fx = gold["fixture"]
    tr = O.shape_trace(fx["S"], fx["B"], fx["H"], fx["F"], fx["P"])
    assert tr["dense_shapes"] == gold["dense_shapes"]
    assert tr["rank_local_shapes"] == gold["rank_local_shapes"]
    # the arrays the oracle actually builds have these shapes
    S, B, H, F, P = fx["S"], fx["B"], fx["H"], fx["F"], fx["P"]
    p, x, tgt = _params(8, S * B, H, F, "swiglu")
    q = O.local_params(p, P, 1, "swiglu")
    part, c = O.rank_forward(q, x, 1e-6, "swiglu")
    loc = gold["rank_local_shapes"]
    assert list(q["w_gate_up"].shape) == loc["gate_up_weight"]
    assert list(q["w_down"].shape) == loc["down_weight"]
    assert [S, B] + [c["gate"].shape[1]] == loc["gate"]
    assert [S, B] + [c["hidden"].shape[1]] == loc["swiglu"]
    assert [S, B] + [part.shape[1]] == loc["partial_output"]


def _diff_table(d, s):
    def md(a, b):
        return float(np.max(np.abs(np.asarray(a) - np.asarray(b))))
    return {
        "forward": md(s["y"], d["y"]),
        "loss": abs(s["loss"] - d["loss"]),
        "input_grad": md(s["grads"]["x"], d["grads"]["x"]),
        "norm_grad": md(s["grads"]["norm_w"], d["grads"]["norm_w"]),
        "gate_up_grad": md(s["grads"]["w_gate_up"], d["grads"]["w_gate_up"]),
        "down_grad": md(s["grads"]["w_down"], d["grads"]["w_down"]),
        "down_bias_grad": md(s["grads"]["b_down"], d["grads"]["b_down"]),
        "post_step_weight": max(md(s["new_params"][k], d["new_params"][k]) for k in d["new_params"]),
    }


@pytest.mark.parametrize("view", [0, 1])
def test_fault_patterns_match_page(view):
    """The two broken variants fail exactly where "Remove each collective" says."""
    gold = json.load(open(os.path.join(GOLDEN, "fault_pattern_p2.json")))
    fx = json.load(open(os.path.join(GOLDEN, "p2_inspect_shapes.json")))["fixture"]
    p, x, tgt = _params(9, fx["S"] * fx["B"], fx["H"], fx["F"], "swiglu")
    d = O.dense_step(p, x, tgt, 1e-6, 0.1)
    modes = {
        "equivalence": {},
        "missing_forward_reduce": {"skip_forward_reduce": True},
        "missing_backward_reduce": {"skip_backward_reduce": True},
    }
    for mode, kw in modes.items():
        s = O.sharded_step(p, x, tgt, 1e-6, 0.1, fx["P"], "swiglu", view_rank=view, **kw)
        diffs = _diff_table(d, s)
        for key, want in gold[mode].items():
            if want == "match":
                assert diffs[key] < 1e-13, (mode, key, diffs[key])
            else:
                assert diffs[key] > 1e-4, (mode, key, diffs[key])
    # Without the backward reduction the forward is bit-identical to the
    # equivalence run (the page prints the same 1.2665987e-07 for both).
    ok = O.sharded_step(p, x, tgt, 1e-6, 0.1, 2)
    nb = O.sharded_step(p, x, tgt, 1e-6, 0.1, 2, skip_backward_reduce=True, view_rank=view)
    np.testing.assert_array_equal(ok["y"], nb["y"])
    np.testing.assert_array_equal(ok["grads"]["w_gate_up"], nb["grads"]["w_gate_up"])


def test_single_view_backward_variants():
    """backward_dy='view' differs from 'own' only when the forward reduction is
    skipped, and then only through the f all-reduce (dx, norm grad) and the
    other ranks' shards."""
    p, x, tgt = _params(10, 6, 8, 12, "swiglu")
    for kw in ({}, {"skip_backward_reduce": True}):
        a = O.sharded_step(p, x, tgt, 1e-6, 0.1, 2, backward_dy="own", view_rank=1, **kw)
        b = O.sharded_step(p, x, tgt, 1e-6, 0.1, 2, backward_dy="view", view_rank=1, **kw)
        for k in a["grads"]:
            np.testing.assert_array_equal(a["grads"][k], b["grads"][k])
    a = O.sharded_step(p, x, tgt, 1e-6, 0.1, 2, skip_forward_reduce=True, backward_dy="own", view_rank=1)
    b = O.sharded_step(p, x, tgt, 1e-6, 0.1, 2, skip_forward_reduce=True, backward_dy="view", view_rank=1)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["grads"]["b_down"], b["grads"]["b_down"])
    # the view rank's own shard of the weight gradients is the same either way
    np.testing.assert_array_equal(a["grads"]["w_down"][:, 6:], b["grads"]["w_down"][:, 6:])
    np.testing.assert_array_equal(a["grads"]["w_gate_up"][:, 6:], b["grads"]["w_gate_up"][:, 6:])
    assert np.max(np.abs(a["grads"]["x"] - b["grads"]["x"])) > 1e-6


# --------------------------------------------------------------------------- generator


def test_generator_known_answers():
    # splitmix64 from state 0: first output 0xE220A8397B1DCDAF (published test vector)
    u = synth._u64_block(0, 0, 3)
    assert int(u[0]) == 0xE220A8397B1DCDAF
    assert int(u[1]) == 0x6E789E6AA1B965F4
    assert int(u[2]) == 0x06C45D188009454F
    a = synth.normal(1234, 1, (1 << 20,))
    assert abs(a.mean()) < 5e-3 and abs(a.std() - 1) < 5e-3
    # independent of chunking and of the requested shape
    big = synth.normal(1234, 1, (1 << 23,))
    np.testing.assert_array_equal(big[: 1 << 20], a)
    np.testing.assert_array_equal(synth.normal(7, 3, (4, 5)).ravel(), synth.normal(7, 3, (20,)))


def test_bf16_rounding():
    v = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -7, -3.0 + 2 ** -7, 1e-20])
    r = synth.round_to_bf16(v)
    assert r[0] == 1.0                      # tie -> even
    assert r[1] == 1.0 + 2 ** -6            # tie -> even (upwards)
    assert r[2] == 1.0 + 2 ** -7            # representable
    assert r[3] == -3.0                     # exactly half an ulp (2^-6 on [2,4)): tie -> even
    assert abs(r[4] - 1e-20) / 1e-20 < 2 ** -8
    assert synth.bf16_bits(np.array([1.0]))[0] == 0x3F80
