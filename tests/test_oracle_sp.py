"""Pins for the oracle's sequence-parallel form (walkthrough, "Deep dive:
sequence parallelism, memory for free" and "Stage 7: finalize_model_grads"):

* the page's identity: a reduce-scatter followed by an all-gather is the
  all-reduce (bit for bit here, since both sum in rank order);
* the sequence-parallel step equals the dense block for every t and both
  activations, and a token count not divisible by t is rejected;
* leaving out the all-reduce of the norm-weight and output-bias gradients
  changes exactly those two (and their updates): every rank keeps the sum
  over its own tokens, which is the dense per-token contribution summed over
  that slice, and the slices add up to the dense gradient.  Everything else
  (y, loss, dx, the projection gradients) is unchanged -- the page's
  "trains, slowly diverging, with no crash".
"""
import numpy as np
import pytest

from oracle import tpmlp_oracle as O


def _fixture(seed, N, H, F, act):
    rng = np.random.default_rng(seed)
    p = {"norm_w": 1.0 + 0.1 * rng.standard_normal(H), "w_down": 0.3 * rng.standard_normal((H, F)),
         "b_down": 0.05 * rng.standard_normal(H)}
    if act == "swiglu":
        p["w_gate_up"] = 0.3 * rng.standard_normal((2, F, H))
    else:
        p["w_1"] = 0.3 * rng.standard_normal((F, H))
        p["b_1"] = 0.05 * rng.standard_normal(F)
    return p, rng.standard_normal((N, H)), rng.standard_normal((N, H))


def test_reduce_scatter_then_all_gather_is_all_reduce():
    rng = np.random.default_rng(2)
    for t in (1, 2, 3, 4, 8):
        parts = [rng.standard_normal((8 * t, 5)) for _ in range(t)]
        rs = O.reduce_scatter_to_sequence_parallel_region(parts)
        assert all(r.shape == (8, 5) for r in rs)
        ag = O.gather_from_sequence_parallel_region(rs)
        np.testing.assert_array_equal(ag, O.reduce_from_tp_region_forward(parts))


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sp_step_equals_dense(act, t):
    p, x, tgt = _fixture(4, 16, 8, 24, act)
    d = O.dense_step(p, x, tgt, 1e-6, 0.1, act)
    s = O.sp_step(p, x, tgt, 1e-6, 0.1, t, act)
    close = lambda a, b: np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
    close(s["y"], d["y"])
    assert s["loss"] == pytest.approx(d["loss"], rel=1e-13)
    close(s["dy"], d["dy"])
    close(s["grads"]["x"], d["grads"]["x"])
    for k in p:
        close(s["grads"][k], d["grads"][k])
        close(s["new_params"][k], d["new_params"][k])
    # every rank ends with the same replicated gradients
    for rk in s["ranks"]:
        close(rk["grads"]["norm_w"], d["grads"]["norm_w"])
        close(rk["grads"]["b_down"], d["grads"]["b_down"])


def test_sp_rejects_indivisible_tokens():
    p, x, tgt = _fixture(1, 10, 8, 24, "swiglu")
    with pytest.raises(O.ShapeError):
        O.sp_step(p, x, tgt, 1e-6, 0.1, 4)
    with pytest.raises(O.ShapeError):
        O.sp_step(p, x[:8], tgt[:8], 1e-6, 0.1, 5)  # neither 8 tokens nor ffn 24 divide by 5


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
@pytest.mark.parametrize("t", [2, 4])
def test_sp_skipped_grad_sync_pattern(act, t):
    N = 16
    p, x, tgt = _fixture(8, N, 8, 24, act)
    d = O.dense_step(p, x, tgt, 1e-6, 0.1, act)
    c = d["cache"]
    dn = d["grads"]["_dn"]
    for view in range(t):
        s = O.sp_step(p, x, tgt, 1e-6, 0.1, t, act, skip_sp_grad_sync=True, view_rank=view)
        close = lambda a, b: np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
        close(s["y"], d["y"])
        close(s["grads"]["x"], d["grads"]["x"])
        for k in p:
            if k not in ("norm_w", "b_down"):
                close(s["grads"][k], d["grads"][k])
        lo, hi = O.token_interval(N, t, view)
        close(s["grads"]["norm_w"], np.sum(dn[lo:hi] * c["xhat"][lo:hi], axis=0))
        close(s["grads"]["b_down"], np.sum(d["dy"][lo:hi], axis=0))
        assert not np.allclose(s["grads"]["norm_w"], d["grads"]["norm_w"], rtol=1e-6, atol=0)
        assert not np.allclose(s["new_params"]["norm_w"], d["new_params"]["norm_w"], rtol=1e-9, atol=0)
        # the slices add up to the synchronised gradient
        close(sum(rk["local_norm_w_grad"] for rk in s["ranks"]), d["grads"]["norm_w"])
        close(sum(rk["local_b_down_grad"] for rk in s["ranks"]), d["grads"]["b_down"])
