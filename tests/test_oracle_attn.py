"""Pins for the oracle's tensor-parallel attention sublayer:

* a pure-Python loop over sequences, heads, queries and keys (the causal
  softmax written out element by element) on a tiny grouped-query case --
  pins the head/group mapping and every reshape;
* central finite differences of the loss for every parameter and the input;
* closed forms: one-token sequences (attention returns the group's value);
  W_q = 0 (uniform weights over the causal prefix, so z_i is the mean of
  v_0..v_i); W_o = 0 (y = x + b_o);
* causality: perturbing token j of a sequence changes no earlier token and no
  other sequence;
* the t-rank decomposition with complete head groups per rank equals the
  dense sublayer for every t dividing n_kv (MHA, GQA, MQA), and an indivisible
  t is rejected.
"""
import math

import numpy as np
import pytest

from oracle import tpmlp_oracle as O


def _fixture(seed, B, S, H, n_q, n_kv, d, w=0.3):
    rng = np.random.default_rng(seed)
    p = {"norm_w": 1.0 + 0.1 * rng.standard_normal(H),
         "w_qkv": w * rng.standard_normal(((n_q + 2 * n_kv) * d, H)),
         "w_o": w * rng.standard_normal((H, n_q * d)), "b_o": 0.05 * rng.standard_normal(H)}
    return p, rng.standard_normal((B * S, H)), rng.standard_normal((B * S, H))


def _brute_attention(q, k, v, B, n_q, n_kv, d):
    N = len(q)
    S = N // B
    z = [[0.0] * (n_q * d) for _ in range(N)]
    for b in range(B):
        for h in range(n_q):
            g = h // (n_q // n_kv)
            for i in range(S):
                qi = q[b * S + i][h * d:(h + 1) * d]
                logits = []
                for j in range(i + 1):
                    kj = k[b * S + j][g * d:(g + 1) * d]
                    logits.append(sum(a * c for a, c in zip(qi, kj)) / math.sqrt(d))
                mx = max(logits)
                e = [math.exp(l - mx) for l in logits]
                tot = sum(e)
                for c in range(d):
                    z[b * S + i][h * d + c] = sum(e[j] / tot * v[b * S + j][g * d + c] for j in range(i + 1))
    return np.array(z)


def test_attention_brute_force():
    p, x, _ = _fixture(1, 2, 5, 12, 4, 2, 3)
    y, c = O.attn_dense_forward(p, x, 1e-6, 2, 4, 2)
    z = _brute_attention(c["q"].tolist(), c["k"].tolist(), c["v"].tolist(), 2, 4, 2, 3)
    np.testing.assert_allclose(c["z"], z, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y, x + z @ p["w_o"].T + p["b_o"], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (2, 2), (4, 1)])
def test_attention_finite_differences(n_q, n_kv):
    B, S, H, d = 2, 3, 6, 2
    p, x, tgt = _fixture(2, B, S, H, n_q, n_kv, d)
    base = O.attn_dense_step(p, x, tgt, 1e-6, 0.0, B, n_q, n_kv)
    h = 1e-6

    def loss(pp, xx):
        y, _ = O.attn_dense_forward(pp, xx, 1e-6, B, n_q, n_kv)
        return O.mse_loss(y, tgt)[0]

    for key in list(p) + ["x"]:
        arr = x if key == "x" else p[key]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            if key == "x":
                fd[idx] = (loss(p, a1) - loss(p, a2)) / (2 * h)
            else:
                fd[idx] = (loss(dict(p, **{key: a1}), x) - loss(dict(p, **{key: a2}), x)) / (2 * h)
        g = base["grads"][key]
        assert np.max(np.abs(fd - g)) <= 1e-6 * max(1.0, np.max(np.abs(g))) + 1e-9, key


def test_attention_closed_forms():
    # one-token sequences: softmax of one logit is 1, so z = v of the head's group
    p, x, _ = _fixture(3, 6, 1, 8, 4, 2, 2)
    _, c = O.attn_dense_forward(p, x, 1e-6, 6, 4, 2)
    v = c["v"]
    for h in range(4):
        g = h // 2
        np.testing.assert_allclose(c["z"][:, 2 * h:2 * h + 2], v[:, 2 * g:2 * g + 2], rtol=1e-14)
    # W_q = 0: every logit is 0, the weights are uniform over the causal prefix
    p, x, _ = _fixture(4, 2, 6, 8, 2, 1, 3)
    p["w_qkv"][:2 * 3] = 0.0
    _, c = O.attn_dense_forward(p, x, 1e-6, 2, 2, 1)
    v = c["v"].reshape(2, 6, 3)
    prefix_mean = np.cumsum(v, axis=1) / np.arange(1, 7)[None, :, None]
    for h in range(2):
        np.testing.assert_allclose(c["z"][:, 3 * h:3 * h + 3], prefix_mean.reshape(12, 3), rtol=1e-12)
    # W_o = 0: the sublayer is the identity plus the bias
    p, x, _ = _fixture(5, 2, 4, 8, 2, 2, 2)
    p["w_o"][:] = 0.0
    y, _ = O.attn_dense_forward(p, x, 1e-6, 2, 2, 2)
    np.testing.assert_array_equal(y, x + p["b_o"])


def test_attention_is_causal_per_sequence():
    B, S = 3, 5
    p, x, _ = _fixture(6, B, S, 8, 4, 2, 2)
    y0, _ = O.attn_dense_forward(p, x, 1e-6, B, 4, 2)
    for j in range(S):
        x1 = x.copy()
        x1[1 * S + j] += 1.0
        y1, _ = O.attn_dense_forward(p, x1, 1e-6, B, 4, 2)
        changed = np.any(np.abs(y1 - y0) > 0, axis=1).reshape(B, S)
        assert not changed[0].any() and not changed[2].any()
        assert not changed[1, :j].any() and changed[1, j:].all()


@pytest.mark.parametrize("n_q,n_kv,ts", [(8, 8, (1, 2, 4, 8)), (8, 4, (1, 2, 4)), (8, 1, (1,))])
def test_attention_sharded_equals_dense(n_q, n_kv, ts):
    p, x, tgt = _fixture(7, 2, 6, 16, n_q, n_kv, 2)
    d = O.attn_dense_step(p, x, tgt, 1e-6, 0.1, 2, n_q, n_kv)
    for t in ts:
        s = O.attn_sharded_step(p, x, tgt, 1e-6, 0.1, t, 2, n_q, n_kv)
        np.testing.assert_allclose(s["y"], d["y"], rtol=1e-12, atol=1e-14)
        for k in list(p) + ["x"]:
            np.testing.assert_allclose(s["grads"][k], d["grads"][k], rtol=1e-11, atol=1e-15)
            if k != "x":
                np.testing.assert_allclose(s["new_params"][k], d["new_params"][k], rtol=1e-12, atol=1e-15)
    with pytest.raises(O.ShapeError):
        O.attn_sharded_step(p, x, tgt, 1e-6, 0.1, 3, 2, n_q, n_kv)
