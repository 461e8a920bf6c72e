"""CPU oracle for the tensor-parallel pre-RMSNorm MLP sublayer (numpy, float64).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Sources (web pages, cited by title and section):

* "Megatron tensor-parallel MLP" (synapticradio.com/post/megatron-tensor-
  parallel-mlp) -- the dense block under test ("Start with the dense block"),
  the shared FFN interval, the column-parallel expansion ("Split the
  expansion"), the row-parallel contraction and its forward all-reduce
  ("Split the contraction"), the backward all-reduce ("Put the other
  collective in backward"), the one-step training comparison ("Reproduce one
  dense training step") and the two broken variants ("Remove each
  collective").
* "Megatron-LM walkthrough" (stanleyjacob.dev) -- the f and g operators
  ("Deep dive: tensor parallelism and the f and g operators"), the GeLU MLP
  built from ColumnParallelLinear/RowParallelLinear (Part II), fp32 master
  parameters and the clipped AdamW step ("Stage 8"), whose hyperparameters
  come from the launch example near the top of the page; the sequence-
  parallel form ("Deep dive: sequence parallelism, memory for free") and the
  all-reduce of its norm-weight gradients ("Stage 7: finalize_model_grads").
* "Megatron-LM Explained" (trishampatil.com) -- the GeLU MLP split A by
  columns, B by rows ("The MLP block: column-parallel, then row-parallel").
* "Megatron-Core Architecture: 5D Distributed Parallelism, ... FP8
  Transformer Engine" -- FP8 GEMMs with per-tensor scaling (its list of
  Megatron-Core subsystems, item 6); W_QKV split column-wise and W_out
  row-wise with one all-reduce for the attention block.
* "Megatron-LM Explained" -- "Self-attention: split across heads"; and the
  TP-MLP page's closing note on grouped-query attention with complete
  query/KV head groups per rank.

Readings where the pages are silent:

* RMSNorm is called but never defined: y = x * (mean_h x^2 + eps)^(-1/2) * w,
  eps inside the root, no centring, no bias.
* The display equations of the dense block are missing from the extracted
  text; the algebra is that of ``F.linear`` as used by the printed code
  (``linear(x, W) = x W^T``).
* GeLU is the exact erf form.
* Loss is 0.5 * mean((y - target)^2) over all N*H elements.
* SGD is plain ``w <- w - lr * g`` (no momentum, no weight decay).
* AdamW: Adam's published moment rates and epsilon (0.9, 0.999, 1e-8);
  decoupled decay in PyTorch's parametrisation, on the projection matrices
  only; clip coefficient max_norm / (norm + 1e-6) capped at 1; bias
  correction with a 1-based step count; the global norm counts replicated
  parameters once.
* Sequence parallelism: contiguous token slices per rank (N % t == 0); the
  output bias is added on the slice after the reduce-scatter, so its
  gradient, like the norm weight's, is a per-slice sum that the all-reduce
  completes; the loss is the mean over every token.
* FP8: E4M3 codes (the OCP "fn" encoding: no infinities, largest 448) for
  every GEMM operand, one scale per tensor from its current absolute maximum
  (448 / amax, float32; 1 if the tensor is all zero), round to nearest even
  with saturation, products summed exactly and divided by both scales.  The
  page names delayed scaling (a scale from earlier steps' maxima) without
  defining it; the current maximum is the limiting case of that history.
* Attention: W_qkv stacks the query, key and value rows [(n_q + 2 n_kv) d, H]
  (no bias); scores are scaled by 1/sqrt(d); the mask is causal (GPT-style
  decoder); no positional rotation is applied inside the sublayer; query head
  h reads group h // (n_q / n_kv); rank r holds KV groups
  [r n_kv / t, (r+1) n_kv / t) and their query heads; only the output
  projection has a bias, added once after the reduction.
* Backward formulas (never written on the pages) are derived by hand from the
  forward and pinned by central finite differences in the tests.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py``
against closed forms, brute-force loops, finite differences and the page's
invariants (sharded == dense; the two fault patterns).  No function is
"parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# Element-wise pieces
# ---------------------------------------------------------------------------


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float):
    """Pre-norm of the block ("Start with the dense block": ``rms_norm(x,
    norm_weight)``).  Returns (normed, rstd [N], xhat)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1)
    rstd = 1.0 / np.sqrt(ms + eps)
    xhat = x * rstd[:, None]
    return xhat * np.asarray(w, dtype=np.float64), rstd, xhat


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    """SiLU(z) = z * sigmoid(z) -- ``F.silu`` in the dense block."""
    return z * sigmoid(z)


def silu_grad(z):
    """d SiLU / dz = s * (1 + z * (1 - s)), s = sigmoid(z)."""
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


_ERF = np.vectorize(math.erf, otypes=[np.float64])


def _erf(z):
    try:
        from scipy.special import erf  # exact to double rounding
        return erf(z)
    except Exception:  # pragma: no cover - scipy absent
        return _ERF(z)


def gelu(z):
    """Exact GeLU, z * Phi(z) (Megatron-LM walkthrough, Part II ``gelu(y)``)."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def gelu_grad(z):
    """d GeLU / dz = Phi(z) + z * phi(z)."""
    return 0.5 * (1.0 + _erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def linear(x, w, b=None):
    """``F.linear(x, w, b) = x w^T + b`` (weights stored [out, in])."""
    y = x @ w.T
    return y if b is None else y + b


# ---------------------------------------------------------------------------
# Dense block (the result the sharded path must reproduce)
# ---------------------------------------------------------------------------


def dense_forward(p: dict, x: np.ndarray, eps: float, act: str = "swiglu"):
    """Dense pre-RMSNorm MLP ("Start with the dense block").

    SwiGLU: y = x + W_d (SiLU(W_g n) * (W_u n)) + b_d, n = RMSNorm(x).
    GeLU (walkthrough Part II; "The MLP block"): y = x + W_d GeLU(W_1 n + b_1) + b_d.
    Returns (y, cache)."""
    x = np.asarray(x, dtype=np.float64)
    n, rstd, xhat = rms_norm(x, p["norm_w"], eps)
    c = {"x": x, "n": n, "rstd": rstd, "xhat": xhat, "act": act}
    if act == "swiglu":
        gate = linear(n, p["w_gate_up"][0])
        up = linear(n, p["w_gate_up"][1])
        hidden = silu(gate) * up
        c.update(gate=gate, up=up)
    else:
        z = linear(n, p["w_1"], p["b_1"])
        hidden = gelu(z)
        c.update(z=z)
    c["hidden"] = hidden
    y = x + linear(hidden, p["w_down"], p["b_down"])
    return y, c


def mse_loss(y: np.ndarray, target: np.ndarray):
    """Loss of the training step: 0.5 * mean((y - target)^2); returns (loss, dy)."""
    d = np.asarray(y, dtype=np.float64) - np.asarray(target, dtype=np.float64)
    return 0.5 * float(np.mean(d * d)), d / d.size


def rms_norm_backward(dn, xhat, rstd, w):
    """Gradient through n = xhat * w, xhat = x * rstd.

    Returns (dx_norm, dnorm_w): dx_norm = rstd * (g - xhat * mean_h(g * xhat)),
    g = dn * w; dnorm_w = sum_tokens dn * xhat."""
    g = dn * w
    dxn = rstd[:, None] * (g - xhat * np.mean(g * xhat, axis=-1, keepdims=True))
    return dxn, np.sum(dn * xhat, axis=0)


def dense_backward(p: dict, c: dict, dy: np.ndarray) -> dict:
    """Backward of ``dense_forward`` (what autograd computes in the dense
    reference of "Reproduce one dense training step").  Keys of the result:
    x, norm_w, w_gate_up | (w_1, b_1), w_down, b_down."""
    g = {"b_down": np.sum(dy, axis=0), "w_down": dy.T @ c["hidden"]}
    dh = dy @ p["w_down"]
    if c["act"] == "swiglu":
        dgate = dh * c["up"] * silu_grad(c["gate"])
        dup = dh * silu(c["gate"])
        g["w_gate_up"] = np.stack([dgate.T @ c["n"], dup.T @ c["n"]])
        dn = dgate @ p["w_gate_up"][0] + dup @ p["w_gate_up"][1]
    else:
        dz = dh * gelu_grad(c["z"])
        g["w_1"] = dz.T @ c["n"]
        g["b_1"] = np.sum(dz, axis=0)
        dn = dz @ p["w_1"]
    dxn, g["norm_w"] = rms_norm_backward(dn, c["xhat"], c["rstd"], p["norm_w"])
    g["x"] = dy + dxn
    g["_dn"] = dn
    return g


def sgd(p: dict, g: dict, lr: float) -> dict:
    """Plain SGD, the update that closes the page's one-step comparison:
    w <- w - lr * g."""
    return {k: p[k] - lr * g[k] for k in p}


def dense_step(p: dict, x, target, eps: float, lr: float, act: str = "swiglu") -> dict:
    """Forward, loss, backward and SGD of the dense block."""
    y, c = dense_forward(p, x, eps, act)
    loss, dy = mse_loss(y, target)
    g = dense_backward(p, c, dy)
    return {"y": y, "loss": loss, "dy": dy, "grads": g, "new_params": sgd(p, {k: g[k] for k in p}, lr),
            "cache": c}


# ---------------------------------------------------------------------------
# Literal t-rank decomposition
# ---------------------------------------------------------------------------


class ShapeError(ValueError):
    pass


def shard_interval(ffn: int, t: int, rank: int):
    """Shared FFN interval of one rank ("Start with the dense block", the
    fixture's slicing): asserts F % t == 0; rank r owns [r F/t, (r+1) F/t)
    of the gate rows, the up rows and the down columns alike."""
    if t < 1 or ffn % t != 0:
        raise ShapeError(f"ffn={ffn} is not divisible by t={t}")
    local = ffn // t
    return rank * local, (rank + 1) * local


def local_params(p: dict, t: int, rank: int, act: str) -> dict:
    """Rank-local parameters: FFN-sliced projections, replicated norm_w/b_down."""
    F = p["w_down"].shape[1]
    lo, hi = shard_interval(F, t, rank)
    q = {"norm_w": p["norm_w"], "w_down": p["w_down"][:, lo:hi], "b_down": p["b_down"]}
    if act == "swiglu":
        q["w_gate_up"] = p["w_gate_up"][:, lo:hi, :]
    else:
        q["w_1"] = p["w_1"][lo:hi]
        q["b_1"] = p["b_1"][lo:hi]
    return q


def copy_to_tp_region_forward(n):
    """f forward: identity ("Put the other collective in backward")."""
    return n


def reduce_from_tp_region_forward(partials):
    """g forward: all-reduce(SUM) of the rank partials, summed in rank order
    0..t-1 ("Split the contraction")."""
    acc = np.zeros_like(partials[0])
    for pr in partials:
        acc = acc + pr
    return acc


def copy_to_tp_region_backward(local_grads):
    """f backward: all-reduce(SUM) of the rank-local normed-input gradients."""
    return reduce_from_tp_region_forward(local_grads)


def rank_forward(q: dict, x, eps: float, act: str):
    """One rank's work up to its partial output ("Split the expansion",
    "Split the contraction"): partial = local hidden @ W_d_local^T."""
    n, rstd, xhat = rms_norm(x, q["norm_w"], eps)
    partial, c = rank_forward_normed(q, copy_to_tp_region_forward(n), act)
    c.update(rstd=rstd, xhat=xhat)
    return partial, c


def rank_forward_normed(q: dict, n_par, act: str):
    """The tensor-parallel region of one rank, from the normed input it
    receives: column-parallel expansion, activation, row-parallel partial."""
    c = {"n": n_par, "act": act}
    if act == "swiglu":
        gate = linear(n_par, q["w_gate_up"][0])
        up = linear(n_par, q["w_gate_up"][1])
        c.update(gate=gate, up=up)
        hidden = silu(gate) * up
    else:
        z = linear(n_par, q["w_1"], q["b_1"])
        c["z"] = z
        hidden = gelu(z)
    c["hidden"] = hidden
    return linear(hidden, q["w_down"]), c


def rank_backward_local(q: dict, c: dict, dy):
    """Rank-local part of the backward, before the f all-reduce: local weight
    gradients and the local contribution to the normed-input gradient.
    g backward is the identity, so every rank starts from the same dy."""
    g = {"w_down": dy.T @ c["hidden"], "b_down": np.sum(dy, axis=0)}
    dh = dy @ q["w_down"]
    if c["act"] == "swiglu":
        dgate = dh * c["up"] * silu_grad(c["gate"])
        dup = dh * silu(c["gate"])
        g["w_gate_up"] = np.stack([dgate.T @ c["n"], dup.T @ c["n"]])
        dn_local = dgate @ q["w_gate_up"][0] + dup @ q["w_gate_up"][1]
    else:
        dz = dh * gelu_grad(c["z"])
        g["w_1"] = dz.T @ c["n"]
        g["b_1"] = np.sum(dz, axis=0)
        dn_local = dz @ q["w_1"]
    return g, dn_local


def sharded_step(p: dict, x, target, eps: float, lr: float, t: int, act: str = "swiglu",
                 skip_forward_reduce: bool = False, skip_backward_reduce: bool = False,
                 view_rank: int = 0, backward_dy: str = "own") -> dict:
    """One training step of the t-rank decomposition, rank by rank.

    ``skip_forward_reduce`` / ``skip_backward_reduce`` reproduce the two broken
    variants of "Remove each collective": the g (forward) or f (backward)
    all-reduce replaced by each rank's own local value.

    ``backward_dy``: "own" -- every rank back-propagates the dy of its own
    loss (the multi-process behaviour); "view" -- every rank uses the dy of
    ``view_rank`` (a single-process view; identical to "own" unless the forward
    reduction is skipped).

    Returns the quantities as rank ``view_rank`` sees them, with the sharded
    weights (gradients and updated values) assembled from all ranks, plus the
    per-rank records under "ranks"."""
    x = np.asarray(x, dtype=np.float64)
    F = p["w_down"].shape[1]
    shard_interval(F, t, 0)  # divisibility check
    qs = [local_params(p, t, r, act) for r in range(t)]
    parts, caches = [], []
    for r in range(t):
        pr, c = rank_forward(qs[r], x, eps, act)
        parts.append(pr)
        caches.append(c)
    if skip_forward_reduce:
        mlp_out = parts
    else:
        red = reduce_from_tp_region_forward(parts)
        mlp_out = [red for _ in range(t)]
    ys = [x + mlp_out[r] + p["b_down"] for r in range(t)]
    losses, dys = zip(*[mse_loss(ys[r], target) for r in range(t)])
    use_dy = list(dys) if backward_dy == "own" else [dys[view_rank]] * t
    gl, dnl = [], []
    for r in range(t):
        g, dn = rank_backward_local(qs[r], caches[r], use_dy[r])
        gl.append(g)
        dnl.append(dn)
    if skip_backward_reduce:
        dns = dnl
    else:
        red = copy_to_tp_region_backward(dnl)
        dns = [red for _ in range(t)]
    ranks = []
    for r in range(t):
        dxn, dnw = rms_norm_backward(dns[r], caches[r]["xhat"], caches[r]["rstd"], p["norm_w"])
        gr = dict(gl[r])
        gr["norm_w"] = dnw
        gr["x"] = use_dy[r] + dxn
        gr["_dn"] = dns[r]
        newq = {k: qs[r][k] - lr * gr[k] for k in qs[r]}
        ranks.append({"y": ys[r], "loss": losses[r], "dy": use_dy[r], "grads": gr, "new_params": newq})
    v = ranks[view_rank]
    grads = {"x": v["grads"]["x"], "norm_w": v["grads"]["norm_w"], "b_down": v["grads"]["b_down"],
             "_dn": v["grads"]["_dn"]}
    newp = {"norm_w": v["new_params"]["norm_w"], "b_down": v["new_params"]["b_down"]}
    grads["w_down"] = np.concatenate([rk["grads"]["w_down"] for rk in ranks], axis=1)
    newp["w_down"] = np.concatenate([rk["new_params"]["w_down"] for rk in ranks], axis=1)
    if act == "swiglu":
        grads["w_gate_up"] = np.concatenate([rk["grads"]["w_gate_up"] for rk in ranks], axis=1)
        newp["w_gate_up"] = np.concatenate([rk["new_params"]["w_gate_up"] for rk in ranks], axis=1)
    else:
        for k, ax in (("w_1", 0), ("b_1", 0)):
            grads[k] = np.concatenate([rk["grads"][k] for rk in ranks], axis=ax)
            newp[k] = np.concatenate([rk["new_params"][k] for rk in ranks], axis=ax)
    return {"y": v["y"], "loss": v["loss"], "dy": v["dy"], "grads": grads, "new_params": newp,
            "ranks": ranks}


# ---------------------------------------------------------------------------
# Shape trace ("Reproduce one dense training step", the inspect output)
# ---------------------------------------------------------------------------


def shape_trace(S: int, B: int, H: int, F: int, t: int) -> dict:
    """Dense and rank-local tensor shapes of the block laid out [S, B, H]."""
    lo, hi = shard_interval(F, t, 0)
    f = hi - lo
    return {
        "dense_shapes": {"x": [S, B, H], "norm_weight": [H], "w_gate_up": [2, F, H],
                         "w_down": [H, F], "output": [S, B, H]},
        "rank_local_shapes": {"gate_up_weight": [2, f, H], "gate": [S, B, f], "up": [S, B, f],
                              "swiglu": [S, B, f], "down_weight": [H, f],
                              "partial_output": [S, B, H]},
    }


# ---------------------------------------------------------------------------
# AdamW with global gradient-norm clipping (the optimizer step of the
# walkthrough, "Stage 8": the gradient norm is taken over every model-parallel
# dimension and clipped, then AdamW updates the fp32 master parameters; its
# launch example sets --weight-decay 0.1, --clip-grad 1.0 and --lr 1.5e-4)
# ---------------------------------------------------------------------------

# Unstated on the pages: the moment rates and epsilon are Adam's published
# defaults (Kingma & Ba); the decay follows the decoupled form of Loshchilov &
# Hutter in PyTorch's parametrisation (w <- w - lr*wd*w - lr*adam); decay
# applies to the projection matrices only, not to the norm weight or biases;
# the clip coefficient is max_norm / (norm + 1e-6), capped at 1.
ADAMW_DEFAULTS = {"lr": 1.5e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.1,
                  "max_grad_norm": 1.0}
CLIP_EPS = 1e-6
DECAYED = ("w_gate_up", "w_1", "w_down", "w_qkv", "w_o")  # MLP and attention projection matrices
REPLICATED = ("norm_w", "b_down")


def global_grad_norm(g: dict) -> float:
    """L2 norm of every parameter gradient taken together: sqrt(sum_k sum g_k^2)."""
    total = 0.0
    for k in sorted(g):
        total += float(np.sum(np.square(np.asarray(g[k], dtype=np.float64))))
    return math.sqrt(total)


def clip_coefficient(norm: float, max_norm: float) -> float:
    """Factor applied to every gradient so the global norm is at most max_norm;
    1 when clipping is off (max_norm <= 0) or the norm is already within it."""
    if max_norm <= 0:
        return 1.0
    return min(1.0, max_norm / (norm + CLIP_EPS))


def adamw(p: dict, g: dict, m: dict, v: dict, step: int, lr: float, beta1: float, beta2: float,
          eps: float, weight_decay: float, max_grad_norm: float) -> dict:
    """One AdamW update of every parameter after global-norm clipping.

    For each parameter, with c the clip coefficient and k = step (1-based):
        g' = c g;  m <- b1 m + (1 - b1) g';  v <- b2 v + (1 - b2) g'^2
        w  <- w - lr wd w - lr (m / (1 - b1^k)) / (sqrt(v / (1 - b2^k)) + eps)
    wd is weight_decay for the projection matrices and 0 for the rest."""
    if step < 1:
        raise ValueError("step is 1-based")
    norm = global_grad_norm(g)
    c = clip_coefficient(norm, max_grad_norm)
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    new_p, new_m, new_v = {}, {}, {}
    for k in p:
        gk = c * np.asarray(g[k], dtype=np.float64)
        mk = beta1 * m[k] + (1.0 - beta1) * gk
        vk = beta2 * v[k] + (1.0 - beta2) * gk * gk
        wd = weight_decay if k in DECAYED else 0.0
        new_p[k] = p[k] - lr * wd * p[k] - lr * (mk / bc1) / (np.sqrt(vk / bc2) + eps)
        new_m[k] = mk
        new_v[k] = vk
    return {"params": new_p, "m": new_m, "v": new_v, "grad_norm": norm, "clip": c}


def dense_step_adamw(p: dict, x, target, eps: float, m: dict, v: dict, step: int, hp: dict,
                     act: str = "swiglu") -> dict:
    """Forward, loss, backward and one AdamW update of the dense block."""
    y, c = dense_forward(p, x, eps, act)
    loss, dy = mse_loss(y, target)
    g = dense_backward(p, c, dy)
    pg = {k: g[k] for k in p}
    upd = adamw(p, pg, m, v, step, **hp)
    return {"y": y, "loss": loss, "dy": dy, "grads": g, "new_params": upd["params"], "m": upd["m"],
            "v": upd["v"], "grad_norm": upd["grad_norm"], "clip": upd["clip"]}


def rank_grad_sqnorm(rank_grads: dict, rank: int, count_replicated_once: bool = True) -> float:
    """One rank's share of the squared global norm: its FFN-sliced gradients,
    plus the replicated ones (norm_w, b_down), which every rank holds
    identically and which only rank 0 contributes.  With
    ``count_replicated_once=False`` every rank adds them (the double-counting
    mistake)."""
    total = 0.0
    for k, gk in rank_grads.items():
        if k in ("x", "_dn"):
            continue
        if k in REPLICATED and count_replicated_once and rank != 0:
            continue
        total += float(np.sum(np.square(gk)))
    return total


def sharded_grad_norm(ranks: list, count_replicated_once: bool = True) -> float:
    """Global norm across the t ranks: each rank's squared share, summed in
    rank order (the all-reduce), then the square root."""
    return math.sqrt(reduce_from_tp_region_forward(
        [np.float64(rank_grad_sqnorm(rk["grads"], r, count_replicated_once)) for r, rk in enumerate(ranks)]))


# ---------------------------------------------------------------------------
# Sequence-parallel form (walkthrough, "Deep dive: sequence parallelism,
# memory for free"; "Stage 7: finalize_model_grads"): the regions outside the
# tensor-parallel linears (RMSNorm, residual, bias) hold a slice of the tokens
# per rank; an all-gather enters the tensor-parallel region and a
# reduce-scatter leaves it; the gradients of the replicated norm weight and
# output bias, each computed from one rank's tokens, are all-reduced.
# ---------------------------------------------------------------------------


def token_interval(tokens: int, t: int, rank: int):
    """Rank r's contiguous token slice [r N/t, (r+1) N/t); N % t == 0."""
    if t < 1 or tokens % t != 0:
        raise ShapeError(f"tokens={tokens} is not divisible by t={t}")
    n = tokens // t
    return rank * n, (rank + 1) * n


def gather_from_sequence_parallel_region(shards):
    """All-gather along the tokens: the rank slices concatenated in rank order."""
    return np.concatenate(shards, axis=0)


def reduce_scatter_to_sequence_parallel_region(partials):
    """Reduce-scatter along the tokens: rank r receives the sum, in rank order,
    of every rank's rows [r N/t, (r+1) N/t)."""
    t = len(partials)
    out = []
    for r in range(t):
        lo, hi = token_interval(partials[0].shape[0], t, r)
        out.append(reduce_from_tp_region_forward([pr[lo:hi] for pr in partials]))
    return out


def sp_step(p: dict, x, target, eps: float, lr: float, t: int, act: str = "swiglu",
            skip_sp_grad_sync: bool = False, view_rank: int = 0) -> dict:
    """One training step of the sequence-parallel decomposition, rank by rank.

    Forward: RMSNorm of each rank's token slice; all-gather into the full
    normed input; the tensor-parallel region; reduce-scatter of the partial
    outputs; bias and residual on the slice.  The loss is the mean over every
    token (its sum is all-reduced).  Backward: all-gather of dy (the
    reduce-scatter's backward); the rank-local weight gradients over every
    token; reduce-scatter of the normed-input gradients (the all-gather's
    backward); RMSNorm backward on the slice; then the all-reduce of the
    norm-weight and output-bias gradients, which ``skip_sp_grad_sync``
    leaves out (each rank keeps the sum over its own tokens).

    Returns the assembled tensors (token slices and FFN slices concatenated)
    and the replicated parameters' gradients as rank ``view_rank`` sees them,
    plus the per-rank records under "ranks"."""
    x = np.asarray(x, dtype=np.float64)
    N, H = x.shape
    F = p["w_down"].shape[1]
    shard_interval(F, t, 0)
    token_interval(N, t, 0)
    qs = [local_params(p, t, r, act) for r in range(t)]
    sl = [slice(*token_interval(N, t, r)) for r in range(t)]
    normed = [rms_norm(x[sl[r]], p["norm_w"], eps) for r in range(t)]
    n_full = gather_from_sequence_parallel_region([nr[0] for nr in normed])
    parts, caches = [], []
    for r in range(t):
        pr, c = rank_forward_normed(qs[r], n_full, act)
        parts.append(pr)
        caches.append(c)
    out = reduce_scatter_to_sequence_parallel_region(parts)
    ys = [x[sl[r]] + out[r] + p["b_down"] for r in range(t)]
    sq = reduce_from_tp_region_forward([np.float64(np.sum((ys[r] - target[sl[r]]) ** 2)) for r in range(t)])
    loss = 0.5 * float(sq) / (N * H)
    dys = [(ys[r] - target[sl[r]]) / (N * H) for r in range(t)]
    dy_full = gather_from_sequence_parallel_region(dys)
    gl, dnl = [], []
    for r in range(t):
        g, dn = rank_backward_local(qs[r], caches[r], dy_full)
        g["b_down"] = np.sum(dys[r], axis=0)  # the bias is added on the rank's own slice
        gl.append(g)
        dnl.append(dn)
    dns = reduce_scatter_to_sequence_parallel_region(dnl)
    dxs, local_dnw = [], []
    for r in range(t):
        dxn, dnw = rms_norm_backward(dns[r], normed[r][2], normed[r][1], p["norm_w"])
        dxs.append(dys[r] + dxn)
        local_dnw.append(dnw)
    local_dbd = [gl[r]["b_down"] for r in range(t)]
    if skip_sp_grad_sync:
        dnws, dbds = local_dnw, local_dbd
    else:
        dnw = reduce_from_tp_region_forward(local_dnw)
        dbd = reduce_from_tp_region_forward(local_dbd)
        dnws, dbds = [dnw] * t, [dbd] * t
    ranks = []
    for r in range(t):
        gr = dict(gl[r])
        gr["norm_w"], gr["b_down"] = dnws[r], dbds[r]
        newq = {k: qs[r][k] - lr * gr[k] for k in qs[r]}
        ranks.append({"y": ys[r], "dy": dys[r], "dx": dxs[r], "grads": gr, "new_params": newq,
                      "local_norm_w_grad": local_dnw[r], "local_b_down_grad": local_dbd[r]})
    v = ranks[view_rank]
    grads = {"x": np.concatenate(dxs, axis=0), "norm_w": v["grads"]["norm_w"], "b_down": v["grads"]["b_down"],
             "w_down": np.concatenate([rk["grads"]["w_down"] for rk in ranks], axis=1)}
    newp = {"norm_w": v["new_params"]["norm_w"], "b_down": v["new_params"]["b_down"],
            "w_down": np.concatenate([rk["new_params"]["w_down"] for rk in ranks], axis=1)}
    if act == "swiglu":
        grads["w_gate_up"] = np.concatenate([rk["grads"]["w_gate_up"] for rk in ranks], axis=1)
        newp["w_gate_up"] = np.concatenate([rk["new_params"]["w_gate_up"] for rk in ranks], axis=1)
    else:
        for k in ("w_1", "b_1"):
            grads[k] = np.concatenate([rk["grads"][k] for rk in ranks], axis=0)
            newp[k] = np.concatenate([rk["new_params"][k] for rk in ranks], axis=0)
    return {"y": np.concatenate(ys, axis=0), "loss": loss, "dy": np.concatenate(dys, axis=0), "grads": grads,
            "new_params": newp, "ranks": ranks}


# ---------------------------------------------------------------------------
# FP8 GEMMs (the explainer's "FP8 Transformer Engine" GEMMs with per-tensor
# scaling): every GEMM operand is cast to E4M3 with a per-tensor scale taken
# from its absolute maximum, the products of the codes are summed exactly and
# the sum is divided by both scales.
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def _e4m3_positive_table() -> np.ndarray:
    """Values of the non-negative finite E4M3 codes 0x00..0x7e in code order
    (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 holds
    the subnormals m/8 * 2^-6; code 0x7f is NaN, so there is no infinity)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


E4M3_TABLE = _e4m3_positive_table()


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (uint8)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, E4M3_TABLE[np.minimum(mag, 0x7E)])
    return np.where(c & 0x80, -out, out)


def e4m3_encode(x) -> np.ndarray:
    """Round each value to the nearest E4M3 code, ties to the even code,
    saturating at +-448 (finite values never become NaN); NaN -> 0x7f.
    A negative value (or -0) keeps the sign bit, also when it rounds to 0."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    a_sat = np.minimum(np.where(np.isnan(a), 0.0, a), E4M3_MAX)
    hi = np.clip(np.searchsorted(E4M3_TABLE, a_sat, side="left"), 0, 0x7E)  # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a_sat - E4M3_TABLE[lo]
    d_hi = E4M3_TABLE[hi] - a_sat
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def fp8_scale(amax: float) -> np.float32:
    """Per-tensor scale that maps the absolute maximum onto the E4M3 maximum,
    448 / amax, computed in float32; 1 for an all-zero (or non-finite) amax."""
    amax = np.float32(amax)
    if not (amax > 0 and np.isfinite(amax)):
        return np.float32(1.0)
    return np.float32(E4M3_MAX) / amax


def quantize_e4m3(x):
    """Cast a tensor to E4M3 with its current per-tensor scale: the product
    x * scale is formed in float32 and rounded to a code.  Returns (codes,
    scale)."""
    x32 = np.asarray(x, dtype=np.float32)
    s = fp8_scale(float(np.max(np.abs(x32))) if x32.size else 0.0)
    return e4m3_encode((x32 * s).astype(np.float32)), s


def fp8_linear(a, b):
    """a [M, K] times b [N, K] transposed, both cast to E4M3 with their own
    per-tensor scales: (decode(qa) decode(qb)^T) / (s_a s_b), exact in
    float64 apart from the final division."""
    qa, sa = quantize_e4m3(a)
    qb, sb = quantize_e4m3(b)
    return (e4m3_decode(qa) @ e4m3_decode(qb).T) / (np.float64(sa) * np.float64(sb))


def dense_step_fp8(p: dict, x, target, eps: float, lr: float, act: str = "swiglu",
                   store=None) -> dict:
    """The dense step with every GEMM replaced by ``fp8_linear``.  ``store``
    (e.g. ``synth.round_to_bf16``) is applied to each activation where it is
    stored before it becomes a GEMM operand (the normed input, the
    activation, dy and the gate/up gradient), so that the per-tensor scale
    and the codes are taken from the stored values; None keeps float64."""
    st = store if store is not None else (lambda v: v)
    x = np.asarray(x, dtype=np.float64)
    N, H = x.shape
    n, rstd, xhat = rms_norm(x, p["norm_w"], eps)
    n_s = st(n)
    c = {"n": n_s, "rstd": rstd, "xhat": xhat}
    if act == "swiglu":
        F = p["w_gate_up"].shape[1]
        gu = fp8_linear(n_s, p["w_gate_up"].reshape(2 * F, H))
        gate, up = gu[:, :F], gu[:, F:]
        hidden = silu(gate) * up
        c.update(gate=gate, up=up)
    else:
        z = fp8_linear(n_s, p["w_1"]) + p["b_1"]
        hidden = gelu(z)
        c["z"] = z
    h_s = st(hidden)
    y = x + fp8_linear(h_s, p["w_down"]) + p["b_down"]
    loss, dy = mse_loss(y, target)
    dy_s = st(dy)
    g = {"b_down": np.sum(dy_s, axis=0)}
    dh = fp8_linear(dy_s, p["w_down"].T)
    g["w_down"] = fp8_linear(dy_s.T, h_s.T)
    if act == "swiglu":
        dgate = dh * up * silu_grad(gate)
        dup = dh * silu(gate)
        dgu = st(np.concatenate([dgate, dup], axis=1))
        g["w_gate_up"] = fp8_linear(dgu.T, n_s.T).reshape(2, F, H)
        dn = fp8_linear(dgu, p["w_gate_up"].reshape(2 * F, H).T)
    else:
        dz = st(dh * gelu_grad(c["z"]))
        g["w_1"] = fp8_linear(dz.T, n_s.T)
        g["b_1"] = np.sum(dz, axis=0)
        dn = fp8_linear(dz, p["w_1"].T)
    dxn, g["norm_w"] = rms_norm_backward(dn, xhat, rstd, p["norm_w"])
    g["x"] = dy + dxn
    g["_dn"] = dn
    return {"y": y, "loss": loss, "dy": dy, "grads": g, "new_params": sgd(p, {k: g[k] for k in p}, lr)}


# ---------------------------------------------------------------------------
# Tensor-parallel attention sublayer (the explainer, "Self-attention: split
# across heads"; the architecture page's W_QKV split column-wise and W_out
# row-wise with one all-reduce; the TP-MLP page's closing note: grouped-query
# attention with complete query/KV head groups kept together per rank).
# Pre-RMSNorm, QKV projection, causal softmax attention per query head (each
# query head reads the K/V of its group), output projection, bias, residual.
# ---------------------------------------------------------------------------


def attn_split_heads(p: dict, n_q: int, n_kv: int):
    """W_qkv [(n_q + 2 n_kv) d, H] -> (W_q [n_q d, H], W_k [n_kv d, H], W_v [n_kv d, H]), d."""
    rows = p["w_qkv"].shape[0]
    d = rows // (n_q + 2 * n_kv)
    if d * (n_q + 2 * n_kv) != rows or n_q % n_kv != 0:
        raise ShapeError("w_qkv rows must be (n_q + 2 n_kv) d with n_q a multiple of n_kv")
    wq = p["w_qkv"][: n_q * d]
    wk = p["w_qkv"][n_q * d: (n_q + n_kv) * d]
    wv = p["w_qkv"][(n_q + n_kv) * d:]
    return wq, wk, wv, d


def causal_softmax(s):
    """Row softmax of s [..., S, S] over keys j <= i (the causal mask)."""
    S = s.shape[-1]
    mask = np.triu(np.ones((S, S), dtype=bool), k=1)
    s = np.where(mask, -np.inf, s)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_heads(q, k, v, batch: int, n_q: int, n_kv: int, d: int):
    """Causal attention of every (sequence, query head): q [N, n_q d], k, v
    [N, n_kv d], tokens grouped as batch sequences of N / batch.  Returns
    z [N, n_q d] and the probabilities P [batch, n_q, S, S]."""
    N = q.shape[0]
    S = N // batch
    hpg = n_q // n_kv
    qh = q.reshape(batch, S, n_q, d).transpose(0, 2, 1, 3)
    kh = k.reshape(batch, S, n_kv, d).transpose(0, 2, 1, 3)
    vh = v.reshape(batch, S, n_kv, d).transpose(0, 2, 1, 3)
    kq = np.repeat(kh, hpg, axis=1)  # query head h reads group h // hpg
    vq = np.repeat(vh, hpg, axis=1)
    P = causal_softmax(qh @ kq.transpose(0, 1, 3, 2) / math.sqrt(d))
    z = (P @ vq).transpose(0, 2, 1, 3).reshape(N, n_q * d)
    return z, P


def attn_dense_forward(p: dict, x, eps: float, batch: int, n_q: int, n_kv: int):
    """y = x + Attention(RMSNorm(x) W_qkv^T) W_o^T + b_o; p holds norm_w,
    w_qkv, w_o [H, n_q d], b_o."""
    x = np.asarray(x, dtype=np.float64)
    wq, wk, wv, d = attn_split_heads(p, n_q, n_kv)
    n, rstd, xhat = rms_norm(x, p["norm_w"], eps)
    q, k, v = linear(n, wq), linear(n, wk), linear(n, wv)
    z, P = attention_heads(q, k, v, batch, n_q, n_kv, d)
    y = x + linear(z, p["w_o"]) + p["b_o"]
    return y, {"n": n, "rstd": rstd, "xhat": xhat, "q": q, "k": k, "v": v, "z": z, "P": P, "d": d,
               "batch": batch, "n_q": n_q, "n_kv": n_kv}


def attention_heads_backward(c: dict, dz):
    """Gradients of the attention outputs with respect to q, k and v:
    dP = dZ V^T, dS = P (dP - rowsum(dP P)) / sqrt(d), dQ = dS K, dK = dS^T Q,
    dV = P^T dZ, with the K/V gradients of a group summed over its heads."""
    batch, n_q, n_kv, d = c["batch"], c["n_q"], c["n_kv"], c["d"]
    N = dz.shape[0]
    S = N // batch
    hpg = n_q // n_kv
    P = c["P"]
    sh = lambda t, h: t.reshape(batch, S, h, d).transpose(0, 2, 1, 3)
    qh, kq, vq = sh(c["q"], n_q), np.repeat(sh(c["k"], n_kv), hpg, axis=1), np.repeat(sh(c["v"], n_kv), hpg, axis=1)
    dzh = sh(dz, n_q)
    dP = dzh @ vq.transpose(0, 1, 3, 2)
    dS = P * (dP - np.sum(dP * P, axis=-1, keepdims=True)) / math.sqrt(d)
    dq = dS @ kq
    dk = (dS.transpose(0, 1, 3, 2) @ qh).reshape(batch, n_kv, hpg, S, d).sum(axis=2)
    dv = (P.transpose(0, 1, 3, 2) @ dzh).reshape(batch, n_kv, hpg, S, d).sum(axis=2)
    un = lambda t, h: t.transpose(0, 2, 1, 3).reshape(N, h * d)
    return un(dq, n_q), un(dk, n_kv), un(dv, n_kv)


def attn_dense_backward(p: dict, c: dict, dy) -> dict:
    """Parameter and input gradients of the attention sublayer."""
    wq, wk, wv, d = attn_split_heads(p, c["n_q"], c["n_kv"])
    g = {"b_o": np.sum(dy, axis=0), "w_o": dy.T @ c["z"]}
    dz = dy @ p["w_o"]
    dq, dk, dv = attention_heads_backward(c, dz)
    dqkv = np.concatenate([dq, dk, dv], axis=1)
    g["w_qkv"] = dqkv.T @ c["n"]
    dn = dqkv @ p["w_qkv"]
    dxn, g["norm_w"] = rms_norm_backward(dn, c["xhat"], c["rstd"], p["norm_w"])
    g["x"] = dy + dxn
    g["_dn"] = dn
    return g


def attn_dense_step(p: dict, x, target, eps: float, lr: float, batch: int, n_q: int, n_kv: int) -> dict:
    """Forward, MSE loss, backward and SGD of the attention sublayer."""
    y, c = attn_dense_forward(p, x, eps, batch, n_q, n_kv)
    loss, dy = mse_loss(y, target)
    g = attn_dense_backward(p, c, dy)
    return {"y": y, "loss": loss, "dy": dy, "grads": g, "new_params": sgd(p, {k: g[k] for k in p}, lr),
            "cache": c}


def attn_local_params(p: dict, t: int, rank: int, n_q: int, n_kv: int) -> dict:
    """Rank r's slices: KV groups [r n_kv/t, (r+1) n_kv/t) with their query
    heads (complete groups per rank), the matching rows of W_q, W_k, W_v and
    columns of W_o; norm_w and b_o replicated."""
    if n_kv % t != 0:
        raise ShapeError(f"n_kv={n_kv} is not divisible by t={t}")
    wq, wk, wv, d = attn_split_heads(p, n_q, n_kv)
    gq, gk = n_q // t, n_kv // t
    sq = slice(rank * gq * d, (rank + 1) * gq * d)
    sk = slice(rank * gk * d, (rank + 1) * gk * d)
    return {"norm_w": p["norm_w"], "w_qkv": np.concatenate([wq[sq], wk[sk], wv[sk]], axis=0),
            "w_o": p["w_o"][:, sq], "b_o": p["b_o"]}


def attn_sharded_step(p: dict, x, target, eps: float, lr: float, t: int, batch: int, n_q: int, n_kv: int) -> dict:
    """One step of the t-rank decomposition: each rank runs its head groups'
    attention on the replicated normed input and produces a partial output
    z_r W_o,r^T; the partials are summed (the all-reduce closing attention),
    then bias and residual.  In the backward each rank's normed-input
    gradient is partial and is summed the same way (the f all-reduce)."""
    x = np.asarray(x, dtype=np.float64)
    qs = [attn_local_params(p, t, r, n_q, n_kv) for r in range(t)]
    parts, caches = [], []
    for r in range(t):
        n, rstd, xhat = rms_norm(x, p["norm_w"], eps)
        wq, wk, wv, d = attn_split_heads(qs[r], n_q // t, n_kv // t)
        q, k, v = linear(n, wq), linear(n, wk), linear(n, wv)
        z, P = attention_heads(q, k, v, batch, n_q // t, n_kv // t, d)
        parts.append(linear(z, qs[r]["w_o"]))
        caches.append({"n": n, "rstd": rstd, "xhat": xhat, "q": q, "k": k, "v": v, "z": z, "P": P, "d": d,
                       "batch": batch, "n_q": n_q // t, "n_kv": n_kv // t})
    y = x + reduce_from_tp_region_forward(parts) + p["b_o"]
    loss, dy = mse_loss(y, target)
    gl, dnl = [], []
    for r in range(t):
        c = caches[r]
        g = {"w_o": dy.T @ c["z"], "b_o": np.sum(dy, axis=0)}
        dq, dk, dv = attention_heads_backward(c, dy @ qs[r]["w_o"])
        dqkv = np.concatenate([dq, dk, dv], axis=1)
        g["w_qkv"] = dqkv.T @ c["n"]
        gl.append(g)
        dnl.append(dqkv @ qs[r]["w_qkv"])
    dn = copy_to_tp_region_backward(dnl)
    c0 = caches[0]
    dxn, dnw = rms_norm_backward(dn, c0["xhat"], c0["rstd"], p["norm_w"])
    # reassemble the sharded gradients in the dense layout
    d = c0["d"]
    gq = [g["w_qkv"][: (n_q // t) * d] for g in gl]
    gk = [g["w_qkv"][(n_q // t) * d: (n_q // t + n_kv // t) * d] for g in gl]
    gv = [g["w_qkv"][(n_q // t + n_kv // t) * d:] for g in gl]
    grads = {"x": dy + dxn, "norm_w": dnw, "b_o": gl[0]["b_o"], "_dn": dn,
             "w_qkv": np.concatenate(gq + gk + gv, axis=0),
             "w_o": np.concatenate([g["w_o"] for g in gl], axis=1)}
    return {"y": y, "loss": loss, "dy": dy, "grads": grads,
            "new_params": sgd(p, {k: grads[k] for k in p}, lr)}
