"""Shared helpers for the GPU tests: move seeded inputs to the device, run one
step through the C ABI, and compare with the oracle under the stated
tolerances.

Tolerances (written here, used by every parity test):

* fp32 configuration: per element |gpu - oracle| <= 1e-5 * |oracle| +
  1e-5 * max|oracle|, and ||gpu - oracle||_2 <= 1e-5 * ||oracle||_2.
* bf16 configuration (fp32 accumulation): per element |gpu - oracle| <=
  2e-2 * |oracle| + 1e-2 * max|oracle|, and ||gpu - oracle||_2 <= 2e-2 *
  ||oracle||_2 per tensor.

* FP8 GEMM operands, against the oracle's FP8 step (``tol="fp8"``): per
  element |gpu - oracle| <= 0.1 * |oracle| + 0.05 * max|oracle|, normwise
  0.05.  Both sides quantise with the same rule, but from stored operands
  that differ by bf16 rounding (and whose maxima, hence scales, may differ
  by one bf16 unit, 2^-8): a fraction of about 2^-8 / 2^-3 = 3% of the codes
  then round the other way, each by one E4M3 unit (up to 2^-3 relative).
  Through a sum of K such products with mixed signs that is a normwise
  error of about sqrt(0.03) * 2^-3 / sqrt(3) ~ 1.2% per GEMM, compounded
  over the chained GEMMs of the backward; small elements of a cancelling
  sum see several times that, hence the per-element bound.

The absolute term is the stated absolute tolerance applied to the tensor
divided by its largest magnitude: gradients of a mean loss are ~1e-8..1e-4,
where a fixed absolute 1e-2 would accept anything.  Scaling by the rms instead
is too tight for bf16 storage: its rounding noise is ~0.4% of the rms and a
million-element tensor has ~5-sigma elements (checked with a bf16-storage
simulation of the step).  The normwise check carries most of the weight.
"""
from __future__ import annotations

import numpy as np
import torch

import synth

TOL = {
    "f32": dict(rtol=1e-5, atol_max=1e-5, norm=1e-5),
    "bf16": dict(rtol=2e-2, atol_max=1e-2, norm=2e-2),
    "fp8": dict(rtol=1e-1, atol_max=5e-2, norm=5e-2),
}


def to_dev(a, dtype: str, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.to(device)


def fma_f32(a, b, c):
    """a * b + c over float32 arrays with one rounding to float32 (nearest even), as fmaf does.

    The product of two float32 values is exact in float64; the sum is formed in
    float64 with its exact error (two-sum), and where the float64 sum lies on a
    float32 midpoint the error decides the side, so the result never suffers
    double rounding.  Finite inputs whose result stays finite and normal."""
    a, b, c = (np.asarray(v, dtype=np.float32) for v in (a, b, c))
    p = a.astype(np.float64) * b.astype(np.float64)
    q = c.astype(np.float64)
    s = p + q
    bv = s - p
    err = (p - (s - bv)) + (q - bv)
    r = s.astype(np.float32)
    r64 = r.astype(np.float64)
    up = np.nextafter(r, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(r, np.float32(-np.inf)).astype(np.float64)
    r = np.where((s == (r64 + up) / 2) & (err > 0), up.astype(np.float32), r)
    r = np.where((s == (r64 + dn) / 2) & (err < 0), dn.astype(np.float32), r)
    return r


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(name: str, gpu, ora, dtype: str, report: dict | None = None, extra=None):
    """Element-wise and normwise check; ``extra`` is an optional per-element
    allowance added to the bound (storage rounding of a quantity that is a
    difference of two stored values)."""
    g = np.asarray(gpu, dtype=np.float64)
    o = np.asarray(ora, dtype=np.float64)
    assert g.shape == o.shape, (name, g.shape, o.shape)
    tol = TOL[dtype]
    amax = float(np.max(np.abs(o))) if o.size else 0.0
    atol = tol["atol_max"] * max(amax, 1e-30)
    err = np.abs(g - o)
    ex = np.zeros_like(o) if extra is None else np.asarray(extra, dtype=np.float64)
    bound = tol["rtol"] * np.abs(o) + atol + ex
    bad = err > bound
    nrm = float(max(0.0, np.linalg.norm(g - o) - np.linalg.norm(ex)) / max(np.linalg.norm(o), 1e-300)) \
        if o.size else 0.0
    if report is not None:
        report[name] = {"max_abs": float(err.max()) if err.size else 0.0, "rel_norm": nrm, "n_bad": int(bad.sum())}
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu={g[i]!r} oracle={o[i]!r} bound={bound[i]!r}; rel_norm={nrm:.3e}")
    assert nrm <= tol["norm"], f"{name}: normwise relative error {nrm:.3e} > {tol['norm']}"


def device_inputs(cfg: synth.Config, inp: dict):
    d = {k: to_dev(v, cfg.dtype) for k, v in inp.items()}
    return d


def gpu_step(cfg: synth.Config, inp: dict, t: int, lr: float, flags: int = 0, shard: int = 0,
             masters: bool = True, mod=None, with_params: bool = True, update_in_backward: bool = False):
    """Forward, loss, backward and SGD through the binding; numpy results
    (the updated parameters only when ``with_params``).  With
    ``update_in_backward`` the backward applies the SGD update itself."""
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    m = mod or TPMLP(max(cfg.tokens, 1), cfg.hidden, cfg.ffn, max_t=max(8, t), dtype=cfg.dtype, act=cfg.act)
    d = device_inputs(cfg, inp)
    gu_key = "w_gate_up" if cfg.act == "swiglu" else "w_1"
    params = {k: d[k] for k in synth.param_names(cfg.act)}
    ms = None
    if cfg.dtype == "bf16" and masters:
        ms = {("w_gate_up" if k == "w_1" else k): torch.from_numpy(np.asarray(inp[k], dtype=np.float32)).cuda()
              for k in synth.param_names(cfg.act)}
        m.bind_master(ms)
    m.set_debug(flags, shard)
    if update_in_backward:
        m.set_update_in_backward(True, lr)
    y = m.forward(d["x"], d["norm_w"], d[gu_key], d["w_down"], d["b_down"], cfg.eps, t,
                  b_1=d.get("b_1"))
    loss, dy = m.mse_loss_grad(y, d["target"])
    dx, g = m.backward(dy)
    grads = {k: to_np(v) for k, v in g.items()}
    out = {"y": to_np(y), "loss": float(loss.item()), "dy": to_np(dy), "dx": to_np(dx), "grads": grads}
    if update_in_backward:
        m.set_update_in_backward(False)
    else:
        m.sgd_step(lr)
    m.sync()
    if with_params:
        if ms is not None:
            out["new_master"] = {k: to_np(v) for k, v in ms.items()}
        out["new_params"] = {k: to_np(params[k]) for k in params}
    if cfg.act == "gelu":
        out["grads"]["w_1"] = out["grads"].pop("w_gate_up")
        if ms is not None and with_params:
            out["new_master"]["w_1"] = out["new_master"].pop("w_gate_up")
    m.set_debug(0, 0)
    return out


def compare_step(cfg: synth.Config, gpu: dict, ora: dict, inp: dict, lr: float, report: dict | None = None,
                 grad_keys=None, tol: str | None = None):
    dt = tol or cfg.dtype
    compare("y", gpu["y"], ora["y"], dt, report)
    assert abs(gpu["loss"] - ora["loss"]) <= TOL[dt]["rtol"] * abs(ora["loss"]) + 1e-12, (gpu["loss"], ora["loss"])
    compare("dx", gpu["dx"], ora["grads"]["x"], dt, report)
    for k in grad_keys or synth.param_names(cfg.act):
        compare("d" + k, gpu["grads"][k], ora["grads"][k], dt, report)
    # SGD ("post-step weights"): the stored float weights (masters for bf16)
    # equal the oracle's w - lr * g, and the applied update w' - w equals
    # -lr * g up to half an fp32 ulp of the stored w'.
    for k in synth.param_names(cfg.act):
        new = gpu["new_master"][k] if "new_master" in gpu else gpu["new_params"][k]
        w0 = np.asarray(inp[k], dtype=np.float32).astype(np.float64)
        compare("post_step_" + k, new, w0 - lr * ora["grads"][k], dt, report,
                extra=0.5 * np.spacing(np.abs(new).astype(np.float32)).astype(np.float64))
        compare("update_" + k, new - w0, -lr * ora["grads"][k], dt, report,
                extra=0.5 * np.spacing(np.abs(new).astype(np.float32)).astype(np.float64))
