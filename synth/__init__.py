"""Seeded synthetic inputs for the tensor-parallel MLP sublayer.

This module is shared by the CPU oracle, the GPU tests and the benchmark.  It
holds no arithmetic of the method itself: only counter-based random numbers,
the workload shapes, and the rounding of generated values to the storage
dtype.  Both sides of a parity check receive the *same* values from here.

Generator (stated so it can be re-implemented anywhere):

* ``splitmix64`` finaliser (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014), used as a counter-based
  hash: ``u64(i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)``.
* ``key = mix(seed * 0xD1B54A32D192ED03 + stream)`` with one ``stream`` id per
  tensor, so tensors are independent and can be generated in any order.
* Uniforms ``u = ((u64 >> 11) + 0.5) * 2**-53`` lie in (0, 1).
* Normals by the Box-Muller transform, element ``i`` using counters ``2i`` and
  ``2i+1``: ``sqrt(-2 ln u0) * cos(2 pi u1)``.

Workloads are the five sublayer configurations the study measures (fp32
parity case, three bf16 SwiGLU shapes and one bf16 GeLU shape); their sizes
and initialisation recipes are listed in ``CONFIGS``.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_SEEDMUL = 0xD1B54A32D192ED03
_MASK64 = (1 << 64) - 1

# Stream ids, one per tensor.
STREAM = {
    "x": 1, "target": 2, "norm_w": 3, "w_gate_up": 4, "w_down": 5,
    "b_down": 6, "b_1": 7, "dy": 8, "grad": 9, "extra": 10,
}


def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return _mix_int(seed * _SEEDMUL + stream)


def _u64_block(key: int, c0: int, n: int) -> np.ndarray:
    ctr = np.arange(c0 + 1, c0 + 1 + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + ctr * _GOLDEN
        return _mix_np(z)


def _normal_block(key: int, start: int, n: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        u = _u64_block(key, 2 * start, 2 * n).reshape(n, 2)
    f = ((u >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(f[:, 0])) * np.cos(2.0 * np.pi * f[:, 1])


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    return _POOL


def normal(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """Seeded N(mean, std^2) samples as float64, element i independent of shape."""
    n = int(np.prod(shape)) if len(shape) else 1
    key = stream_key(seed, stream)
    out = np.empty(n, dtype=np.float64)
    chunk = 1 << 22
    if n <= chunk:
        out[:] = _normal_block(key, 0, n)
    else:
        def work(s):
            e = min(n, s + chunk)
            out[s:e] = _normal_block(key, s, e - s)
        list(_pool().map(work, range(0, n, chunk)))
    out *= std
    out += mean
    return out.reshape(shape)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (round-to-nearest-even) and return them
    as float64 (exactly representable), so both sides see identical values."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The uint16 bit patterns of values already rounded by ``round_to_bf16``."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@dataclasses.dataclass(frozen=True)
class Config:
    """One workload of the sublayer: sizes, dtype, activation and init recipe."""
    name: str
    dtype: str          # "f32" or "bf16" (bf16 storage, fp32 accumulation)
    act: str            # "swiglu" or "gelu"
    tokens: int         # N = batch * seq
    batch: int
    seq: int
    hidden: int         # H
    ffn: int            # F
    t_list: tuple       # logical tensor-parallel degrees exercised
    w_std: float
    norm_w: str         # "ones" or "one_plus_0.1"
    b_down_std: float   # 0 => zeros
    b_1_std: float      # GeLU first-projection bias; 0 for SwiGLU
    lr: float
    eps: float = 1e-6

    def with_tokens(self, n: int) -> "Config":
        return dataclasses.replace(self, tokens=n, batch=1, seq=n)

    def with_shape(self, tokens: int, hidden: int, ffn: int) -> "Config":
        return dataclasses.replace(self, tokens=tokens, batch=1, seq=tokens,
                                   hidden=hidden, ffn=ffn)

    @property
    def gemm_flops(self) -> float:
        """Algorithmic GEMM flops of one fwd+bwd step (18NHF SwiGLU, 12NHF GeLU)."""
        k = 18 if self.act == "swiglu" else 12
        return float(k) * self.tokens * self.hidden * self.ffn


CONFIGS = {
    "fp32_small": Config("fp32_small", "f32", "swiglu", 16, 2, 8, 64, 256, (2, 1, 4, 8),
                         0.02, "ones", 0.0, 0.0, 0.1),
    "bf16_h2048": Config("bf16_h2048", "bf16", "swiglu", 4096, 2, 2048, 2048, 5632, (1, 2, 4),
                         0.02, "one_plus_0.1", 0.01, 0.0, 1e-3),
    "bf16_gelu_h4096": Config("bf16_gelu_h4096", "bf16", "gelu", 8192, 4, 2048, 4096, 16384, (8,),
                              0.02, "ones", 0.01, 0.01, 1e-3),
    "bf16_llama8b": Config("bf16_llama8b", "bf16", "swiglu", 16384, 4, 4096, 4096, 14336, (8, 4),
                           0.02, "ones", 0.0, 0.0, 1e-3),
    "bf16_70b_n2048": Config("bf16_70b_n2048", "bf16", "swiglu", 2048, 1, 2048, 8192, 28672, (8,),
                             0.015, "ones", 0.0, 0.0, 1e-3),
}

# Token counts swept for the 70B-shaped block.
SWEEP_70B_TOKENS = (512, 2048, 8192, 32768)


def make_inputs(cfg: Config, seed: int = 1234) -> dict:
    """All inputs of one training step as float64 arrays holding values that
    are exactly representable in ``cfg.dtype``.

    Keys: x [N,H], target [N,H], norm_w [H], w_gate_up [2,F,H] (SwiGLU) or
    w_1 [F,H] (GeLU), b_1 [F] (GeLU only), w_down [H,F], b_down [H].
    """
    N, H, F = cfg.tokens, cfg.hidden, cfg.ffn
    rnd = round_to_bf16 if cfg.dtype == "bf16" else (lambda a: a.astype(np.float32).astype(np.float64))
    d = {}
    d["x"] = rnd(normal(seed, STREAM["x"], (N, H)))
    d["target"] = rnd(normal(seed, STREAM["target"], (N, H)))
    if cfg.norm_w == "ones":
        d["norm_w"] = np.ones(H)
    else:
        d["norm_w"] = rnd(normal(seed, STREAM["norm_w"], (H,), 1.0, 0.1))
    if cfg.act == "swiglu":
        d["w_gate_up"] = rnd(normal(seed, STREAM["w_gate_up"], (2, F, H), 0.0, cfg.w_std))
    else:
        d["w_1"] = rnd(normal(seed, STREAM["w_gate_up"], (F, H), 0.0, cfg.w_std))
        d["b_1"] = rnd(normal(seed, STREAM["b_1"], (F,), 0.0, cfg.b_1_std)) if cfg.b_1_std > 0 else np.zeros(F)
    d["w_down"] = rnd(normal(seed, STREAM["w_down"], (H, F), 0.0, cfg.w_std))
    d["b_down"] = rnd(normal(seed, STREAM["b_down"], (H,), 0.0, cfg.b_down_std)) if cfg.b_down_std > 0 else np.zeros(H)
    return d


def make_optimizer_state(cfg: Config, seed: int = 1234, grad_std: float = 1e-4, m_std: float = 5e-5,
                         v_std: float = 1e-4) -> dict:
    """Seeded stand-ins for one optimizer step's inputs, per parameter, as
    float64 arrays of fp32-representable values: a gradient g ~ N(0, grad_std),
    a first moment m ~ N(0, m_std) and a second moment v = |N(0, v_std)|^2
    (non-negative).  Streams 100 + 3k, 101 + 3k, 102 + 3k for the k-th
    parameter of ``param_names``."""
    shapes = {"norm_w": (cfg.hidden,), "w_gate_up": (2, cfg.ffn, cfg.hidden), "w_1": (cfg.ffn, cfg.hidden),
              "b_1": (cfg.ffn,), "w_down": (cfg.hidden, cfg.ffn), "b_down": (cfg.hidden,)}
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    out = {"grad": {}, "m": {}, "v": {}}
    for k, name in enumerate(param_names(cfg.act)):
        shp = shapes[name]
        out["grad"][name] = f32(normal(seed, 100 + 3 * k, shp, 0.0, grad_std))
        out["m"][name] = f32(normal(seed, 101 + 3 * k, shp, 0.0, m_std))
        out["v"][name] = f32(np.square(normal(seed, 102 + 3 * k, shp, 0.0, v_std)))
    return out


def param_names(act: str) -> tuple:
    return ("norm_w", "w_gate_up", "w_down", "b_down") if act == "swiglu" else \
           ("norm_w", "w_1", "b_1", "w_down", "b_down")


@dataclasses.dataclass(frozen=True)
class AttnConfig:
    """One workload of the attention sublayer: batch sequences of seq tokens,
    hidden H, n_q query heads in n_kv groups of head dimension d."""
    name: str
    batch: int
    seq: int
    hidden: int
    n_q: int
    n_kv: int
    d: int
    t_list: tuple
    w_std: float = 0.02
    lr: float = 1e-3
    eps: float = 1e-6

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def gemm_flops(self) -> float:
        """Algorithmic flops of one fwd+bwd step: the projections, 2 N H (W + n_q d) forward and twice
        that backward, and the attention contractions Q K^T and P V forward (2 S^2 d each per sequence
        and query head) and their four backward products, each counted for the causal half of the
        score square (S (S + 1) / 2 entries)."""
        N, H, d = self.tokens, self.hidden, self.d
        W = (self.n_q + 2 * self.n_kv) * d
        proj = 2.0 * N * H * (W + self.n_q * d)
        att = 2.0 * 2.0 * self.batch * self.n_q * (self.seq * (self.seq + 1) / 2.0) * d
        return 3.0 * (proj + att)


ATTN_CONFIGS = {
    "attn_small": AttnConfig("attn_small", 2, 128, 256, 4, 2, 64, (1, 2)),
    "attn_gpt_h4096": AttnConfig("attn_gpt_h4096", 4, 2048, 4096, 32, 8, 128, (8, 4)),
    # the same sublayer on one long sequence (fused attention only)
    "attn_gpt_h4096_s8k": AttnConfig("attn_gpt_h4096_s8k", 1, 8192, 4096, 32, 8, 128, (8, 4)),
    "attn_gpt_h4096_s32k": AttnConfig("attn_gpt_h4096_s32k", 1, 32768, 4096, 32, 8, 128, (8, 4)),
}


def make_attn_inputs(cfg: AttnConfig, seed: int = 1234) -> dict:
    """All inputs of one attention step as float64 arrays of bf16-representable
    values: x, target [N, H] ~ N(0, 1); norm_w ~ 1 + N(0, 0.1); w_qkv
    [(n_q + 2 n_kv) d, H] and w_o [H, n_q d] ~ N(0, w_std); b_o ~ N(0, 0.01).
    Streams 40..45."""
    N, H, d = cfg.tokens, cfg.hidden, cfg.d
    W = (cfg.n_q + 2 * cfg.n_kv) * d
    r = round_to_bf16
    return {"x": r(normal(seed, 40, (N, H))), "target": r(normal(seed, 41, (N, H))),
            "norm_w": r(normal(seed, 42, (H,), 1.0, 0.1)), "w_qkv": r(normal(seed, 43, (W, H), 0.0, cfg.w_std)),
            "w_o": r(normal(seed, 44, (H, cfg.n_q * d), 0.0, cfg.w_std)),
            "b_o": r(normal(seed, 45, (H,), 0.0, 0.01))}


def make_attn_optimizer_state(cfg: AttnConfig, seed: int = 1234, grad_std: float = 1e-4, m_std: float = 5e-5,
                              v_std: float = 1e-4) -> dict:
    """Seeded optimizer-step inputs for the attention parameters, drawn as in
    ``make_optimizer_state``: g ~ N(0, grad_std), m ~ N(0, m_std), v =
    |N(0, v_std)|^2, fp32-representable float64.  Streams 150 + 3k, 151 + 3k,
    152 + 3k for the k-th of norm_w, w_qkv, w_o, b_o."""
    H, d = cfg.hidden, cfg.d
    shapes = {"norm_w": (H,), "w_qkv": ((cfg.n_q + 2 * cfg.n_kv) * d, H), "w_o": (H, cfg.n_q * d), "b_o": (H,)}
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    out = {"grad": {}, "m": {}, "v": {}}
    for k, name in enumerate(("norm_w", "w_qkv", "w_o", "b_o")):
        shp = shapes[name]
        out["grad"][name] = f32(normal(seed, 150 + 3 * k, shp, 0.0, grad_std))
        out["m"][name] = f32(normal(seed, 151 + 3 * k, shp, 0.0, m_std))
        out["v"][name] = f32(np.square(normal(seed, 152 + 3 * k, shp, 0.0, v_std)))
    return out
