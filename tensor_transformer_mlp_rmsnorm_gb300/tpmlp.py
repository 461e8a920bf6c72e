"""ctypes binding of the tpmlp C ABI (``include/tpmlp.h``).

Argument marshalling only: every step of the sublayer runs in the CUDA
library.  torch supplies device memory and the stream; nothing here computes.
The module raises ``TPMLPError`` if the shared library has not been built --
there is no fallback.

Functions named like the C entry points take torch tensors; ``TPMLP`` wraps a
context together with its workspace.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtpmlp.so")

OK, ERR_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_ORDER, ERR_CUDA, ERR_TIMEOUT = range(7)
F32, BF16 = 0, 1
SWIGLU, GELU = 0, 1
DBG_SKIP_FWD_REDUCE, DBG_SKIP_BWD_REDUCE, DBG_FORCE_TIMEOUT, DBG_GEMM_SINGLE_CTA = 1, 2, 4, 8
DBG_SKIP_SP_GRAD_SYNC = 16
PREC_BF16, PREC_FP8 = 0, 1

_DTYPES = {"f32": F32, "bf16": BF16}
_ACTS = {"swiglu": SWIGLU, "gelu": GELU}
_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


class TPMLPError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"tpmlp status {status}: {msg}")
        self.status = status


class AttnConfig(ctypes.Structure):
    """tpattn_config."""
    _fields_ = [("max_tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("max_seq", ctypes.c_int32),
                ("max_t", ctypes.c_int32), ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


class ParamSet(ctypes.Structure):
    """tpmlp_param_set: one device float* per parameter (b_1 for GeLU only)."""
    _fields_ = [("norm_w", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("b_1", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("b_down", ctypes.c_void_p)]


class AttnParamSet(ctypes.Structure):
    """tpattn_param_set: one device float* per attention parameter."""
    _fields_ = [("norm_w", ctypes.c_void_p), ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("b_o", ctypes.c_void_p)]


class AdamWParams(ctypes.Structure):
    """tpmlp_adamw_params."""
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("max_grad_norm", ctypes.c_float),
                ("step", ctypes.c_int64)]


class Config(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("max_t", ctypes.c_int32), ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_vp, _i32, _i64, _u32, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
_fp = ctypes.c_void_p  # float* (device)
_SIGNATURES = {
    "tpmlp_create": (_i32, [ctypes.POINTER(Config), _vp, ctypes.POINTER(_vp)]),
    "tpmlp_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config)]),
    "tpmlp_bind_workspace": (_i32, [_vp, _vp, ctypes.c_size_t]),
    "tpmlp_set_stream": (_i32, [_vp, _vp]),
    "tpmlp_forward": (_i32, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _i32, _vp]),
    "tpmlp_mse_loss_grad": (_i32, [_vp, _vp, _vp, _vp, _fp]),
    "tpmlp_backward": (_i32, [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp]),
    "tpmlp_bind_master": (_i32, [_vp, _fp, _fp, _fp, _fp, _fp]),
    "tpmlp_sgd_step": (_i32, [_vp, _f32]),
    "tpmlp_bind_adam_state": (_i32, [_vp, ctypes.POINTER(ParamSet), ctypes.POINTER(ParamSet)]),
    "tpmlp_adamw_step": (_i32, [_vp, ctypes.POINTER(AdamWParams), _fp]),
    "tpmlp_set_debug": (_i32, [_vp, _u32, _i32]),
    "tpmlp_set_sequence_parallel": (_i32, [_vp, _i32]),
    "tpmlp_set_update_in_backward": (_i32, [_vp, _i32, _f32]),
    "tpmlp_update_in_epilogue": (_i32, [_vp]),
    "tpmlp_fp8_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config)]),
    "tpmlp_bind_fp8_workspace": (_i32, [_vp, _vp, ctypes.c_size_t]),
    "tpmlp_set_precision": (_i32, [_vp, _i32]),
    "tpmlp_sync": (_i32, [_vp]),
    "tpmlp_set_timing": (_i32, [_vp, _i32]),
    "tpmlp_read_kernel_times": (_i32, [_vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int64), _i32]),
    "tpmlp_kernel_name": (ctypes.c_char_p, [_i32]),
    "tpmlp_num_kernel_ids": (_i32, []),
    "tpmlp_launch_count": (ctypes.c_uint64, [_vp]),
    "tpmlp_status_string": (ctypes.c_char_p, [_i32]),
    "tpmlp_last_error": (ctypes.c_char_p, [_vp]),
    "tpmlp_destroy": (None, [_vp]),
    "tpmlp_mse_loss_grad_noalloc": (_i32, [_i32, _i64, _vp, _vp, _vp, _fp, _vp]),
    "tpattn_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(AttnConfig)]),
    "tpattn_create": (_i32, [ctypes.POINTER(AttnConfig), _vp, ctypes.POINTER(_vp)]),
    "tpattn_bind_workspace": (_i32, [_vp, _vp, ctypes.c_size_t]),
    "tpattn_forward": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _f32, _i32, _vp]),
    "tpattn_backward": (_i32, [_vp, _vp, _vp, _fp, _fp, _fp, _fp]),
    "tpattn_bind_master": (_i32, [_vp, _fp, _fp, _fp, _fp]),
    "tpattn_sgd_step": (_i32, [_vp, _f32]),
    "tpattn_set_update_in_backward": (_i32, [_vp, _i32, _f32]),
    "tpattn_update_in_epilogue": (_i32, [_vp]),
    "tpattn_bind_adam_state": (_i32, [_vp, ctypes.POINTER(AttnParamSet), ctypes.POINTER(AttnParamSet)]),
    "tpattn_adamw_step": (_i32, [_vp, ctypes.POINTER(AdamWParams), _fp]),
    "tpattn_set_fused": (_i32, [_vp, _i32]),
    "tpattn_fused_active": (_i32, [_vp]),
    "tpattn_sync": (_i32, [_vp]),
    "tpattn_set_timing": (_i32, [_vp, _i32]),
    "tpattn_read_kernel_times": (_i32, [_vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int64), _i32]),
    "tpattn_kernel_name": (ctypes.c_char_p, [_i32]),
    "tpattn_num_kernel_ids": (_i32, []),
    "tpattn_launch_count": (ctypes.c_uint64, [_vp]),
    "tpattn_last_error": (ctypes.c_char_p, [_vp]),
    "tpattn_destroy": (None, [_vp]),
    "tpmlp_fp8_quantize": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _fp, _vp, _vp]),
    "tpmlp_fp8_gemm": (_i32, [_vp, _i64, _vp, _i64, _i64, _i64, _i64, _fp, _fp, _fp, _i64, _vp, _vp]),
}
TPATTN_FUSED_ONLY = 1  # tpattn_config.flags: only the fused attention kernels, no score square
FP8_SCRATCH_BYTES = 4096
NOALLOC_LOSS_MAX_BLOCKS = 1024

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise TPMLPError(ERR_UNSUPPORTED, f"{LIB_PATH} is missing: build it with "
                             "tensor_transformer_mlp_rmsnorm_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int, ctx=None):
    if status != OK:
        msg = lib().tpmlp_last_error(ctx).decode(errors="replace")
        raise TPMLPError(status, msg or lib().tpmlp_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def kernel_names() -> list:
    L = lib()
    return [L.tpmlp_kernel_name(i).decode() for i in range(L.tpmlp_num_kernel_ids())]


def make_config(max_tokens: int, hidden: int, ffn: int, max_t: int = 8, dtype: str = "bf16",
                act: str = "swiglu") -> Config:
    return Config(max_tokens, hidden, ffn, max_t, _DTYPES[dtype], _ACTS[act], 0)


def tpmlp_workspace_bytes(cfg: Config) -> int:
    return int(lib().tpmlp_workspace_bytes(ctypes.byref(cfg)))


def tpmlp_create(cfg: Config, stream=None):
    out = ctypes.c_void_p()
    s = None if stream is None else ctypes.c_void_p(stream)
    _check(lib().tpmlp_create(ctypes.byref(cfg), s, ctypes.byref(out)))
    return out


def tpmlp_mse_loss_grad_noalloc(y, target, dy, loss, stream=None):
    """Loss and gradient without a context or workspace (no device allocation
    by the library); y, target, dy: same dtype and size, loss: one float."""
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(y.dtype)
    if dt is None or target.dtype != y.dtype or dy.dtype != y.dtype or loss.dtype != torch.float32:
        raise TPMLPError(ERR_ARG, "y/target/dy must share dtype float32 or bfloat16; loss must be float32")
    if target.numel() != y.numel() or dy.numel() != y.numel() or loss.numel() < 1:
        raise TPMLPError(ERR_ARG, "y, target and dy must have the same number of elements")
    for t in (y, target, dy, loss):
        if not t.is_cuda or not t.is_contiguous():
            raise TPMLPError(ERR_ARG, "tensors must be contiguous CUDA tensors")
    s = stream if stream is not None else torch.cuda.current_stream(y.device).cuda_stream
    with torch.cuda.device(y.device):
        _check(lib().tpmlp_mse_loss_grad_noalloc(dt, y.numel(), _ptr(y), _ptr(target), _ptr(dy), _ptr(loss),
                                                 ctypes.c_void_p(s)))
    return loss, dy


def _pitch16(n: int) -> int:
    return (n + 15) // 16 * 16


def fp8_quantize(src, rows_major: bool = True, transposed: bool = True, stream=None):
    """E4M3 codes of a bf16 tensor [rows, cols] with its per-tensor scale
    (tpmlp_fp8_quantize).  Returns (codes [rows, pitch] or None,
    codes_t [cols, pitch] or None, inv_scale [1] float): the pitches are
    rounded up to 16 bytes; columns past cols (rows past rows) are padding."""
    if src.dtype != torch.bfloat16 or src.dim() != 2 or not src.is_contiguous():
        raise TPMLPError(ERR_ARG, "src must be a contiguous 2-D bf16 tensor")
    rows, cols = src.shape
    dev = src.device
    dst = torch.empty(rows, _pitch16(cols), dtype=torch.uint8, device=dev) if rows_major else None
    dst_t = torch.empty(cols, _pitch16(rows), dtype=torch.uint8, device=dev) if transposed else None
    inv = torch.empty(1, dtype=torch.float32, device=dev)
    scratch = torch.empty(FP8_SCRATCH_BYTES, dtype=torch.uint8, device=dev)
    st = (stream or torch.cuda.current_stream(dev)).cuda_stream
    _check(lib().tpmlp_fp8_quantize(_ptr(src), rows, cols, _ptr(dst) if dst is not None else None,
                                    dst.shape[1] if dst is not None else 0,
                                    _ptr(dst_t) if dst_t is not None else None,
                                    dst_t.shape[1] if dst_t is not None else 0, _ptr(inv), _ptr(scratch), st))
    return dst, dst_t, inv


def fp8_gemm(a, b, k: int, inv_a, inv_b, n: int | None = None, stream=None):
    """c = (a b^T) * inv_a * inv_b from E4M3 codes a [M, pitch], b [N, pitch]
    whose first k bytes per row are the operand (tpmlp_fp8_gemm)."""
    M = a.shape[0]
    N = b.shape[0] if n is None else n
    c = torch.empty(M, N, dtype=torch.float32, device=a.device)
    status = torch.zeros(1, dtype=torch.int32, device=a.device)
    st = (stream or torch.cuda.current_stream(a.device)).cuda_stream
    _check(lib().tpmlp_fp8_gemm(_ptr(a), a.shape[1], _ptr(b), b.shape[1], M, N, k, _ptr(inv_a), _ptr(inv_b),
                                _ptr(c), N, _ptr(status), st))
    return c, status


class TPMLP:
    """One context of the sublayer with its caller-owned workspace.

    Methods mirror the C entry points: ``forward``, ``mse_loss_grad``,
    ``backward``, ``bind_master``, ``sgd_step``, ``set_debug``, ``sync``."""

    def __init__(self, max_tokens: int, hidden: int, ffn: int, max_t: int = 8, dtype: str = "bf16",
                 act: str = "swiglu", device=None, stream: torch.cuda.Stream | None = None):
        dev = torch.device(device) if device is not None else torch.device("cuda")
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.cfg = make_config(max_tokens, hidden, ffn, max_t, dtype, act)
        self.dtype = _TORCH_DTYPE[_DTYPES[dtype]]
        self.act = act
        self.H, self.F = hidden, ffn
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.device(self.device):
            self.ctx = tpmlp_create(self.cfg, self.stream.cuda_stream)
            nbytes = tpmlp_workspace_bytes(self.cfg)
            self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        _check(lib().tpmlp_bind_workspace(self.ctx, _ptr(self.workspace), nbytes), self.ctx)
        self.tokens = 0
        self._fwd = False
        self._loss = torch.zeros(1, dtype=torch.float32, device=self.device)
        self._gn = torch.zeros(1, dtype=torch.float32, device=self.device)
        self._adam = None

    def close(self):
        if getattr(self, "ctx", None):
            lib().tpmlp_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- checks ------------------------------------------------------------
    def _t(self, t, shape, dtype=None, name="tensor"):
        if t is None:
            raise TPMLPError(ERR_ARG, f"{name} is None")
        want = dtype if dtype is not None else self.dtype
        if t.device != self.device or t.dtype != want or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise TPMLPError(ERR_ARG, f"{name}: need contiguous {want} {tuple(shape)} on {self.device}, "
                                      f"got {t.dtype} {tuple(t.shape)} on {t.device}")
        return _ptr(t)

    def _gu_shape(self):
        return (2, self.F, self.H) if self.act == "swiglu" else (self.F, self.H)

    # -- entry points --------------------------------------------------------
    def forward(self, x, norm_w, w_gate_up, w_down, b_down, eps: float, t: int, y=None, b_1=None):
        n = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        args = (self._t(x, (n, self.H), name="x"), self._t(norm_w, (self.H,), name="norm_w"),
                self._t(w_gate_up, self._gu_shape(), name="w_gate_up"),
                self._t(b_1, (self.F,), name="b_1") if self.act == "gelu" else None,
                self._t(w_down, (self.H, self.F), name="w_down"), self._t(b_down, (self.H,), name="b_down"))
        yp = self._t(y, (n, self.H), name="y")
        self._fwd = False
        _check(lib().tpmlp_forward(self.ctx, n, *args, float(eps), int(t), yp), self.ctx)
        # the library keeps these pointers (backward reads x; the updates write the parameters):
        # hold the tensors until the next forward so that a temporary argument is not freed
        self._fwd_tensors = (x, norm_w, w_gate_up, b_1, w_down, b_down)
        self.tokens = n
        self._fwd = True
        return y

    def _need_forward(self, what):
        if not self._fwd:
            raise TPMLPError(ERR_ORDER, f"{what} before forward")

    def mse_loss_grad(self, y, target, dy=None, loss=None):
        self._need_forward("mse_loss_grad")
        n = self.tokens
        dy = torch.empty_like(y) if dy is None else dy
        loss = self._loss if loss is None else loss
        _check(lib().tpmlp_mse_loss_grad(self.ctx, self._t(y, (n, self.H), name="y"),
                                         self._t(target, (n, self.H), name="target"),
                                         self._t(dy, (n, self.H), name="dy"),
                                         self._t(loss, (1,), torch.float32, "loss")), self.ctx)
        return loss, dy

    def new_grads(self):
        f32 = dict(dtype=torch.float32, device=self.device)
        g = {"norm_w": torch.empty(self.H, **f32), "w_gate_up": torch.empty(self._gu_shape(), **f32),
             "w_down": torch.empty(self.H, self.F, **f32), "b_down": torch.empty(self.H, **f32)}
        if self.act == "gelu":
            g["b_1"] = torch.empty(self.F, **f32)
        return g

    def backward(self, dy, dx=None, grads=None):
        self._need_forward("backward")
        n = self.tokens
        dx = torch.empty_like(dy) if dx is None else dx
        g = self.new_grads() if grads is None else grads
        f32 = torch.float32
        _check(lib().tpmlp_backward(
            self.ctx, self._t(dy, (n, self.H), name="dy"), self._t(dx, (n, self.H), name="dx"),
            self._t(g["norm_w"], (self.H,), f32, "dnorm_w"), self._t(g["w_gate_up"], self._gu_shape(), f32, "dw_gate_up"),
            self._t(g["b_1"], (self.F,), f32, "db_1") if self.act == "gelu" else None,
            self._t(g["w_down"], (self.H, self.F), f32, "dw_down"), self._t(g["b_down"], (self.H,), f32, "db_down")),
            self.ctx)
        # the updates read these gradients later: hold them until the next backward
        self._grads = g
        return dx, g

    def bind_master(self, masters: dict | None):
        f32 = torch.float32
        if masters is None:
            _check(lib().tpmlp_bind_master(self.ctx, None, None, None, None, None), self.ctx)
            self._masters = None
            return
        _check(lib().tpmlp_bind_master(
            self.ctx, self._t(masters["norm_w"], (self.H,), f32, "norm_w"),
            self._t(masters["w_gate_up"], self._gu_shape(), f32, "w_gate_up"),
            self._t(masters["b_1"], (self.F,), f32, "b_1") if self.act == "gelu" else None,
            self._t(masters["w_down"], (self.H, self.F), f32, "w_down"),
            self._t(masters["b_down"], (self.H,), f32, "b_down")), self.ctx)
        self._masters = masters  # keep the tensors alive while bound

    def sgd_step(self, lr: float):
        _check(lib().tpmlp_sgd_step(self.ctx, float(lr)), self.ctx)

    def set_update_in_backward(self, enable: bool, lr: float = 0.0):
        """Have backward apply the SGD update itself (bf16 with bound masters); sgd_step is then not called."""
        _check(lib().tpmlp_set_update_in_backward(self.ctx, int(bool(enable)), float(lr)), self.ctx)

    def update_in_epilogue(self) -> bool:
        """Whether the last backward updated the weight matrices inside their gradient GEMMs' epilogues."""
        return bool(lib().tpmlp_update_in_epilogue(self.ctx))

    def _param_set(self, d: dict, what: str) -> ParamSet:
        f32 = torch.float32
        return ParamSet(self._t(d["norm_w"], (self.H,), f32, f"{what}.norm_w"),
                        self._t(d["w_gate_up"], self._gu_shape(), f32, f"{what}.w_gate_up"),
                        self._t(d["b_1"], (self.F,), f32, f"{what}.b_1") if self.act == "gelu" else None,
                        self._t(d["w_down"], (self.H, self.F), f32, f"{what}.w_down"),
                        self._t(d["b_down"], (self.H,), f32, f"{what}.b_down"))

    def new_adam_state(self):
        """Zeroed first and second moments shaped like the parameters (fp32), bound to this context."""
        m = {k: torch.zeros_like(v) for k, v in self.new_grads().items()}
        v = {k: torch.zeros_like(t) for k, t in m.items()}
        self.bind_adam_state(m, v)
        return m, v

    def bind_adam_state(self, m: dict | None, v: dict | None):
        if m is None and v is None:
            _check(lib().tpmlp_bind_adam_state(self.ctx, None, None), self.ctx)
            self._adam = None
            return
        ms, vs = self._param_set(m, "m"), self._param_set(v, "v")
        _check(lib().tpmlp_bind_adam_state(self.ctx, ctypes.byref(ms), ctypes.byref(vs)), self.ctx)
        self._adam = (m, v)  # keep the tensors alive while bound

    def adamw_step(self, lr: float, step: int, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                   weight_decay: float = 0.1, max_grad_norm: float = 1.0, grad_norm=None):
        """One clipped AdamW update; returns the device float holding the global gradient norm."""
        gn = self._gn if grad_norm is None else grad_norm
        hp = AdamWParams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                         float(max_grad_norm), int(step))
        _check(lib().tpmlp_adamw_step(self.ctx, ctypes.byref(hp), self._t(gn, (1,), torch.float32, "grad_norm")),
               self.ctx)
        return gn

    def set_precision(self, precision: str):
        """"bf16" or "fp8" GEMM operands; the first switch to FP8 allocates and binds its workspace."""
        prec = {"bf16": PREC_BF16, "fp8": PREC_FP8}[precision]
        if prec == PREC_FP8 and getattr(self, "workspace8", None) is None:
            nbytes = lib().tpmlp_fp8_workspace_bytes(ctypes.byref(self.cfg))
            if nbytes == 0:
                raise TPMLPError(ERR_UNSUPPORTED, "FP8 needs the bf16 dtype")
            self.workspace8 = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            _check(lib().tpmlp_bind_fp8_workspace(self.ctx, _ptr(self.workspace8), nbytes), self.ctx)
        _check(lib().tpmlp_set_precision(self.ctx, prec), self.ctx)
        self._fwd = False

    def set_sequence_parallel(self, enable: bool):
        _check(lib().tpmlp_set_sequence_parallel(self.ctx, int(bool(enable))), self.ctx)
        self._fwd = False

    def set_debug(self, flags: int, shard: int = 0):
        _check(lib().tpmlp_set_debug(self.ctx, int(flags), int(shard)), self.ctx)

    def sync(self):
        _check(lib().tpmlp_sync(self.ctx), self.ctx)

    def set_timing(self, enable: bool):
        _check(lib().tpmlp_set_timing(self.ctx, 1 if enable else 0), self.ctx)

    def read_kernel_times(self) -> dict:
        n = lib().tpmlp_num_kernel_ids()
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int64 * n)()
        m = lib().tpmlp_read_kernel_times(self.ctx, ms, cnt, n)
        if m < 0:
            raise TPMLPError(ERR_CUDA, "reading kernel times failed")
        names = kernel_names()
        return {names[i]: (float(ms[i]), int(cnt[i])) for i in range(m) if cnt[i] > 0}

    def launch_count(self) -> int:
        return int(lib().tpmlp_launch_count(self.ctx))


def _acheck(status: int, ctx=None):
    if status != OK:
        msg = lib().tpattn_last_error(ctx).decode(errors="replace")
        raise TPMLPError(status, msg or lib().tpmlp_status_string(status).decode())


class TPAttn:
    """The tensor-parallel attention sublayer through the C ABI (tpattn_*):
    bf16 tensors on one CUDA device; the workspace is a torch uint8 tensor."""

    def __init__(self, max_tokens: int, hidden: int, n_heads: int, n_kv_heads: int, head_dim: int,
                 max_seq: int, max_t: int = 8, device=None, stream=None, fused_only: bool = False):
        dev = torch.device(device) if device is not None else torch.device("cuda")
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.cfg = AttnConfig(max_tokens, hidden, n_heads, n_kv_heads, head_dim, max_seq, max_t, BF16,
                              TPATTN_FUSED_ONLY if fused_only else 0)
        self.H, self.nq, self.nkv, self.d = hidden, n_heads, n_kv_heads, head_dim
        self.W = (n_heads + 2 * n_kv_heads) * head_dim
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        ctx = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _acheck(lib().tpattn_create(ctypes.byref(self.cfg), self.stream.cuda_stream, ctypes.byref(ctx)))
            self.ctx = ctx
            nbytes = int(lib().tpattn_workspace_bytes(ctypes.byref(self.cfg)))
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        _acheck(lib().tpattn_bind_workspace(self.ctx, _ptr(self.workspace), nbytes), self.ctx)
        self._masters = None
        self.tokens = None  # set by forward; the C ABI reports a backward before it

    def close(self):
        if getattr(self, "ctx", None):
            lib().tpattn_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _t(self, t, shape, dtype=torch.bfloat16, name="tensor"):
        if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or t.device != self.device:
            raise TPMLPError(ERR_ARG, f"{name}: expected contiguous {dtype} {tuple(shape)} on {self.device}")
        return _ptr(t)

    def forward(self, x, norm_w, w_qkv, w_o, b_o, eps: float, t: int, batch: int, seq: int, y=None):
        y = torch.empty_like(x) if y is None else y
        n = batch * seq
        _acheck(lib().tpattn_forward(self.ctx, batch, seq, self._t(x, (n, self.H), name="x"),
                                     self._t(norm_w, (self.H,), name="norm_w"),
                                     self._t(w_qkv, (self.W, self.H), name="w_qkv"),
                                     self._t(w_o, (self.H, self.nq * self.d), name="w_o"),
                                     self._t(b_o, (self.H,), name="b_o"), float(eps), int(t),
                                     self._t(y, (n, self.H), name="y")), self.ctx)
        # the library keeps these pointers (backward reads x; the updates write the parameters):
        # hold the tensors until the next forward so that a temporary argument is not freed
        self._fwd_tensors = (x, norm_w, w_qkv, w_o, b_o)
        self.params = (norm_w, w_qkv, w_o, b_o)
        self.tokens = n
        return y

    def new_grads(self):
        f = dict(dtype=torch.float32, device=self.device)
        return {"norm_w": torch.empty(self.H, **f), "w_qkv": torch.empty(self.W, self.H, **f),
                "w_o": torch.empty(self.H, self.nq * self.d, **f), "b_o": torch.empty(self.H, **f)}

    def backward(self, dy, dx=None, grads=None):
        dx = torch.empty_like(dy) if dx is None else dx
        g = self.new_grads() if grads is None else grads
        f32 = torch.float32
        n = dy.shape[0] if self.tokens is None else self.tokens
        _acheck(lib().tpattn_backward(self.ctx, self._t(dy, (n, self.H), name="dy"),
                                      self._t(dx, (n, self.H), name="dx"),
                                      self._t(g["norm_w"], (self.H,), f32, "dnorm_w"),
                                      self._t(g["w_qkv"], (self.W, self.H), f32, "dw_qkv"),
                                      self._t(g["w_o"], (self.H, self.nq * self.d), f32, "dw_o"),
                                      self._t(g["b_o"], (self.H,), f32, "db_o")), self.ctx)
        # the updates read these gradients later: hold them until the next backward
        self._grads = g
        return dx, g

    def bind_master(self, m: dict | None):
        if m is None:
            _acheck(lib().tpattn_bind_master(self.ctx, None, None, None, None), self.ctx)
            self._masters = None
            return
        f32 = torch.float32
        _acheck(lib().tpattn_bind_master(self.ctx, self._t(m["norm_w"], (self.H,), f32, "norm_w"),
                                         self._t(m["w_qkv"], (self.W, self.H), f32, "w_qkv"),
                                         self._t(m["w_o"], (self.H, self.nq * self.d), f32, "w_o"),
                                         self._t(m["b_o"], (self.H,), f32, "b_o")), self.ctx)
        self._masters = m

    def sgd_step(self, lr: float):
        _acheck(lib().tpattn_sgd_step(self.ctx, float(lr)), self.ctx)

    def set_update_in_backward(self, enable: bool, lr: float = 0.0):
        """Have backward apply the SGD update itself (needs bound masters); sgd_step is then not called."""
        _acheck(lib().tpattn_set_update_in_backward(self.ctx, int(bool(enable)), float(lr)), self.ctx)

    def update_in_epilogue(self) -> bool:
        """Whether the last backward updated W_qkv and W_o inside their gradient GEMMs' epilogues."""
        return bool(lib().tpattn_update_in_epilogue(self.ctx))

    def _param_set(self, d: dict, what: str) -> AttnParamSet:
        f32 = torch.float32
        return AttnParamSet(self._t(d["norm_w"], (self.H,), f32, f"{what}.norm_w"),
                            self._t(d["w_qkv"], (self.W, self.H), f32, f"{what}.w_qkv"),
                            self._t(d["w_o"], (self.H, self.nq * self.d), f32, f"{what}.w_o"),
                            self._t(d["b_o"], (self.H,), f32, f"{what}.b_o"))

    def new_adam_state(self):
        """Zeroed first and second moments shaped like the parameters (fp32), bound to this context."""
        m = {k: torch.zeros_like(v) for k, v in self.new_grads().items()}
        v = {k: torch.zeros_like(t) for k, t in m.items()}
        self.bind_adam_state(m, v)
        return m, v

    def bind_adam_state(self, m: dict | None, v: dict | None):
        if m is None and v is None:
            _acheck(lib().tpattn_bind_adam_state(self.ctx, None, None), self.ctx)
            self._adam = None
            return
        ms, vs = self._param_set(m, "m"), self._param_set(v, "v")
        _acheck(lib().tpattn_bind_adam_state(self.ctx, ctypes.byref(ms), ctypes.byref(vs)), self.ctx)
        self._adam = (m, v)  # keep the tensors alive while bound

    def adamw_step(self, lr: float, step: int, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                   weight_decay: float = 0.1, max_grad_norm: float = 1.0, grad_norm=None):
        """One clipped AdamW update; returns the device float holding the global gradient norm."""
        if grad_norm is None:
            if getattr(self, "_gn", None) is None:
                self._gn = torch.zeros(1, dtype=torch.float32, device=self.device)
            grad_norm = self._gn
        hp = AdamWParams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                         float(max_grad_norm), int(step))
        _acheck(lib().tpattn_adamw_step(self.ctx, ctypes.byref(hp),
                                        self._t(grad_norm, (1,), torch.float32, "grad_norm")), self.ctx)
        return grad_norm

    def sync(self):
        _acheck(lib().tpattn_sync(self.ctx), self.ctx)

    def set_fused(self, enable: bool):
        """Fused attention kernels where the shape allows (the default), or always the unfused path."""
        _acheck(lib().tpattn_set_fused(self.ctx, int(bool(enable))), self.ctx)

    def fused_active(self) -> bool:
        """Whether the last forward ran the fused kernels."""
        return bool(lib().tpattn_fused_active(self.ctx))

    def set_timing(self, enable: bool):
        _acheck(lib().tpattn_set_timing(self.ctx, int(bool(enable))), self.ctx)

    def read_kernel_times(self) -> dict:
        n = lib().tpattn_num_kernel_ids()
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int64 * n)()
        lib().tpattn_read_kernel_times(self.ctx, ms, cnt, n)
        return {lib().tpattn_kernel_name(i).decode(): (float(ms[i]), int(cnt[i])) for i in range(n) if cnt[i]}

    def launch_count(self) -> int:
        return int(lib().tpattn_launch_count(self.ctx))
