"""Megatron tensor-parallel MLP sublayer (pre-RMSNorm, SwiGLU or GeLU) on one
GB300: hand-written sm_103a CUDA kernels behind the C ABI in
``include/tpmlp.h``, with a thin ctypes binding.

    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP
    m = TPMLP(max_tokens, hidden, ffn, max_t=8, dtype="bf16", act="swiglu")
    y = m.forward(x, norm_w, w_gate_up, w_down, b_down, eps=1e-6, t=8)
    loss, dy = m.mse_loss_grad(y, target)
    dx, grads = m.backward(dy)
    m.sgd_step(lr)                      # or: m.new_adam_state(); m.adamw_step(lr, step=1)

The library must be built first (``build.build()``); without it every call
raises ``TPMLPError``.
"""
from .tpmlp import (  # noqa: F401
    BF16, DBG_FORCE_TIMEOUT, DBG_GEMM_SINGLE_CTA, DBG_SKIP_BWD_REDUCE, DBG_SKIP_FWD_REDUCE, DBG_SKIP_SP_GRAD_SYNC,
    ERR_ARG, ERR_ORDER, ERR_SHAPE, PREC_BF16, PREC_FP8,
    ERR_TIMEOUT, ERR_UNSUPPORTED, F32, GELU, LIB_PATH, SWIGLU, TPMLP, TPAttn, AdamWParams, Config, ParamSet, TPMLPError,
    fp8_gemm, fp8_quantize, kernel_names, lib,
    make_config, tpmlp_create, tpmlp_workspace_bytes,
)
