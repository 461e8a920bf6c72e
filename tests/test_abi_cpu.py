"""The C-ABI library builds, loads and exports every entry point its header
declares; host-side validation rejects bad configurations without a GPU."""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")


@pytest.fixture(scope="module")
def T():
    from tensor_transformer_mlp_rmsnorm_gb300 import build
    build.build()
    import tensor_transformer_mlp_rmsnorm_gb300 as T
    return T


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^TPMLP_API\s+[\w\s\*]+?\b(tp(?:mlp|attn)_\w+)\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("tpmlp_forward", "tpmlp_backward", "tpmlp_sgd_step", "tpmlp_mse_loss_grad", "tpmlp_create",
                 "tpmlp_workspace_bytes", "tpmlp_bind_workspace", "tpmlp_sync", "tpmlp_destroy",
                 "tpmlp_adamw_step", "tpmlp_set_sequence_parallel", "tpmlp_set_precision", "tpmlp_fp8_quantize",
                 "tpmlp_fp8_gemm", "tpattn_forward", "tpattn_backward", "tpattn_sgd_step",
                 "tpattn_bind_adam_state", "tpattn_adamw_step"):
        assert must in names


def test_library_exports_every_declared_symbol(T):
    L = ctypes.CDLL(T.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_every_symbol(T):
    from tensor_transformer_mlp_rmsnorm_gb300 import tpmlp
    assert set(declared_functions()) <= set(tpmlp._SIGNATURES)


def test_config_validation_without_gpu(T):
    good = T.make_config(16, 64, 256, 2, "f32", "swiglu")
    assert T.tpmlp_workspace_bytes(good) > 0
    cases = [
        (dict(ffn=12), T.ERR_SHAPE),          # not a multiple of 8
        (dict(hidden=0), T.ERR_SHAPE),
        (dict(hidden=16384), T.ERR_SHAPE),    # above the supported hidden size
        (dict(max_t=0), T.ERR_SHAPE),
        (dict(max_tokens=-1), T.ERR_SHAPE),
        (dict(dtype=7), T.ERR_UNSUPPORTED),
        (dict(act=3), T.ERR_UNSUPPORTED),
        (dict(reserved=1), T.ERR_ARG),
    ]
    for kw, status in cases:
        c = T.make_config(16, 64, 256, 2, "f32", "swiglu")
        for k, v in kw.items():
            setattr(c, k, v)
        assert T.tpmlp_workspace_bytes(c) == 0, kw
        with pytest.raises(T.TPMLPError) as e:
            T.tpmlp_create(c)
        assert e.value.status == status, (kw, e.value)


def test_workspace_layout_grows_with_tokens(T):
    a = T.tpmlp_workspace_bytes(T.make_config(1024, 512, 1536, 8, "bf16", "swiglu"))
    b = T.tpmlp_workspace_bytes(T.make_config(2048, 512, 1536, 8, "bf16", "swiglu"))
    per_token = 512 * 2 + 4 + 2 * 1536 * 2 + 1536 * 2 + 2 * 1536 * 2 + 512 * 4  # n, rstd, GU, A, dGU, dN
    assert b - a >= 1024 * per_token
    assert a % 256 == 0 and b % 256 == 0


def test_status_strings_and_kernel_names(T):
    L = T.lib()
    for s in range(7):
        assert L.tpmlp_status_string(s)
    names = T.kernel_names()
    assert len(names) == L.tpmlp_num_kernel_ids() and "gemm_down_reduce" in names
    assert L.tpmlp_kernel_name(-1) is None and L.tpmlp_kernel_name(len(names)) is None


def test_null_context_is_rejected(T):
    L = T.lib()
    assert L.tpmlp_sgd_step(None, 0.1) == T.ERR_ARG
    assert L.tpmlp_sync(None) == T.ERR_ARG
    assert L.tpmlp_launch_count(None) == 0
    L.tpmlp_destroy(None)
    assert L.tpmlp_adamw_step(None, None, None) == T.ERR_ARG
    assert L.tpmlp_set_update_in_backward(None, 1, 0.1) == T.ERR_ARG
    assert L.tpmlp_update_in_epilogue(None) == 0
    assert L.tpattn_sgd_step(None, 0.1) == T.ERR_ARG
    assert L.tpattn_set_update_in_backward(None, 1, 0.1) == T.ERR_ARG
    assert L.tpattn_update_in_epilogue(None) == 0
    assert L.tpattn_bind_adam_state(None, None, None) == T.ERR_ARG
    assert L.tpattn_adamw_step(None, None, None) == T.ERR_ARG
    assert L.tpattn_sync(None) == T.ERR_ARG
    assert L.tpattn_launch_count(None) == 0
    L.tpattn_destroy(None)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from tensor_transformer_mlp_rmsnorm_gb300 import tpmlp
    monkeypatch.setattr(tpmlp, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(tpmlp, "_LIB", None)
    with pytest.raises(tpmlp.TPMLPError):
        tpmlp.lib()


def test_fp8_and_attention_validation_without_gpu(T):
    from tensor_transformer_mlp_rmsnorm_gb300 import tpmlp
    L = T.lib()
    bf = T.make_config(64, 128, 512, 8, "bf16", "swiglu")
    f32 = T.make_config(64, 128, 512, 8, "f32", "swiglu")
    assert L.tpmlp_fp8_workspace_bytes(ctypes.byref(bf)) > 0
    assert L.tpmlp_fp8_workspace_bytes(ctypes.byref(f32)) == 0
    buf = ctypes.create_string_buffer(64)  # host memory: every call below is rejected before touching it
    p = ctypes.cast(buf, ctypes.c_void_p)
    # cols not a multiple of 8; no output at all; negative rows
    assert L.tpmlp_fp8_quantize(p, 4, 12, p, 16, None, 0, p, p, None) == T.ERR_SHAPE
    assert L.tpmlp_fp8_quantize(p, 4, 16, None, 0, None, 0, p, p, None) == T.ERR_ARG
    assert L.tpmlp_fp8_quantize(p, -1, 16, p, 16, None, 0, p, p, None) == T.ERR_SHAPE
    # N not a multiple of 4; pitch below K
    assert L.tpmlp_fp8_gemm(p, 16, p, 16, 4, 6, 16, p, p, p, 8, p, None) == T.ERR_SHAPE
    assert L.tpmlp_fp8_gemm(p, 16, p, 16, 4, 8, 32, p, p, p, 8, p, None) == T.ERR_ARG
    # attention configs
    good = tpmlp.AttnConfig(512, 256, 4, 2, 64, 128, 2, T.BF16, 0)
    assert L.tpattn_workspace_bytes(ctypes.byref(good)) > 0
    bad = [dict(n_heads=3), dict(head_dim=96), dict(max_seq=100), dict(max_t=4), dict(dtype=T.F32),
           dict(hidden=12), dict(flags=2), dict(max_seq=8192)]
    for kw in bad:
        c = tpmlp.AttnConfig(512, 256, 4, 2, 64, 128, 2, T.BF16, 0)
        for k, v in kw.items():
            setattr(c, k, v)
        assert L.tpattn_workspace_bytes(ctypes.byref(c)) == 0, kw
        ctx = ctypes.c_void_p()
        assert L.tpattn_create(ctypes.byref(c), None, ctypes.byref(ctx)) == T.ERR_SHAPE, kw
        assert L.tpattn_last_error(None)


def test_attention_fused_only_config_without_gpu(T):
    """TPATTN_FUSED_ONLY drops the score square from the workspace and admits
    sequences past 4096 (multiples of 128), for head_dim 128 only."""
    from tensor_transformer_mlp_rmsnorm_gb300 import tpmlp
    L = T.lib()
    F = tpmlp.TPATTN_FUSED_ONLY

    def ws(**kw):
        c = tpmlp.AttnConfig(8192, 1024, 8, 2, 128, 2048, 2, T.BF16, 0)
        for k, v in kw.items():
            setattr(c, k, v)
        return L.tpattn_workspace_bytes(ctypes.byref(c))

    plain, fused = ws(), ws(flags=F)
    square = 8192 * 2048 * 8 * (4 + 2)  # f32 scores and bf16 probabilities, batch * n_q * S^2
    assert plain - fused >= square
    assert ws(flags=F, max_seq=16384, max_tokens=16384) > 0
    assert ws(max_seq=16384, max_tokens=16384) == 0      # only without the square
    assert ws(flags=F, max_seq=1984) == 0                  # not a multiple of 128
    assert ws(flags=F, head_dim=64) == 0                   # fused kernels need head_dim 128
    assert ws(flags=F, max_seq=65536) == 0


def test_traffic_record_lookup(tmp_path, monkeypatch):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "tensor_transformer_mlp_rmsnorm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for fam in bench.KERNEL_FAMILIES.values():
        for f in fam:
            (csrc / f).write_text("// " + f)
    dg = dict(x.split(":") for x in bench.source_digests().split(","))
    (tmp_path / "profiles" / "x.md").write_text(
        "text\ntraffic-record: workload=w t=8 tokens=16 digest=gemm:%s,rowwise:deadbeef gemm_a=123 sgd_update=7\n"
        "traffic-record: workload=w t=8 tokens=16 precision=fp8 digest=gemm:%s gemm_a=55\n" % (dg["gemm"], dg["gemm"]))
    assert bench.recorded_traffic("w", 8, 16, "gemm_a") == (123.0, "profiles/x.md")
    assert bench.recorded_traffic("w", 8, 16, "gemm_a", "fp8") == (55.0, "profiles/x.md")
    assert bench.recorded_traffic("w", 8, 16, "sgd_update") == (None, None)  # rowwise digest does not match
    assert bench.recorded_traffic("w", 4, 16, "gemm_a") == (None, None)
    (tmp_path / "profiles" / "y.md").write_text(
        "traffic-record: workload=a t=8 tokens=32 digest=flash:%s flash_attn_bwd=99\n" % dg["flash"])
    assert bench.kernel_family("flash_attn_bwd") == "flash"
    assert bench.recorded_traffic("a", 8, 32, "flash_attn_bwd") == (99.0, "profiles/y.md")
    (csrc / "gemm_tc.cu").write_text("// changed")
    assert bench.recorded_traffic("w", 8, 16, "gemm_a") == (None, None)
    assert bench.recorded_traffic("a", 8, 32, "flash_attn_bwd") == (99.0, "profiles/y.md")
    (csrc / "flash_attn.cu").write_text("// changed")
    assert bench.recorded_traffic("a", 8, 32, "flash_attn_bwd") == (None, None)


def test_cpu_baselines_time_the_oracle_on_a_bounded_sample():
    # the bench's CPU legs: both report a positive rate on a sample no larger than asked for
    import dataclasses
    import bench
    import synth
    cfg = synth.CONFIGS["fp32_small"]
    inp = synth.make_inputs(cfg, seed=3)
    v, n, dt = bench.cpu_oracle_tflops(cfg, inp, budget_s=0.0, min_tokens=8, max_tokens=16)
    assert v > 0 and n == 8 and dt > 0
    acfg = dataclasses.replace(synth.ATTN_CONFIGS["attn_small"], batch=2, seq=256, hidden=128, n_q=2, n_kv=1, d=64)
    ainp = synth.make_attn_inputs(acfg, seed=3)
    v, n, dt = bench.cpu_attn_oracle_tflops(acfg, ainp, budget_s=0.0, min_seq=64, max_seq=128)
    assert v > 0 and n == 64 and dt > 0
    v, n, dt = bench.cpu_attn_oracle_tflops(acfg, ainp, budget_s=1e9, min_seq=64, max_seq=128)
    assert n == 128  # doubled up to the cap, never past it


def test_peak_choice_follows_clock_and_region_length():
    # burst only for a short region at near-maximum clock; the contraction-dtype ratio scales both
    import bench
    pk = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    hot = {"sm_mhz": 2000, "sm_max_mhz": 2070}
    slow = {"sm_mhz": 1700, "sm_max_mhz": 2070}
    assert bench.choose_peak(pk, hot, 0.5) == (1900.0, "burst")
    assert bench.choose_peak(pk, hot, 3.0) == (1700.0, "sustained")
    assert bench.choose_peak(pk, slow, 0.5) == (1700.0, "sustained")
    assert bench.choose_peak(pk, None, 0.5) == (1700.0, "sustained")
    assert bench.choose_peak(pk, hot, 0.5, ratio=2.0) == (3800.0, "burst")


def test_reference_arm_prints_the_gpu_arms_config(capsys, monkeypatch):
    # the reference line carries the metric and config the GPU arm builds for the same options
    import argparse
    import bench
    import synth
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    base = dict(steps=1, warmup=0, ref_tokens=16, t=8, tokens=0, optimizer="sgd", precision="bf16",
                sequence_parallel=False, attn_path="fused")
    args = argparse.Namespace(workload="bf16_llama8b", **base)
    assert bench.reference_arm(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    cfg = synth.CONFIGS["bf16_llama8b"]
    n_params = sum(int(v.size) for k, v in synth.make_inputs(cfg.with_tokens(16), seed=1234).items()
                   if k in synth.param_names(cfg.act))
    assert line["config"] == json.loads(json.dumps(bench.mlp_config(cfg, 8, 1, args, n_params)))
    assert line["metric"] == bench.metric_name(args, False) and line["impl"] == "reference"
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    args = argparse.Namespace(workload="attn_gpt_h4096", **dict(base, ref_tokens=64))
    assert bench.reference_arm(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    acfg, t, fused = bench.attn_run(args)
    assert fused and line["config"] == json.loads(json.dumps(bench.attn_config(acfg, t, 1, args, fused)))
    assert line["metric"] == bench.metric_name(args, True)
