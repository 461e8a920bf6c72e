"""Benchmark of one training step of the tensor-parallel MLP sublayer:
forward -> MSE loss -> backward -> SGD, on the Llama-3-8B-shaped bf16 SwiGLU
block (16384 tokens = 4 x 4096, hidden 4096, ffn 14336, t = 8 logical
shards), through the library's public API.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is whole-job GEMM TFLOP/s
(18 N H F algorithmic flops per step) with every input resident in HBM; the
``e2e`` figure adds the per-step host->device copy of x and the target from
pinned memory (on a copy stream, double-buffered so that the next step's copy
overlaps the current step) and the device->host read of the loss.  With N > 1 (torchrun)
every rank runs an independent replica of the step on its own GPU (the path
has no data exchange between replicas), so scaling is weak.

``--impl reference`` times the CPU oracle (float64 numpy) on the host cores on
a bounded token sample of the same workload; it is the reference arm here.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

# the walkthrough's launch example ("Stage 8" optimizer): lr 1.5e-4, weight decay 0.1, clip 1.0;
# Adam's published moment rates and epsilon
ADAMW = {"lr": 1.5e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.1, "max_grad_norm": 1.0}
DESCR = {"bf16_llama8b": "Llama-3-8B-shaped MLP sublayer", "bf16_h2048": "H=2048 MLP sublayer",
         "bf16_gelu_h4096": "GPT-style GeLU MLP sublayer", "bf16_70b_n2048": "Llama-2-70B-shaped MLP sublayer",
         "fp32_small": "small fp32 MLP sublayer"}
METRIC = "TP-MLP fwd+bwd+SGD TFLOP/s at 1 GB300 and % of BF16 dense tensor peak"
WORKLOAD = "bf16_llama8b"
T_SHARDS = 8
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# algorithmic flops per launch of each GEMM, in units of N*H*F (SwiGLU; the GeLU block has one
# first-projection matrix, so its gate/up-shaped GEMMs are 2 N H F as well)
GEMM_UNITS = {"gemm_gateup_act": 4, "gemm_down_reduce": 2, "gemm_dgrad_act": 2, "gemm_wgrad_down": 2,
              "gemm_wgrad_gateup": 4, "gemm_dgrad_norm_reduce": 4}
GELU_UNITS = dict(GEMM_UNITS, gemm_gateup_act=2, gemm_wgrad_gateup=2, gemm_dgrad_norm_reduce=2)
# kernel sources per family: a change to any of them invalidates the recorded DRAM traffic of that
# family's kernels
KERNEL_FAMILIES = {
    "gemm": ("gemm_tc.cu", "gemm_simt.cu", "ptx_sm103.cuh", "epilogue.cuh", "tma_maps.cuh", "f32x2.cuh"),
    "rowwise": ("rowwise.cu", "vec.cuh", "epilogue.cuh"),
    "optim": ("optim.cu", "vec.cuh"),
    "fp8": ("fp8.cu",),
    "flash": ("flash_attn.cu", "ptx_sm103.cuh", "f32x2.cuh", "tma_maps.cuh", "vec.cuh"),
}


def kernel_family(kernel: str) -> str:
    if kernel.startswith("gemm_"):
        return "gemm"
    if kernel.startswith("flash_"):
        return "flash"
    if kernel in ("fp8_amax", "fp8_cast"):
        return "fp8"
    return "optim" if kernel in ("grad_sqnorm", "adamw_update") else "rowwise"


def kernel_source_digest(family: str) -> str:
    """sha256 (first 16 hex digits) over one kernel family's sources, in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_FAMILIES[family]:
        with open(os.path.join(ROOT, "tensor_transformer_mlp_rmsnorm_gb300", "csrc", f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def source_digests() -> str:
    """The `digest=` field of a traffic record for the current sources."""
    return ",".join(f"{fam}:{kernel_source_digest(fam)}" for fam in sorted(KERNEL_FAMILIES))


def recorded_traffic(workload: str, t: int, tokens: int, kernel: str, precision: str = "bf16"):
    """DRAM bytes (read + write) per launch of `kernel`, from a `traffic-record:` line of an ncu
    summary under profiles/ taken on the same workload and on the current sources of the kernel's
    family; None if there is none (never measured, or the kernel changed since)."""
    import glob
    fam = kernel_family(kernel)
    want = kernel_source_digest(fam)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(path):
            if not line.startswith("traffic-record:"):
                continue
            kv = dict(tok.split("=", 1) for tok in line.split()[1:] if "=" in tok)
            digests = dict(d.split(":", 1) for d in kv.get("digest", "").split(",") if ":" in d)
            if (kv.get("workload") == workload and kv.get("t") == str(t) and kv.get("tokens") == str(tokens)
                    and kv.get("precision", "bf16") == precision and digests.get(fam) == want and kernel in kv):
                return float(kv[kernel]), os.path.relpath(path, ROOT)
    return None, None


def hbm_bytes(kernel: str, cfg, masters: bool, update_in_backward: bool = False):
    """Algorithmic HBM bytes of one launch of a memory-bound kernel.  With the update in backward
    the SGD kernel updates only the vectors (the matrices are updated in their GEMMs' epilogues)."""
    N, H, F = cfg.tokens, cfg.hidden, cfg.ffn
    e = 2 if cfg.dtype == "bf16" else 4
    P = 3 * F * H + 2 * H if cfg.act == "swiglu" else 2 * F * H + F + 2 * H
    Pu = (2 * H if cfg.act == "swiglu" else F + 2 * H) if update_in_backward else P
    return {"rmsnorm_fwd": 2 * N * H * e + 4 * N + H * e,
            "mse_loss_grad": 3 * N * H * e,
            "rmsnorm_bwd_residual": N * H * 4 + 3 * N * H * e + 4 * N + H * e,
            "sgd_update": Pu * (12 + e) if masters else Pu * (4 + 2 * e),
            "grad_sqnorm": 4 * P,
            "adamw_update": P * (28 + e) if masters else P * (20 + 2 * e)}.get(kernel)


def update_placement(adamw: bool, in_backward: bool, matrices_in_epilogue: bool) -> str:
    """Where the timed step applies its parameter update."""
    if adamw:
        return "AdamW: norm pass and update kernel after backward"
    if not in_backward:
        return "SGD: update kernel after backward"
    return ("SGD in backward: weight matrices in their gradient GEMMs' epilogues, vectors by the update kernel"
            if matrices_in_epilogue else "SGD in backward: update kernel at the end of backward")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def choose_peak(pk: dict, clk, region_s: float, ratio: float = 1.0):
    """The measured bf16 peak that applies to a kernel timed in this run.

    The burst figure applies when the timed region was short (under about a
    second, inside the power cap's averaging window) and the median SM clock
    stayed within 5% of its maximum; otherwise the sustained figure (the same
    GEMM held seconds under the cap).  Returns (peak, kind)."""
    near_max = bool(clk) and clk.get("sm_max_mhz") and clk["sm_mhz"] >= 0.95 * clk["sm_max_mhz"]
    if near_max and region_s < 1.0:
        return ratio * pk["bf16_tflops"], "burst"
    return ratio * pk["bf16_tflops_sustained"], "sustained"



def max_over_ranks(torch, times, dev, world: int):
    """Each timing as its maximum over the ranks (an all-reduce on `dev`; unchanged at one rank)."""
    if world <= 1:
        return list(times)
    tt = torch.tensor([float(v) for v in times], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in tt.tolist()]


def job_tflops(flops_per_rank_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return flops_per_rank_step * steps * world / (ms / 1e3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7], "sw_power": parts[8]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def instrumented_pass(torch, m, step, stream, steps: int) -> float:
    """Run `steps` more steps with the library's per-kernel CUDA events enabled; returns their
    wall time in ms (device events on the library's stream)."""
    m.set_timing(True)
    m.read_kernel_times()  # start from empty records
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def h2d_gbps(torch, host, dev, reps: int = 3) -> float:
    """Host-to-device copy rate of one pinned buffer alone (GB/s), for reading the e2e figure."""
    dev.copy_(host, non_blocking=True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        dev.copy_(host, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return reps * host.numel() * host.element_size() / (a.elapsed_time(b) / 1e3) / 1e9


def timed_e2e(torch, run_step, stream, x_host, tg_host, xbufs, tbufs, loss, loss_host, steps: int) -> float:
    """Milliseconds for `steps` training steps fed from pinned host memory.

    Every step copies its x and target host->device and reads its loss back device->host. The
    copies run on a second stream into two device buffers, so the copy for step i+1 overlaps the
    compute of step i (as a training loop with a prefetching loader does); the compute stream
    itself carries no copy. A buffer is refilled only after the step that used it has finished,
    since the backward reads x again. The timer starts before the first copy and stops once the
    last step has finished and its loss has been read.
    """
    copy = torch.cuda.Stream(device=stream.device)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    done = torch.cuda.Event()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    copy.wait_event(f0)

    def fill(i):
        b = i % 2
        if i >= 2:
            copy.wait_event(free[b])
        with torch.cuda.stream(copy):
            xbufs[b].copy_(x_host, non_blocking=True)
            tbufs[b].copy_(tg_host, non_blocking=True)
        ready[b].record(copy)

    fill(0)
    if steps > 1:
        fill(1)
    for i in range(steps):
        b = i % 2
        stream.wait_event(ready[b])
        if i > 0:
            stream.wait_event(done)  # the previous step's loss has been read before it is overwritten
        with torch.cuda.stream(stream):
            run_step(xbufs[b], tbufs[b])
        free[b].record(stream)
        # the loss read, then the next-but-one step's inputs, queue on the copy stream behind it
        copy.wait_event(free[b])
        with torch.cuda.stream(copy):
            loss_host.copy_(loss, non_blocking=True)
        done.record(copy)
        if i + 2 < steps:
            fill(i + 2)
    stream.wait_event(done)
    f1.record(stream)
    torch.cuda.synchronize()
    return f0.elapsed_time(f1)


def cpu_oracle_tflops(cfg, inp, budget_s: float, min_tokens: int = 16, max_tokens: int = 4096):
    """Time the oracle's dense step on a token sample sized to about budget_s."""
    from oracle import tpmlp_oracle as O
    p = {k: inp[k] for k in synth.param_names(cfg.act)}

    def run(n):
        t0 = time.perf_counter()
        O.dense_step(p, inp["x"][:n], inp["target"][:n], cfg.eps, cfg.lr, cfg.act)
        return time.perf_counter() - t0

    n = min_tokens
    dt = run(n)
    while dt < budget_s / 4 and n < max_tokens:
        n = min(max_tokens, n * 2)
        dt = run(n)
    flops = cfg.gemm_flops * n / cfg.tokens
    return flops / dt / 1e12, n, dt


def cpu_attn_oracle_tflops(cfg, inp, budget_s: float, min_seq: int = 128, max_seq: int = 2048):
    """Time the attention oracle's dense step on the first tokens of sequence 0 (a causal prefix
    is a complete smaller problem), doubling the prefix up to about budget_s."""
    from oracle import tpmlp_oracle as O
    p = {k: inp[k] for k in ("norm_w", "w_qkv", "w_o", "b_o")}

    def run(n):
        t0 = time.perf_counter()
        O.attn_dense_step(p, inp["x"][:n], inp["target"][:n], cfg.eps, cfg.lr, 1, cfg.n_q, cfg.n_kv)
        return time.perf_counter() - t0

    n = min(min_seq, cfg.seq)
    dt = run(n)
    while dt < budget_s / 4 and n < min(max_seq, cfg.seq):
        n = min(max_seq, cfg.seq, n * 2)
        dt = run(n)
    flops = dataclasses.replace(cfg, batch=1, seq=n).gemm_flops
    return flops / dt / 1e12, n, dt


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def workload_config(cfg, t: int, world: int) -> dict:
    return {"workload": f"{cfg.name}: {DESCR.get(cfg.name, 'MLP sublayer')}, "
                        f"{'SwiGLU' if cfg.act == 'swiglu' else 'GeLU'}, tokens={cfg.tokens} "
                        f"({cfg.batch}x{cfg.seq}), hidden={cfg.hidden}, ffn={cfg.ffn}, t={t} logical shards, "
                        f"lr={cfg.lr}",
            "global_batch": cfg.batch * world, "seq_len": cfg.seq, "tokens_per_gpu": cfg.tokens, "t": t,
            "parallelism": f"replicas x{world}"}


def mlp_config(cfg, t: int, world: int, args, n_params: int) -> dict:
    """The MLP run's `config`, identical in both arms."""
    N, H, F = cfg.tokens, cfg.hidden, cfg.ffn
    e = 2 if cfg.dtype == "bf16" else 4
    # activations saved and produced per step (x, y, dy, dx, n, G|U, A, dGU, dN) + parameters,
    # fp32 masters and fp32 gradients
    ws_gb = (N * H * (5 * e + 4) + N * F * (5 * e if cfg.act == "swiglu" else 3 * e) + n_params * (e + 8)) / 1e9
    return dict(workload_config(cfg, t, world), optimizer=args.optimizer, gemm_operands=args.precision,
                sequence_parallel=bool(args.sequence_parallel),
                l2=f"no flush: per-step working set ~{ws_gb:.1f} GB >> 129 MB L2")


def attn_run(args):
    """The attention workload of this run: (config object, t, whether the fused kernels run)."""
    cfg = synth.ATTN_CONFIGS[args.workload]
    if args.tokens:
        cfg = dataclasses.replace(cfg, batch=max(1, args.tokens // cfg.seq))
    t = args.t if cfg.n_kv % args.t == 0 else cfg.t_list[0]
    fused = args.attn_path == "fused" and cfg.d == 128 and cfg.seq % 128 == 0
    return cfg, t, fused


def attn_config(cfg, t: int, world: int, args, fused: bool) -> dict:
    """The attention run's `config`, identical in both arms."""
    return {"workload": f"{cfg.name}: attention sublayer, {cfg.batch}x{cfg.seq} tokens, hidden={cfg.hidden}, "
                        f"{cfg.n_q} query heads in {cfg.n_kv} KV groups, head dim {cfg.d}, causal, t={t} logical shards"
                        + (f", AdamW {ADAMW}" if args.optimizer == "adamw" else f", lr={cfg.lr}"),
            "optimizer": args.optimizer,
            "attention_kernels": "fused (scores never stored)" if fused else "unfused (scores materialised)",
            "global_batch": cfg.batch * world, "seq_len": cfg.seq, "tokens_per_gpu": cfg.tokens, "t": t,
            "parallelism": f"replicas x{world}", "l2": "no flush: per-step working set >> 129 MB L2"}


def metric_name(args, attention: bool) -> str:
    m = METRIC if not attention else "TP-attention fwd+bwd+SGD TFLOP/s at 1 GB300 and % of BF16 dense tensor peak"
    return m.replace("SGD", "AdamW") if args.optimizer == "adamw" else m


def reference_arm(args):
    """The oracle, as it stands, on this run's workload and options, timed on the host cores.

    Each step is the oracle's step for the same options (dense SGD step, the AdamW step, the
    E4M3 step, the sequence-parallel rank decomposition, or the attention sublayer's step) on
    a bounded token sample with the full weights; the sample is halved until warm-up plus timed
    steps fit in about 150 s.  The line carries the same metric and config as this run's GPU
    arm."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import tpmlp_oracle as O
    attention = args.workload in synth.ATTN_CONFIGS
    budget = 150.0  # seconds for warmup + timed steps
    nstep = [0]
    if attention:
        if args.precision != "bf16" or args.sequence_parallel:
            print(json.dumps({"impl": "reference", "unavailable": "the attention sublayer has neither E4M3 "
                                                                  "operands nor a sequence-parallel form"}))
            return 0
        cfg, t, fused = attn_run(args)
        config = attn_config(cfg, t, world, args, fused)
        inp = synth.make_attn_inputs(cfg, seed=1234)
        p = {k: inp[k] for k in ("norm_w", "w_qkv", "w_o", "b_o")}
        mom = {k: np.zeros_like(v) for k, v in p.items()}
        vel = {k: np.zeros_like(v) for k, v in p.items()}
        sample = min(cfg.seq, max(64, args.ref_tokens))

        def step(n):
            # a causal prefix of sequence 0 is a complete smaller problem
            x, tg = inp["x"][:n], inp["target"][:n]
            if args.optimizer == "adamw":
                nstep[0] += 1
                y, c = O.attn_dense_forward(p, x, cfg.eps, 1, cfg.n_q, cfg.n_kv)
                _, dy = O.mse_loss(y, tg)
                g = O.attn_dense_backward(p, c, dy)
                O.adamw(p, {k: g[k] for k in p}, mom, vel, nstep[0], **ADAMW)
            else:
                O.attn_dense_step(p, x, tg, cfg.eps, cfg.lr, 1, cfg.n_q, cfg.n_kv)

        def flops_of(n):
            return dataclasses.replace(cfg, batch=1, seq=n).gemm_flops

        def halve(n):
            return max(16, n // 2)

        what = "tokens of sequence 0 (a causal prefix)"
    else:
        cfg = synth.CONFIGS[args.workload]
        if args.tokens:
            cfg = cfg.with_tokens(args.tokens)
        t = args.t
        options = (args.optimizer == "adamw") + (args.precision == "fp8") + bool(args.sequence_parallel)
        if options > 1:
            print(json.dumps({"impl": "reference", "unavailable": "the oracle has no step combining AdamW, E4M3 "
                                                                  "operands and the sequence-parallel form"}))
            return 0
        # the oracle needs the full weights but only a token sample
        sample = max(16, args.ref_tokens)
        if args.sequence_parallel:
            sample = max(t, sample // t * t)
        inp = synth.make_inputs(cfg.with_tokens(sample), seed=1234)
        p = {k: inp[k] for k in synth.param_names(cfg.act)}
        config = mlp_config(cfg, t, world, args, sum(int(v.size) for v in p.values()))
        mom = {k: np.zeros_like(v) for k, v in p.items()}
        vel = {k: np.zeros_like(v) for k, v in p.items()}

        def step(n):
            x, tg = inp["x"][:n], inp["target"][:n]
            if args.optimizer == "adamw":
                nstep[0] += 1
                O.dense_step_adamw(p, x, tg, cfg.eps, mom, vel, nstep[0], ADAMW, cfg.act)
            elif args.precision == "fp8":
                O.dense_step_fp8(p, x, tg, cfg.eps, cfg.lr, cfg.act, store=synth.round_to_bf16)
            elif args.sequence_parallel:
                O.sp_step(p, x, tg, cfg.eps, cfg.lr, t, cfg.act)
            else:
                O.dense_step(p, x, tg, cfg.eps, cfg.lr, cfg.act)

        def flops_of(n):
            return cfg.gemm_flops * n / cfg.tokens

        def halve(n):
            return max(t, n // 2 // t * t) if args.sequence_parallel else max(1, n // 2)

        what = f"of {cfg.tokens} tokens"
    n = sample
    t0 = time.perf_counter()
    step(n)
    one = time.perf_counter() - t0
    while one * (args.steps + args.warmup) > budget and halve(n) < n:
        n = halve(n)
        t0 = time.perf_counter()
        step(n)
        one = time.perf_counter() - t0
    for _ in range(args.warmup):
        step(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(n)
    el = time.perf_counter() - t0
    val = flops_of(n) * args.steps / el / 1e12
    cores = host_cores()
    line = {
        "impl": "reference", "metric": metric_name(args, attention), "value": val, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} {what} per step, full weights, float64 numpy"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def ours_attn(args):
    """The attention sublayer's training step (tpattn_* + the allocation-free loss) on one GPU."""
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    from tensor_transformer_mlp_rmsnorm_gb300 import TPAttn, build
    from tensor_transformer_mlp_rmsnorm_gb300.tpmlp import tpmlp_mse_loss_grad_noalloc
    build.build()
    cfg, t, fused_only = attn_run(args)
    inp = synth.make_attn_inputs(cfg, seed=1234 + rank)
    names = ("norm_w", "w_qkv", "w_o", "b_o")
    bf = torch.bfloat16
    p = {k: torch.from_numpy(np.ascontiguousarray(inp[k], dtype=np.float32)).to(dev).to(bf) for k in names}
    masters = {k: torch.from_numpy(np.ascontiguousarray(inp[k], dtype=np.float32)).to(dev) for k in names}
    x_host = torch.from_numpy(np.ascontiguousarray(inp["x"], dtype=np.float32)).to(bf).pin_memory()
    tg_host = torch.from_numpy(np.ascontiguousarray(inp["target"], dtype=np.float32)).to(bf).pin_memory()
    cpu_inp = inp if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    del inp
    x, target = x_host.to(dev), tg_host.to(dev)
    # the fused path needs no score square in its workspace
    m = TPAttn(cfg.tokens, cfg.hidden, cfg.n_q, cfg.n_kv, cfg.d, cfg.seq, max_t=t, device=dev, fused_only=fused_only)
    m.bind_master(masters)
    if not fused_only:
        m.set_fused(args.attn_path == "fused")
    y, dy, dx = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    grads = m.new_grads()
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    loss_host = torch.zeros(1, dtype=torch.float32).pin_memory()
    stream = m.stream
    adamw = args.optimizer == "adamw"
    if adamw:
        m.new_adam_state()
    # SGD: backward applies the update (W_qkv and W_o in their gradient GEMMs' epilogues), as for
    # the MLP, unless --separate-update asks for the separate kernel
    fused_update = not adamw and not args.separate_update
    if fused_update:
        m.set_update_in_backward(True, cfg.lr)
    nstep = [0]

    def step(xb=x, tb=target):
        m.forward(xb, p["norm_w"], p["w_qkv"], p["w_o"], p["b_o"], cfg.eps, t, cfg.batch, cfg.seq, y=y)
        tpmlp_mse_loss_grad_noalloc(y, tb, dy, loss, stream=stream.cuda_stream)
        m.backward(dy, dx=dx, grads=grads)
        if adamw:
            nstep[0] += 1
            m.adamw_step(step=nstep[0], **ADAMW)
        elif not fused_update:
            m.sgd_step(cfg.lr)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    m.sync()
    matrices_in_epilogue = fused_update and m.update_in_epilogue()
    fused = m.fused_active()
    if fused != fused_only:
        raise RuntimeError(f"fused attention active={fused}, expected {fused_only}")
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    l0 = m.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    # the loss kernels run outside the context: 2 launches per step
    launches = m.launch_count() - l0 + 2 * args.steps
    ms = e0.elapsed_time(e1)
    barrier()
    time.sleep(0.3)  # the same idle pause as before the device-resident loop
    e2e_steps = max(3, args.steps)
    ems = timed_e2e(torch, step, stream, x_host, tg_host, (x, torch.empty_like(x)),
                    (target, torch.empty_like(target)), loss, loss_host, e2e_steps)
    kms = instrumented_pass(torch, m, step, stream, args.steps)
    ktimes = m.read_kernel_times()
    m.set_timing(False)
    clk = clocks.stop()
    barrier()
    m.sync()
    ms, ems = max_over_ranks(torch, [ms, ems], dev, world)
    flops = cfg.gemm_flops
    value = job_tflops(flops, args.steps, world, ms)
    h2d_rate = h2d_gbps(torch, x_host, y)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    pk, pk_src = peaks()
    N, H, d, S, B, nq, nkv = cfg.tokens, cfg.hidden, cfg.d, cfg.seq, cfg.batch, cfg.n_q, cfg.n_kv
    W = (nq + 2 * nkv) * d
    causal = 2.0 * B * nq * (S * (S + 1) / 2.0) * d  # one attention product over the causal half
    kflops = {"gemm_qkv": 2.0 * N * H * W, "gemm_out_proj": 2.0 * N * nq * d * H, "gemm_dz": 2.0 * N * nq * d * H,
              "gemm_wgrad_out": 2.0 * N * nq * d * H, "gemm_wgrad_qkv": 2.0 * N * H * W,
              "gemm_dgrad_norm": 2.0 * N * H * W, "gemm_scores": causal, "gemm_pv": causal, "gemm_dp": causal,
              "gemm_dv": causal, "gemm_dq": causal, "gemm_dk": causal,
              # fused kernels: the products of the algorithm, not the backward's recomputed scores
              "flash_attn_fwd": 2 * causal, "flash_attn_bwd": 4 * causal}
    top = max(ktimes, key=lambda k: ktimes[k][0])
    per_launch = ktimes[top][0] / max(1, ktimes[top][1])
    # DRAM bytes per launch from a one-launch ncu capture on the current sources (attention GEMMs: none)
    traffic, traffic_src = recorded_traffic(cfg.name, t, N, top) if top.startswith("flash_") else (None, None)
    if top in kflops:
        ach = kflops[top] / (per_launch / 1e3) / 1e12
        peak, kind = choose_peak(pk, clk, (ms + ems + kms) / 1e3)
        roof = {"kernel": top, "bound": "tensor", "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak, "traffic": traffic, "traffic_source": traffic_src,
                "frac_of_burst": ach / pk["bf16_tflops"], "frac_of_sustained": ach / pk["bf16_tflops_sustained"],
                "peak_kind": f"bf16 {kind} ({pk_src})", "avg_launch_ms": per_launch,
                "note": "attention products counted over the causal half of the score square"
                        + ("; the fused backward's score recomputation is not counted" if top == "flash_attn_bwd"
                           else "")}
    else:
        # causal rows: read up to the diagonal, written up to the end of the diagonal's 256-column block
        tri = B * nq * (S * (S + 1) / 2.0)
        pad = B * nq * S * 128.0  # mean zero tail written past the diagonal
        nbytes = {"softmax_fwd": 4.0 * tri + 2.0 * (tri + pad), "softmax_bwd": 6.0 * tri + 2.0 * (tri + pad),
                  "flash_bwd_prep": N * nq * d * (2.0 + 2.0 + 4.0) + 4.0 * N * nq,
                  "flash_dq_cast": N * nq * d * (4.0 + 2.0)}.get(top)
        ach = nbytes / (per_launch / 1e3) / 1e9 if nbytes else None
        roof = {"kernel": top, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": ach / pk["hbm_gbs"] if ach else None, "traffic": traffic, "traffic_source": traffic_src,
                "avg_launch_ms": per_launch}
    gemm_ms = sum(v[0] for k, v in ktimes.items() if k in kflops)
    cpu = None
    if cpu_inp is not None:
        v, n, dt = cpu_attn_oracle_tflops(cfg, cpu_inp, budget_s=args.cpu_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"dense fwd+loss+bwd+SGD of the first {n} tokens of sequence 0 (a causal prefix) "
                         f"with the full weights, float64 numpy, {dt:.1f} s"}
    line = {
        "metric": metric_name(args, True),
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": attn_config(cfg, t, world, args, fused),
        "pct_of_bf16_peak": {"of_burst": 100.0 * value / world / pk["bf16_tflops"],
                             "of_sustained": 100.0 * value / world / pk["bf16_tflops_sustained"], "source": pk_src},
        "gemm_only_tflops": flops * args.steps / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None,
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in sorted(ktimes.items(), key=lambda kv: -kv[1][0])},
        "instrumented_ms_per_step": kms / args.steps,
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": job_tflops(flops, e2e_steps, world, ems), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * N * H * 2, "d2h_bytes_per_step": 4, "steps": e2e_steps,
                "h2d": "pinned host -> device on a copy stream, double-buffered (step i+1's copy overlaps step i)",
                "h2d_gbps_alone": h2d_rate},
        "clocks": clk, "gpu_launches": launches, "loss": float(loss_host.item()),
        "update": update_placement(adamw, fused_update, matrices_in_epilogue),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    from tensor_transformer_mlp_rmsnorm_gb300 import TPMLP, build
    build.build()
    cfg = synth.CONFIGS[args.workload]
    if args.tokens:
        cfg = cfg.with_tokens(args.tokens)
    N, H, F = cfg.tokens, cfg.hidden, cfg.ffn
    t = args.t
    inp = synth.make_inputs(cfg, seed=1234 + rank)
    bf = torch.bfloat16

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(bf)

    # the library names the first projection w_gate_up for both activations
    lib_name = {"w_1": "w_gate_up"}
    params = {lib_name.get(k, k): dev_bf16(inp[k]) for k in synth.param_names(cfg.act)}
    masters = {lib_name.get(k, k): torch.from_numpy(np.ascontiguousarray(inp[k], dtype=np.float32)).to(dev)
               for k in synth.param_names(cfg.act)}
    x_host = torch.from_numpy(np.ascontiguousarray(inp["x"], dtype=np.float32)).to(bf).pin_memory()
    tg_host = torch.from_numpy(np.ascontiguousarray(inp["target"], dtype=np.float32)).to(bf).pin_memory()
    cpu_inp = inp if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    del inp
    x = x_host.to(dev)
    target = tg_host.to(dev)
    m = TPMLP(N, H, F, max_t=max(8, t), dtype=cfg.dtype, act=cfg.act, device=dev)
    m.bind_master(masters)
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    dx = torch.empty_like(x)
    grads = m.new_grads()
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    loss_host = torch.zeros(1, dtype=torch.float32).pin_memory()

    if args.sequence_parallel:
        m.set_sequence_parallel(True)
    if args.precision == "fp8":
        m.set_precision("fp8")
    adamw = args.optimizer == "adamw"
    if adamw:
        m.new_adam_state()
    # SGD: backward applies the update to the weight matrices where their gradients are produced
    # (bit-identical to a separate sgd_step), unless --separate-update asks for the separate kernel
    fused_update = not adamw and not args.separate_update
    if fused_update:
        m.set_update_in_backward(True, cfg.lr)
    nstep = [0]

    def step(xb=x, tb=target):
        m.forward(xb, params["norm_w"], params["w_gate_up"], params["w_down"], params["b_down"], cfg.eps, t, y=y,
                  b_1=params.get("b_1"))
        m.mse_loss_grad(y, tb, dy=dy, loss=loss)
        m.backward(dy, dx=dx, grads=grads)
        if adamw:
            nstep[0] += 1
            m.adamw_step(step=nstep[0], **ADAMW)
        elif not fused_update:
            m.sgd_step(cfg.lr)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    m.sync()
    matrices_in_epilogue = fused_update and m.update_in_epilogue()
    stream = m.stream
    # ---------------------------------------------------------- device-resident timing
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = m.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = m.launch_count() - launches0
    ms = e0.elapsed_time(e1)
    # ---------------------------------------------------------- end-to-end through the public API
    # The same number of steps, started like the device-resident loop: after the same idle pause,
    # so that both begin at the same point of the power cap's averaging window.
    barrier()
    time.sleep(0.3)
    e2e_steps = max(3, args.steps)
    ems = timed_e2e(torch, step, stream, x_host, tg_host, (x, torch.empty_like(x)),
                    (target, torch.empty_like(target)), loss, loss_host, e2e_steps)
    # Per-kernel times come from a third pass of the same steps with the library's CUDA events
    # around every launch (on its stream), so that the headline loops run uninstrumented.
    kms = instrumented_pass(torch, m, step, stream, args.steps)
    ktimes = m.read_kernel_times()
    m.set_timing(False)
    clk = clocks.stop()
    barrier()
    m.sync()
    ms, ems = max_over_ranks(torch, [ms, ems], dev, world)
    flops_step = cfg.gemm_flops
    e = 2 if cfg.dtype == "bf16" else 4
    nP = sum(v.numel() for v in params.values())
    value = job_tflops(flops_step, args.steps, world, ms)
    e2e_value = job_tflops(flops_step, e2e_steps, world, ems)
    h2d_rate = h2d_gbps(torch, x_host, y)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    pk, pk_src = peaks()
    # dominant kernel and its roofline
    ktot = {k: v[0] for k, v in ktimes.items()}
    top = max(ktot, key=ktot.get)
    top_ms, top_n = ktimes[top]
    per_launch_ms = top_ms / max(1, top_n)
    units = GEMM_UNITS if cfg.act == "swiglu" else GELU_UNITS
    gemm_ms = sum(ktimes[k][0] for k in ktimes if k in units)
    traffic, traffic_src = recorded_traffic(cfg.name, t, N, top, args.precision)
    # E4M3 operands: the measured bf16 peaks times the nominal dense ratio 4.5 / 2.25
    ratio, pname = (2.0, "e4m3 = 2 x measured bf16") if args.precision == "fp8" else (1.0, "bf16")
    if top in units:
        achieved = units[top] * N * H * F / (per_launch_ms / 1e3) / 1e12
        peak_s, peak_b = ratio * pk["bf16_tflops_sustained"], ratio * pk["bf16_tflops"]
        peak, kind = choose_peak(pk, clk, (ms + ems + kms) / 1e3, ratio)
        roof = {"kernel": top, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": f"{pname} {kind} ({pk_src}): " + (
                    "timed region under 1 s at the maximum SM clock" if kind == "burst"
                    else "timed region long enough for the power cap, or SM clock below its maximum"),
                "frac_of_burst": achieved / peak_b, "frac_of_sustained": achieved / peak_s, "traffic": traffic,
                "flops_per_launch": units[top] * N * H * F, "avg_launch_ms": per_launch_ms}
    else:
        nbytes = hbm_bytes(top, cfg, masters=True, update_in_backward=matrices_in_epilogue)
        achieved = nbytes / (per_launch_ms / 1e3) / 1e9 if nbytes else None
        roof = {"kernel": top, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"] if achieved else None, "peak_kind": f"hbm_gbs ({pk_src})",
                "traffic": traffic, "bytes_per_launch": nbytes, "avg_launch_ms": per_launch_ms}
    roof["traffic_source"] = traffic_src if traffic is not None else \
        "null: no ncu DRAM record for this workload on the current kernel sources"
    # every kernel against its own roofline: GEMMs' algorithmic flops against the bf16 peak the
    # dominant kernel uses, memory-bound kernels' algorithmic bytes against the measured copy rate
    tpeak, _ = choose_peak(pk, clk, (ms + ems + kms) / 1e3, ratio)
    kfrac = {}
    for kname, (kms_tot, kn) in ktimes.items():
        per = kms_tot / max(1, kn) / 1e3
        if kname in units:
            kfrac[kname] = units[kname] * N * H * F / per / 1e12 / tpeak
        else:
            nb = hbm_bytes(kname, cfg, masters=True, update_in_backward=matrices_in_epilogue)
            if nb:
                kfrac[kname] = nb / per / 1e9 / pk["hbm_gbs"]
    cpu = None
    if cpu_inp is not None:
        v, n, dt = cpu_oracle_tflops(cfg, cpu_inp, budget_s=args.cpu_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"dense fwd+loss+bwd+SGD of the first {n} of {N} tokens with the full weights, "
                         f"float64 numpy, {dt:.1f} s"}
    metric = metric_name(args, False)
    line = {
        "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if args.precision == "fp8" else cfg.dtype,
        "data": "synthetic",
        "config": mlp_config(cfg, t, world, args, nP),
        "pct_of_bf16_peak": {"of_burst": 100.0 * value / world / pk["bf16_tflops"],
                             "of_sustained": 100.0 * value / world / pk["bf16_tflops_sustained"],
                             "source": pk_src},
        "gemm_only_tflops": flops_step * args.steps / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None,
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in sorted(ktimes.items(), key=lambda kv: -kv[1][0])},
        "instrumented_ms_per_step": kms / args.steps,
        "kernel_frac_of_roofline": {k: round(v, 3) for k, v in sorted(kfrac.items(), key=lambda kv: -kv[1])},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 2 * N * H * e,
                "d2h_bytes_per_step": 4, "steps": e2e_steps,
                "h2d": "pinned host -> device on a copy stream, double-buffered (step i+1's copy overlaps step i)",
                "h2d_gbps_alone": h2d_rate},
        "clocks": clk,
        "gpu_launches": launches,
        "loss": float(loss_host.item()),
        "update": update_placement(adamw, fused_update, matrices_in_epilogue),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.CONFIGS) + sorted(synth.ATTN_CONFIGS))
    ap.add_argument("--t", type=int, default=T_SHARDS)
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--optimizer", choices=["sgd", "adamw"], default="sgd")
    ap.add_argument("--precision", choices=["bf16", "fp8"], default="bf16",
                    help="GEMM operands: bf16, or E4M3 with per-tensor scales (fp32 accumulation either way)")
    ap.add_argument("--sequence-parallel", action="store_true",
                    help="sequence-parallel form: per-shard norm-weight / bias gradients, then their sum")
    ap.add_argument("--attn-path", choices=["fused", "unfused"], default="fused",
                    help="attention workloads: fused kernels (scores never stored) or materialised scores")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--separate-update", action="store_true",
                    help="SGD: run the update as its own kernel after backward instead of in backward")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    if args.workload in synth.ATTN_CONFIGS:
        return ours_attn(args)
    return ours(args)


if __name__ == "__main__":
    sys.exit(main())
