"""The page's own setup, on CPU: two gloo ranks, each holding one FFN shard,
with real all-reduces where the f and g operators put them ("Split the
contraction", "Put the other collective in backward").  Each rank runs the
oracle's rank-local functions; the collective sums come from torch.distributed.
The result must equal the dense block, and each removed collective must break
exactly what "Remove each collective" says.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _fixture():
    rng = np.random.default_rng(1234)
    N, H, F = 6, 8, 12
    p = {"norm_w": 1.0 + 0.1 * rng.standard_normal(H),
         "w_gate_up": 0.3 * rng.standard_normal((2, F, H)),
         "w_down": 0.3 * rng.standard_normal((H, F)),
         "b_down": 0.05 * rng.standard_normal(H)}
    return p, rng.standard_normal((N, H)), rng.standard_normal((N, H))


def _all_reduce(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.numpy()


def _rank_main(rank, world, port, mode, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import tpmlp_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p, x, tgt = _fixture()
        eps, lr = 1e-6, 0.1
        q = O.local_params(p, world, rank, "swiglu")
        partial, c = O.rank_forward(q, x, eps, "swiglu")
        mlp_out = partial if mode == "missing_forward_reduce" else _all_reduce(partial)
        y = x + mlp_out + p["b_down"]
        loss, dy = O.mse_loss(y, tgt)
        g, dn_local = O.rank_backward_local(q, c, dy)
        dn = dn_local if mode == "missing_backward_reduce" else _all_reduce(dn_local)
        dxn, g["norm_w"] = O.rms_norm_backward(dn, c["xhat"], c["rstd"], p["norm_w"])
        g["x"] = dy + dxn
        newq = {k: q[k] - lr * g[k] for k in q}
        np.savez(os.path.join(out_dir, f"r{rank}.npz"), y=y, loss=loss, dx=g["x"], dnorm_w=g["norm_w"],
                 dwgu=g["w_gate_up"], dwd=g["w_down"], dbd=g["b_down"], new_norm_w=newq["norm_w"],
                 new_wgu=newq["w_gate_up"], new_wd=newq["w_down"])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["equivalence", "missing_forward_reduce", "missing_backward_reduce"])
def test_two_gloo_ranks(tmp_path, mode):
    from oracle import tpmlp_oracle as O
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), mode, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    p, x, tgt = _fixture()
    d = O.dense_step(p, x, tgt, 1e-6, 0.1)
    s = O.sharded_step(p, x, tgt, 1e-6, 0.1, world,
                       skip_forward_reduce=(mode == "missing_forward_reduce"),
                       skip_backward_reduce=(mode == "missing_backward_reduce"))
    F = p["w_down"].shape[1]
    for r in range(world):
        z = np.load(tmp_path / f"r{r}.npz")
        lo, hi = O.shard_interval(F, world, r)
        # the real-collective ranks agree with the oracle's in-process decomposition
        rk = s["ranks"][r]
        np.testing.assert_allclose(z["y"], rk["y"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(z["dx"], rk["grads"]["x"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(z["dwgu"], rk["grads"]["w_gate_up"], rtol=0, atol=1e-15)
        dense_close = lambda a, b: float(np.max(np.abs(a - b))) < 1e-12
        fwd_ok = dense_close(z["y"], d["y"])
        dx_ok = dense_close(z["dx"], d["grads"]["x"])
        dnw_ok = dense_close(z["dnorm_w"], d["grads"]["norm_w"])
        dwgu_ok = dense_close(z["dwgu"], d["grads"]["w_gate_up"][:, lo:hi])
        dwd_ok = dense_close(z["dwd"], d["grads"]["w_down"][:, lo:hi])
        if mode == "equivalence":
            assert fwd_ok and dx_ok and dnw_ok and dwgu_ok and dwd_ok
            assert dense_close(z["dbd"], d["grads"]["b_down"])
            assert dense_close(z["new_wd"], d["new_params"]["w_down"][:, lo:hi])
        elif mode == "missing_forward_reduce":
            assert not fwd_ok and not dx_ok and not dnw_ok and not dwgu_ok and not dwd_ok
        else:
            assert fwd_ok and dwgu_ok and dwd_ok
            assert not dx_ok and not dnw_ok
            assert not dense_close(z["new_norm_w"], d["new_params"]["norm_w"])


def _adamw_rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import tpmlp_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p, x, tgt = _fixture()
        eps = 1e-6
        q = O.local_params(p, world, rank, "swiglu")
        partial, c = O.rank_forward(q, x, eps, "swiglu")
        y = x + _all_reduce(partial) + p["b_down"]
        loss, dy = O.mse_loss(y, tgt)
        g, dn_local = O.rank_backward_local(q, c, dy)
        _, g["norm_w"] = O.rms_norm_backward(_all_reduce(dn_local), c["xhat"], c["rstd"], p["norm_w"])
        # the global norm: each rank's squared share (replicated grads on rank 0 only), all-reduced
        sq = _all_reduce(np.array([O.rank_grad_sqnorm(g, rank)]))[0]
        norm = float(np.sqrt(sq))
        hp = dict(O.ADAMW_DEFAULTS, lr=0.01, max_grad_norm=0.5 * norm)
        clip = O.clip_coefficient(norm, hp["max_grad_norm"])
        z = {k: np.zeros_like(q[k]) for k in q}
        # each rank updates its own slices with the shared clip factor (clipping off inside)
        out = O.adamw(q, {k: clip * g[k] for k in q}, z, dict(z), 1, **dict(hp, max_grad_norm=0.0))
        np.savez(os.path.join(out_dir, f"a{rank}.npz"), norm=norm, wgu=out["params"]["w_gate_up"],
                 wd=out["params"]["w_down"], nw=out["params"]["norm_w"], bd=out["params"]["b_down"])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_adamw(tmp_path):
    """The walkthrough's clipped AdamW step across two ranks ("Stage 8"): the
    norm all-reduce over the ranks' shares equals the dense norm, and the
    rank-local updates assemble to the dense update."""
    from oracle import tpmlp_oracle as O
    world = 2
    mp.start_processes(_adamw_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    p, x, tgt = _fixture()
    d = O.dense_step(p, x, tgt, 1e-6, 0.0)
    g = {k: d["grads"][k] for k in p}
    norm = O.global_grad_norm(g)
    hp = dict(O.ADAMW_DEFAULTS, lr=0.01, max_grad_norm=0.5 * norm)
    z = {k: np.zeros_like(p[k]) for k in p}
    ref = O.adamw(p, g, z, dict(z), 1, **hp)
    assert ref["clip"] < 1.0
    F = p["w_down"].shape[1]
    for r in range(world):
        a = np.load(tmp_path / f"a{r}.npz")
        lo, hi = O.shard_interval(F, world, r)
        assert float(a["norm"]) == pytest.approx(norm, rel=1e-13)
        np.testing.assert_allclose(a["wgu"], ref["params"]["w_gate_up"][:, lo:hi], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(a["wd"], ref["params"]["w_down"][:, lo:hi], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(a["nw"], ref["params"]["norm_w"], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(a["bd"], ref["params"]["b_down"], rtol=1e-12, atol=1e-15)


def _sp_rank_main(rank, world, port, skip_sync, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import tpmlp_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p, x, tgt = _fixture()
        N, H = x.shape
        eps, lr = 1e-6, 0.1
        lo, hi = O.token_interval(N, world, rank)
        q = O.local_params(p, world, rank, "swiglu")

        def all_gather(a):
            parts = [torch.zeros_like(torch.from_numpy(a)) for _ in range(world)]
            dist.all_gather(parts, torch.from_numpy(np.ascontiguousarray(a)))
            return torch.cat(parts).numpy()

        def reduce_scatter(a):
            out = torch.zeros((a.shape[0] // world,) + a.shape[1:], dtype=torch.float64)
            dist.reduce_scatter_tensor(out, torch.from_numpy(np.ascontiguousarray(a)))
            return out.numpy()

        n_loc, rstd, xhat = O.rms_norm(x[lo:hi], p["norm_w"], eps)
        partial, c = O.rank_forward_normed(q, all_gather(n_loc), "swiglu")
        y = x[lo:hi] + reduce_scatter(partial) + p["b_down"]
        dy = (y - tgt[lo:hi]) / (N * H)
        g, dn_local = O.rank_backward_local(q, c, all_gather(dy))
        dxn, dnw = O.rms_norm_backward(reduce_scatter(dn_local), xhat, rstd, p["norm_w"])
        dbd = np.sum(dy, axis=0)
        if not skip_sync:
            dnw, dbd = _all_reduce(dnw), _all_reduce(dbd)
        np.savez(os.path.join(out_dir, f"sp{rank}.npz"), y=y, dx=dy + dxn, dnw=dnw, dbd=dbd,
                 dwgu=g["w_gate_up"], dwd=g["w_down"])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("skip_sync", [False, True])
def test_two_gloo_ranks_sequence_parallel(tmp_path, skip_sync):
    """The sequence-parallel form with real all-gather / reduce-scatter / all-reduce
    calls on two ranks ("Deep dive: sequence parallelism"): each rank's slices
    equal the oracle's in-process decomposition and the dense block; without
    the norm-gradient all-reduce, only dnorm_w and db_down change."""
    from oracle import tpmlp_oracle as O
    world = 2
    mp.start_processes(_sp_rank_main, args=(world, _free_port(), skip_sync, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    p, x, tgt = _fixture()
    d = O.dense_step(p, x, tgt, 1e-6, 0.1)
    F = p["w_down"].shape[1]
    for r in range(world):
        z = np.load(tmp_path / f"sp{r}.npz")
        s = O.sp_step(p, x, tgt, 1e-6, 0.1, world, skip_sp_grad_sync=skip_sync, view_rank=r)
        lo, hi = O.token_interval(x.shape[0], world, r)
        flo, fhi = O.shard_interval(F, world, r)
        close = lambda a, b: np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
        close(z["y"], d["y"][lo:hi])
        close(z["dx"], d["grads"]["x"][lo:hi])
        close(z["dwgu"], d["grads"]["w_gate_up"][:, flo:fhi])
        close(z["dwd"], d["grads"]["w_down"][:, flo:fhi])
        close(z["dnw"], s["grads"]["norm_w"])
        close(z["dbd"], s["grads"]["b_down"])
        synced = np.allclose(z["dnw"], d["grads"]["norm_w"], rtol=1e-12, atol=1e-15)
        assert synced == (not skip_sync)


# --------------------------------------------------------------------------
# The attention sublayer with real collectives: each rank owns complete KV
# groups and their query heads (W_qkv split by heads, W_out by columns); the
# partial outputs and the normed input's partial gradients are all-reduced.

_AB, _AS, _AH, _ANQ, _ANKV, _AD = 2, 8, 16, 4, 2, 4


def _attn_fixture():
    rng = np.random.default_rng(4321)
    W = (_ANQ + 2 * _ANKV) * _AD
    p = {"norm_w": 1.0 + 0.1 * rng.standard_normal(_AH), "w_qkv": 0.4 * rng.standard_normal((W, _AH)),
         "w_o": 0.3 * rng.standard_normal((_AH, _ANQ * _AD)), "b_o": 0.05 * rng.standard_normal(_AH)}
    N = _AB * _AS
    return p, rng.standard_normal((N, _AH)), rng.standard_normal((N, _AH))


def _attn_rank_main(rank, world, port, mode, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import tpmlp_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p, x, tgt = _attn_fixture()
        eps = 1e-6
        nq, nkv = _ANQ // world, _ANKV // world
        q = O.attn_local_params(p, world, rank, _ANQ, _ANKV)
        n, rstd, xhat = O.rms_norm(x, p["norm_w"], eps)
        wq, wk, wv, d = O.attn_split_heads(q, nq, nkv)
        qq, kk, vv = O.linear(n, wq), O.linear(n, wk), O.linear(n, wv)
        z, P = O.attention_heads(qq, kk, vv, _AB, nq, nkv, d)
        y = x + _all_reduce(O.linear(z, q["w_o"])) + p["b_o"]
        loss, dy = O.mse_loss(y, tgt)
        c = {"n": n, "rstd": rstd, "xhat": xhat, "q": qq, "k": kk, "v": vv, "z": z, "P": P, "d": d,
             "batch": _AB, "n_q": nq, "n_kv": nkv}
        dq, dk, dv = O.attention_heads_backward(c, dy @ q["w_o"])
        dqkv = np.concatenate([dq, dk, dv], axis=1)
        dn_local = dqkv @ q["w_qkv"]
        dn = dn_local if mode == "missing_backward_reduce" else _all_reduce(dn_local)
        dxn, dnw = O.rms_norm_backward(dn, xhat, rstd, p["norm_w"])
        np.savez(os.path.join(out_dir, f"t{rank}.npz"), y=y, dx=dy + dxn, dnorm_w=dnw, dwqkv=dqkv.T @ n,
                 dwo=dy.T @ z)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["equivalence", "missing_backward_reduce"])
def test_two_gloo_ranks_attention(tmp_path, mode):
    from oracle import tpmlp_oracle as O
    world = 2
    mp.start_processes(_attn_rank_main, args=(world, _free_port(), mode, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    p, x, tgt = _attn_fixture()
    dense = O.attn_dense_step(p, x, tgt, 1e-6, 0.0, _AB, _ANQ, _ANKV)
    g = dense["grads"]
    close = lambda a, b: float(np.max(np.abs(a - b))) < 1e-12
    gq, gk, d = _ANQ // world, _ANKV // world, _AD
    for r in range(world):
        z = np.load(tmp_path / f"t{r}.npz")
        sq = slice(r * gq * d, (r + 1) * gq * d)
        sk = slice(r * gk * d, (r + 1) * gk * d)
        dense_rows = np.concatenate([g["w_qkv"][: _ANQ * d][sq], g["w_qkv"][_ANQ * d: (_ANQ + _ANKV) * d][sk],
                                     g["w_qkv"][(_ANQ + _ANKV) * d:][sk]], axis=0)
        # the forward, and the weight gradients of the rank's own heads, need no backward reduction
        assert close(z["y"], dense["y"])
        assert close(z["dwqkv"], dense_rows)
        assert close(z["dwo"], g["w_o"][:, sq])
        if mode == "equivalence":
            assert close(z["dx"], g["x"]) and close(z["dnorm_w"], g["norm_w"])
        else:
            assert not close(z["dx"], g["x"]) and not close(z["dnorm_w"], g["norm_w"])
