"""Multi-process host logic on CPU ranks (gloo, world sizes 2 and 4).

* Context parallelism (LaCT page, "Large Chunk Test-Time Training", §2.2.2):
  each rank computes the gradient of its shard of a chunk's tokens with the
  same fast weights; the all-reduced sum equals the gradient of the whole chunk
  (the chunk gradient is a sum over tokens, §2.1), so every rank can then run
  the same Newton-Schulz step and update.
* The context-parallel driver (long_seq_models_chunked_b300.cp: one rank's chunk
  loop, an all-reduce at every update) over two and four gloo ranks, with each rank's
  steps computed by the fp64 oracle, equals the unsharded layer.
* The benchmark's N-GPU reduction helpers (max of the per-rank step time, sum
  of the tokens) give the whole-job figures.
* A rank that never reaches a collective makes the others fail with a
  process-group timeout instead of hanging.
"""
import multiprocessing as mp
import os
import socket
import traceback

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s=30.0):
    import datetime

    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))
    return dist


def _sharded_grad_worker(rank, world, port, q):
    try:
        import sys
        sys.path.insert(0, ROOT)
        import torch

        from long_seq_models_chunked_b300 import synth
        from oracle import OracleCfg, chunk_grad
        dist = _init(rank, world, port)
        spec = synth.LayerSpec("cp", B=1, H=1, T=96, d=8, dh=16, chunk=96, dtype="fp32", muon=True, seed=7)
        ht = synth.head_tokens(spec, 0, 0)
        W = [w[0].astype(np.float64) for w in synth.initial_weights(spec)]
        cfg = OracleCfg.from_spec(spec)
        # uneven shards: rank 0 gets 40 tokens, rank 1 the other 56
        cut = [0, 40, 96]
        s, e = cut[rank], cut[rank + 1]
        g = chunk_grad(cfg, W, ht["K64"][s:e], ht["V64"][s:e], ht["lr"][s:e].astype(np.float64))
        out = []
        for gj in g:
            t = torch.from_numpy(np.ascontiguousarray(gj))
            dist.all_reduce(t)
            out.append(t.numpy())
        full = chunk_grad(cfg, W, ht["K64"], ht["V64"], ht["lr"].astype(np.float64))
        err = max(float(np.abs(a - b).max() / np.abs(b).max()) for a, b in zip(out, full))
        dist.destroy_process_group()
        q.put((rank, "ok", err))
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


class _OracleShard:
    """One rank's state for the context-parallel driver, computed by the oracle
    (fp64, one head): the gradient is passed around flattened."""

    def __init__(self, cfg, W):
        from oracle import row_norms
        self.cfg = cfg
        self.W = tuple(W)
        self.n0 = [row_norms(w) for w in W]
        self.mom = [np.zeros_like(w) for w in W] if cfg.momentum else None

    def grad(self, K, V, lr, s, n):
        import torch

        from oracle import chunk_grad
        g = chunk_grad(self.cfg, self.W, K[s:s + n], V[s:s + n], lr[s:s + n])
        return torch.from_numpy(np.concatenate([x.ravel() for x in g]))

    def update(self, G):
        from oracle import update
        flat = G.numpy()
        parts, o = [], 0
        for w in self.W:
            parts.append(flat[o:o + w.size].reshape(w.shape))
            o += w.size
        self.W = update(self.cfg, self.W, parts, self.n0, self.mom)

    def apply(self, Q, O, s, n):
        from oracle import swiglu_apply
        O[s:s + n] = swiglu_apply(self.W, Q[s:s + n])


def _cp_driver_worker(rank, world, port, q):
    try:
        import sys
        sys.path.insert(0, ROOT)
        from long_seq_models_chunked_b300 import cp, synth
        from oracle import OracleCfg, ttt_head
        dist = _init(rank, world, port)
        spec = synth.LayerSpec("cp_drv", B=1, H=1, T=96, d=8, dh=16, chunk=32, dtype="fp32", muon=True,
                               update="odd", momentum=0.5, seed=9)
        ht = synth.head_tokens(spec, 0, 0)
        W0 = [w[0].astype(np.float64) for w in synth.initial_weights(spec)]
        cfg = OracleCfg.from_spec(spec)
        C, Cl = spec.chunk, spec.chunk // world
        mine = np.concatenate([np.arange(c + rank * Cl, c + (rank + 1) * Cl) for c in range(0, spec.T, C)])
        Q, K, V = (ht[n][mine] for n in ("Q64", "K64", "V64"))
        lr = ht["lr"][mine].astype(np.float64)
        O = np.zeros((mine.size, spec.d))
        shard = _OracleShard(cfg, W0)
        steps = cp.rank_steps(shard, Q, K, V, lr, O, mine.size, Cl, True, spec.update_mask())
        cp.run_rank(steps, lambda G: dist.all_reduce(G))
        O_ref, W_ref = ttt_head(cfg, ht["Q64"], ht["K64"], ht["V64"], ht["lr"], W0)
        err = max([float(np.abs(O - O_ref[mine]).max() / np.abs(O_ref).max())] +
                  [float(np.abs(a - b).max() / np.abs(b).max()) for a, b in zip(shard.W, W_ref)])
        dist.destroy_process_group()
        q.put((rank, "ok", err))
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


def _bench_reduce_worker(rank, world, port, q):
    try:
        import sys
        sys.path.insert(0, ROOT)
        import bench
        dist = _init(rank, world, port)
        t_max = bench.max_over_ranks(dist, [3.5, 2.0][rank])
        tok = bench.sum_over_ranks(dist, float([65536, 65536][rank]))
        bench.barrier(dist)
        dist.destroy_process_group()
        q.put((rank, "ok", (t_max, tok)))
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


def _absent_rank_worker(rank, world, port, q):
    try:
        import torch
        dist = _init(rank, world, port, timeout_s=3.0)
        if rank == 1:
            # leaves between steps: joins the group, then never enters the collective
            q.put((rank, "ok", "left"))
            return
        t = torch.ones(4)
        try:
            dist.all_reduce(t)
            q.put((rank, "ok", "no error"))
        except Exception as e:  # the timeout surfaces as an exception on the host
            q.put((rank, "ok", "timeout:" + type(e).__name__))
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


def _run(worker, world=2, timeout=120):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = {}
    for _ in range(world):
        r, status, val = q.get(timeout=timeout)
        assert status == "ok", val
        res[r] = val
    for p in ps:
        p.join(timeout=30)
        if p.is_alive():
            p.kill()
    return res


def test_context_parallel_gradient_sum_equals_whole_chunk():
    res = _run(_sharded_grad_worker)
    assert all(v <= 1e-12 for v in res.values()), res


@pytest.mark.parametrize("world", [2, 4])
def test_context_parallel_driver_equals_unsharded_layer(world):
    res = _run(_cp_driver_worker, world=world)
    assert len(res) == world and all(v <= 1e-10 for v in res.values()), res


def test_bench_reductions_over_ranks():
    res = _run(_bench_reduce_worker)
    for r in (0, 1):
        assert res[r] == (3.5, 131072.0), res


def test_absent_rank_times_out_on_the_host():
    res = _run(_absent_rank_worker)
    assert res[1] == "left"
    assert res[0].startswith("timeout:"), res
