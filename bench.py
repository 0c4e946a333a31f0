"""Throughput benchmark of the chunked TTT fast-weight layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one ttt_fwd call over the whole workload: every chunk's apply and
update (LaCT page, "Large Chunk Test-Time Training", §2.1), inputs resident in
device memory. The default workload is the large-chunk language-model layer
(B=2, H=3, d=512, dh=1024, T=32768, chunk=2048, Muon + weight norm, bf16
operands and fp32 state). Rank 0 prints one JSON line.

  value      tokens/s = B*T (all ranks) / device time per step (max over ranks);
             L2 is flushed (a 256 MiB write) before every timed step
  e2e        the same metric through ttt_fwd_host: pinned host inputs copied in,
             the layer, outputs copied back, every step
  roofline   the kernel class with the largest share of device time: its
             algorithmic FLOP (or bytes) per launch / its mean launch time, from
             CUDA events recorded around every launch on the launch stream
  cpu_baseline  the fp64 oracle on the host cores over a bounded sample

--impl reference times the fp64 CPU oracle (the only other implementation of
the method) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TTT-layer tokens/sec (update+apply, 1 B300) and % of bf16 tensor-core peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.02)   # the first sample marks the sampler as running
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}: launch N>1 with torch.distributed.run")
    pg = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if _cuda() else "gloo")
        pg = dist
    return rank, local, world, pg


def _cuda() -> bool:
    import torch
    return torch.cuda.is_available()


def barrier(pg, dev=None):
    import torch
    if pg is not None:
        if dev is not None:
            pg.barrier(device_ids=[dev.index])
        else:
            pg.barrier()
    if dev is not None:
        torch.cuda.synchronize(dev)


def max_over_ranks(pg, x: float, dev=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev if dev is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float, dev=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev if dev is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ accounting
def kernel_flops_per_launch(spec, kind: int, launches: int) -> float:
    """Algorithmic FLOP of one step that a kernel class carries, per launch.

    Per (b, h) head and chunk of C tokens (d, dh as in the spec):
      fwd    (shifted) queries: [A|B] 4 d dh C; keys (updated chunks): [A|B] 4 d dh C + Dm 2 d dh C
      apply  O = H W2^T: 2 d dh C
      grad   G1, G2, G3: 6 d dh C (updated chunks)
      gram / xupd  2 m^2 n per matrix and iteration; poly  2 m^3
      ns (fused)   3 matrices x iters x (4 m^2 n + 2 m^3) per update
    """
    from long_seq_models_chunked_b300 import abi
    heads = spec.B * spec.H
    mask = spec.update_mask()
    T = spec.T
    upd_tok = sum(min(T, (c + 1) * spec.chunk) - c * spec.chunk for c in range(spec.n_chunks) if mask[c])
    n_upd = int(mask.sum())
    d, dh = spec.d, spec.dh
    m, n = min(d, dh), max(d, dh)
    tot = {
        abi.TTT_KERNEL_FWD: heads * (4.0 * d * dh * T + 6.0 * d * dh * upd_tok),
        abi.TTT_KERNEL_APPLY: heads * 2.0 * d * dh * T,
        abi.TTT_KERNEL_GRAD: heads * 6.0 * d * dh * upd_tok,
        abi.TTT_KERNEL_GRAM: heads * n_upd * 3 * spec.ns_iters * 2.0 * m * m * n if spec.muon else 0.0,
        abi.TTT_KERNEL_POLY: heads * n_upd * 3 * spec.ns_iters * 2.0 * m ** 3 if spec.muon else 0.0,
        abi.TTT_KERNEL_XUPD: heads * n_upd * 3 * spec.ns_iters * 2.0 * m * m * n if spec.muon else 0.0,
        abi.TTT_KERNEL_NS: heads * n_upd * 3 * spec.ns_iters * (4.0 * m * m * n + 2.0 * m ** 3) if spec.muon else 0.0,
    }
    if spec.fast_net == "linear":
        tot = {abi.TTT_KERNEL_LINEAR: heads * (2.0 * d * d * T + 4.0 * d * d * upd_tok),
               abi.TTT_KERNEL_SIMT: heads * (2.0 * d * d * T + 4.0 * d * d * upd_tok)}
    f = tot.get(kind)
    if f is None or launches <= 0:
        return None
    return f / launches


def executed_mma_flops(spec) -> float:
    """FLOP the tensor-core path actually issues per step in its default split
    precision: products with one exact bf16 input (queries, keys, values) run
    twice (W = hi + lo, E = hi + lo), products of two computed operands
    (Newton-Schulz) three times; the queries' forward and the apply run once.
    Context for the algorithmic figure, which counts every product once."""
    if spec.fast_net != "swiglu":
        return None
    heads = spec.B * spec.H
    mask = spec.update_mask()
    upd_tok = sum(min(spec.T, (c + 1) * spec.chunk) - c * spec.chunk for c in range(spec.n_chunks) if mask[c])
    n_upd = int(mask.sum())
    d, dh = spec.d, spec.dh
    m, n = min(d, dh), max(d, dh)
    f = 4.0 * d * dh * spec.T + 2.0 * d * dh * spec.T          # queries' [A|B], apply
    f += 2 * 6.0 * d * dh * upd_tok + 2 * 6.0 * d * dh * upd_tok  # keys' forward, gradient (split)
    if spec.muon:
        f += 3 * n_upd * 3 * spec.ns_iters * (4.0 * m * m * n + 2.0 * m ** 3)
    return heads * f


def linear_bytes_per_step(spec) -> float:
    """HBM bytes of the linear small-chunk layer: Q, K, V read and O written
    once (storage type), lr read once, W0 read and Wf written (fp32)."""
    es = 2 if spec.dtype == "bf16" else 4
    tok = spec.B * spec.H * spec.T
    return tok * spec.d * es * 4 + tok * 4 + spec.H * spec.d * spec.d * 4 + spec.B * spec.H * spec.d * spec.d * 4


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload (profiles/<kernel>__<workload>.txt, line 'traffic_bytes_per_launch: X'),
    or None if there is none (or it is marked stale)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.txt")
    try:
        txt = open(p).read()
    except OSError:
        return None
    m = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*$", txt, re.M)
    if not m or re.search(r"^stale:\s*yes", txt, re.M):
        return None
    return float(m.group(1))


# ------------------------------------------------------------------ the GPU arm
def roofline(spec, kinds: dict, steps: int, peaks: dict, peak_src: str) -> dict:
    """The roofline object of the kernel class with the largest device time.

    kinds: kernel name -> (kind, total ms, timed launches, launches) over `steps`
    steps. A tensor-bound class is measured against the burst bf16 peak (each
    launch lasts well under a millisecond, inside a timed region of a fraction of
    a second), with the sustained figure beside it; the linear kernel against the
    measured copy bandwidth."""
    all_ms = sum(v[1] for v in kinds.values()) or 1.0
    top_name, (top_k, top_ms, top_timed, _) = max(kinds.items(), key=lambda kv: kv[1][1])
    per_launch_ms = top_ms / max(top_timed, 1)
    launches_per_step = top_timed / steps
    if spec.fast_net == "linear":
        bytes_launch = linear_bytes_per_step(spec) / max(launches_per_step, 1)
        achieved = bytes_launch / (per_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "kernel": top_name,
                "bytes_per_launch": bytes_launch}
    else:
        fl = kernel_flops_per_launch(spec, top_k, launches_per_step)
        achieved = fl / (per_launch_ms * 1e-3) / 1e12 if fl else None
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s",
                "frac": achieved / pk if achieved else None, "kernel": top_name,
                "peak_kind": f"bf16 dense burst ({peak_src})",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"] if achieved else None,
                "flop_per_launch": fl}
    roof["launch_ms"] = per_launch_ms
    roof["share"] = top_ms / all_ms
    roof["traffic"] = read_traffic(top_name, spec.name)
    return roof


def workload_spec(args):
    from long_seq_models_chunked_b300 import synth
    spec = synth.WORKLOADS[args.workload]
    if args.seq_len:
        spec = spec.replace(T=args.seq_len, chunk=min(spec.chunk, args.seq_len))
    return spec


def check_library_for_world(features: int, world: int) -> None:
    """A process that runs beside ranks on other GPUs must load the build
    without cluster multicast; refuse anything else."""
    from long_seq_models_chunked_b300.abi import TTT_FEATURE_CLUSTER_MULTICAST
    if world > 1 and features & TTT_FEATURE_CLUSTER_MULTICAST:
        raise SystemExit(f"refusing --gpus {world}: the loaded library uses cluster multicast, which is "
                         "built for processes that use one GPU alone; multi-GPU runs load "
                         "libttt_b300_local.so (TTT_B300_LIBRARY=local)")


def run_ours(args, rank, local, world, pg):
    import numpy as np
    import torch

    from long_seq_models_chunked_b300 import abi, accounting, synth

    check_library_for_world(abi.ttt_build_features(), world)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = workload_spec(args)
    x = synth.layer_inputs(spec.replace(seed=spec.seed + 1000 * rank) if rank else spec, exact=False)
    holder = abi.cfg_from_spec(spec)
    cfg = holder.cfg
    tdt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32

    def dev_tensor(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if spec.dtype == "bf16" and a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(dev)

    Q, K, V = (dev_tensor(x[n]) for n in ("Q", "K", "V"))
    lr = torch.from_numpy(x["lr"]).to(dev)
    W0 = [torch.from_numpy(w).to(dev) for w in x["W0"]]
    O = torch.empty_like(Q)
    shapes = abi.weight_shapes(cfg)
    Wf = [torch.empty((cfg.B, cfg.H) + s, dtype=torch.float32, device=dev) for s in shapes]
    ws = torch.empty(abi.ttt_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    w0 = W0 + [None] * (3 - len(W0))
    wf = Wf + [None] * (3 - len(Wf))
    stream = torch.cuda.current_stream(dev)

    def step():
        abi.ttt_fwd(cfg, Q, K, V, lr, w0[0], w0[1], w0[2], O, wf[0], wf[1], wf[2], ws, stream)

    clk = ClockSampler(local).__enter__()   # samples warm-up and timed steps (both under load)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    rc = abi.ttt_status(ws, stream)
    if rc != abi.TTT_OK:
        clk.__exit__(None, None, None)
        raise abi.TTTError(rc, "warm-up")

    # ---- timed region: device time per step, L2 flushed before each step.
    # Per-launch timing is off here: the headline is timed clean.
    abi.ttt_prof_enable(False)
    abi.ttt_prof_reset()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(pg, dev if world > 1 else None)
    torch.cuda.synchronize(dev)
    launches0 = abi.ttt_launch_count()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clk.__exit__(None, None, None)
    launches = abi.ttt_launch_count() - launches0
    barrier(pg, dev if world > 1 else None)
    rc = abi.ttt_status(ws, stream)
    if rc != abi.TTT_OK:
        raise abi.TTTError(rc, "timed steps")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(pg, ms_local, dev if world > 1 else None)
    tokens = sum_over_ranks(pg, float(spec.B * spec.T), dev if world > 1 else None)
    value = tokens / (ms * 1e-3)

    # ---- per-kernel shares: a second pass of the same steps with CUDA events
    # recorded around every launch on its own stream
    abi.ttt_prof_reset()
    abi.ttt_prof_enable(True)
    prof_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        prof_ev[i][0].record(stream)
        step()
        prof_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    abi.ttt_prof_enable(False)
    prof_step_ms = sum(a.elapsed_time(b) for a, b in prof_ev) / len(prof_ev)
    kinds = {}
    for k in range(abi.TTT_KERNEL_COUNT):
        tot_ms, timed, n = abi.ttt_prof_read(k)
        if n:
            kinds[abi.ttt_kernel_name(k)] = (k, tot_ms, timed, n)
    all_ms = sum(v[1] for v in kinds.values()) or 1.0
    peaks, peak_src = load_peaks()
    roof = roofline(spec, kinds, args.steps, peaks, peak_src)
    roof["timing"] = ("CUDA events around every launch on its stream, in a second pass of the same "
                      f"{args.steps} steps (that pass: {prof_step_ms:.3f} ms/step; the headline steps ran "
                      "without per-launch events)")
    layer_flops = accounting.algorithmic_flops(spec)
    layer_tflops = layer_flops / (ms_local * 1e-3) / 1e12
    mma = executed_mma_flops(spec)
    mma_tflops = mma / (ms_local * 1e-3) / 1e12 if mma else None
    shares = {nm: {"share": round(v[1] / all_ms, 4), "launches_per_step": v[3] / args.steps,
                   "ms_per_launch": round(v[1] / max(v[2], 1), 5)} for nm, v in kinds.items()}

    # ---- end to end through the host-buffer entry point
    e2e = run_e2e(args, spec, x, holder, dev, stream)

    return {
        "value": value, "ms_per_step": ms, "step_ms_all": [round(s, 4) for s in step_ms],
        "roofline": roof, "e2e": e2e, "gpu_launches": launches,
        "clocks": clk.summary(), "layer_tflops": layer_tflops,
        "layer_frac_of_peak": layer_tflops / peaks["bf16_tflops"] if spec.fast_net != "linear" else None,
        "layer_frac_of_sustained": layer_tflops / peaks["bf16_tflops_sustained"] if spec.fast_net != "linear" else None,
        "mma_tflops_executed": mma_tflops,
        "mma_frac_executed": mma_tflops / peaks["bf16_tflops"] if mma_tflops else None,
        "kernel_shares": shares, "peaks_source": peak_src,
    }


def run_e2e(args, spec, x, holder, dev, stream):
    """ttt_fwd_host from pinned host buffers, timed per call (H2D + layer + D2H)."""
    import numpy as np
    import torch

    from long_seq_models_chunked_b300 import abi

    cfg = holder.cfg
    tdt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32

    def pinned(a, bf=False):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if bf:
            t = t.view(torch.bfloat16)
        return t.pin_memory()

    bf = spec.dtype == "bf16"
    hQ, hK, hV = (pinned(x[n], bf) for n in ("Q", "K", "V"))
    hlr = pinned(x["lr"])
    hW0 = [pinned(w) for w in x["W0"]]
    hO = torch.empty(hQ.shape, dtype=tdt).pin_memory()
    hWf = [torch.empty((cfg.B, cfg.H) + s, dtype=torch.float32).pin_memory() for s in abi.weight_shapes(cfg)]
    arena = torch.empty(abi.ttt_host_arena_bytes(cfg), dtype=torch.uint8, device=dev)
    w0 = hW0 + [None] * (3 - len(hW0))
    wf = hWf + [None] * (3 - len(hWf))
    h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV, hlr, *hW0))
    d2h = hO.numel() * hO.element_size() + sum(t.numel() * t.element_size() for t in hWf)

    def call():
        abi.ttt_fwd_host(cfg, hQ, hK, hV, hlr, w0[0], w0[1], w0[2], hO, wf[0], wf[1], wf[2], arena, stream)

    for _ in range(max(1, min(args.warmup, 2))):
        call()
    n = max(1, min(args.steps, 5))
    times = []
    for _ in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        call()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = sum(times) / len(times)
    del arena
    return {"value": spec.B * spec.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n}


# ------------------------------------------------------------------ the oracle (CPU)
def oracle_sample(spec, budget_s: float):
    """Time the fp64 oracle on a bounded sample of the workload and scale it to the
    layer's tokens/s. The sample walks the heads (b, h) in order. In shifted mode it
    runs each head's chunks in order, carrying the weights from chunk to chunk. In
    single-chunk mode it runs contiguous blocks of 32768 tokens of the head's chunk,
    each an update then an apply from the head's W0 (the same per-token work). It
    stops once the time budget is spent (after at least one unit) or the workload
    is exhausted. A layer token (b, t) is H head-tokens of work, so the layer's
    tokens/s is the sample's head-tokens/s divided by H.
    Returns (tokens/s, description, seconds spent)."""
    import numpy as np

    from long_seq_models_chunked_b300 import synth
    from oracle import OracleCfg, ttt_head

    cfg = OracleCfg.from_spec(spec)
    C = spec.chunk
    w0 = synth.initial_weights(spec)  # each [H, out, in]
    block = 65536 if C > 65536 else 0
    single = spec.mode == "single"
    unit = min(C, 32768) if single else C
    units_per_head = -(-spec.T // unit) if single else spec.n_chunks
    mask = spec.update_mask()
    done, spent, units, heads = 0, 0.0, 0, 0
    for hi in range(spec.B * spec.H):
        b, h = divmod(hi, spec.H)
        heads += 1
        W = tuple(w[h].astype(np.float64) for w in w0)
        for u in range(units_per_head):
            s = u * unit
            e = min(spec.T, s + unit)
            ht = synth.head_tokens(spec, b, h, s, e)
            sub = OracleCfg(chunk=e - s, fast_net=cfg.fast_net, loss=cfg.loss, mode=cfg.mode, muon=cfg.muon,
                            ns_iters=cfg.ns_iters, wnorm=cfg.wnorm, step=cfg.step,
                            mask=[int(mask[0 if single else u])])
            w_in = tuple(w[h].astype(np.float64) for w in w0) if single else W
            t0 = time.perf_counter()
            _, w_out = ttt_head(sub, ht["Q64"], ht["K64"], ht["V64"], ht["lr"], w_in, block=block)
            spent += time.perf_counter() - t0
            if not single:
                W = w_out
            done += e - s
            units += 1
            if spent >= budget_s:
                break
        if spent >= budget_s:
            break
    value = done / spent / spec.H
    kind = "token blocks of the single chunk (update then apply)" if single else "chunks"
    desc = (f"{units} {kind}, {done} head-tokens over {heads} head(s) from (0,0) in order; "
            f"layer tokens/s = head-tokens/s / H ({spec.H})")
    return value, desc, spent


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, spec):
    vals, descs, secs = [], [], []
    for _ in range(args.warmup):
        oracle_sample(spec, 0.0)
    for _ in range(args.steps):
        v, desc, spent = oracle_sample(spec, args.cpu_budget / max(args.steps, 1))
        vals.append(v)
        descs.append(desc)
        secs.append(spent)
    value = statistics.median(vals)
    return value, descs[0], statistics.median(secs)


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="lm_chunk2k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle time (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override T (small cases for profiling; not a bench configuration)")
    args = ap.parse_args()

    spec = workload_spec(args)
    config = {"workload": spec.name + (f" (T overridden to {spec.T})" if args.seq_len else ""), "B": spec.B, "H": spec.H, "T": spec.T, "d": spec.d, "dh": spec.dh,
              "chunk": spec.chunk, "fast_net": spec.fast_net, "loss": spec.loss, "mode": spec.mode,
              "muon": spec.muon, "ns_iters": spec.ns_iters, "wnorm": spec.wnorm, "update": spec.update,
              "storage": spec.dtype, "state": "fp32", "global_batch": spec.B, "seq_len": spec.T,
              "parallelism": f"dp{args.gpus} (independent sequences per GPU)",
              "l2": "flushed before every timed step (256 MiB write)"}
    dtype = "bf16" if spec.dtype == "bf16" else "f32"

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        value, desc, sample_s = run_reference(args, spec)
        cores = blas_threads()
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": spec.B * spec.T / value * 1e3,
                "ms_per_step_kind": ("extrapolated: the whole workload's tokens divided by the sampled "
                                     "tokens/s; each timed step is a bounded sample, not the whole workload"),
                "sample_seconds_per_step": sample_s,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config, "impl": "reference",
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if args.gpus > 1:
        # ranks on several GPUs load the build without cluster multicast
        os.environ["TTT_B300_LIBRARY"] = "local"
    rank, local, world, pg = dist_setup(args.gpus)
    res = run_ours(args, rank, local, world, pg)
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, desc, spent = oracle_sample(spec, args.cpu_budget)
        cpu = {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle", "sample": desc,
               "seconds": round(spent, 2)}
    line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": config,
            "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
            "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
            "layer_tflops": res["layer_tflops"], "layer_frac_of_peak": res["layer_frac_of_peak"],
            "layer_frac_of_sustained": res["layer_frac_of_sustained"],
            "mma_tflops_executed": res["mma_tflops_executed"], "mma_frac_executed": res["mma_frac_executed"],
            "kernel_shares": res["kernel_shares"], "step_ms_all": res["step_ms_all"]}
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
