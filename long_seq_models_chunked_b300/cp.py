"""Context parallelism of the chunked TTT layer (LaCT page, "Large Chunk
Test-Time Training", §2.2.2): the tokens of every chunk are split into shards
held by different ranks. Each rank computes its shard's partial gradient with
the same fast weights, the partials are summed over the ranks (the all-reduce,
the method's one exchange), and every rank applies the same update to its own
copy of the weights and the apply to its own queries.

`rank_steps` is one rank's chunk loop, written as a generator: it yields its
partial gradient whenever an update is due and expects the sum over the ranks
back. `run_rank` drives it with an all-reduce (torch.distributed on several
GPUs); `run_lockstep` drives several ranks' generators in one process, summing
the partials on the device (one GPU standing in for several, with nothing
running concurrently). Each rank's state is a `Shard`: the C ABI's
context-parallel calls on the rank's own workspace. Argument marshalling only:
every step runs in the CUDA library.
"""
from __future__ import annotations

from typing import Callable, List, Sequence

from . import abi


class Shard:
    """One rank's context-parallel state on the current device.

    `holder` describes the layer (abi.cfg_from_spec) with cfg.chunk = the
    rank's largest shard of a chunk; the local token tensors are
    [B, H, T_local, d]."""

    def __init__(self, holder: abi.CfgHolder, W0: Sequence, T_local: int, stream=None):
        import torch
        self.holder = holder
        self.cfg = holder.cfg
        self.T = T_local
        self.stream = stream
        dev = W0[0].device
        self.ws = torch.empty(abi.ttt_cp_workspace_bytes(self.cfg), dtype=torch.uint8, device=dev)
        c = self.cfg
        self.G = torch.empty((c.B * c.H, 3, c.d, c.dh), dtype=torch.float32, device=dev)
        abi.ttt_cp_begin(c, W0[0], W0[1], W0[2], self.ws, stream)

    def grad(self, K, V, lr, start: int, n: int):
        abi.ttt_cp_grad(self.cfg, K, V, lr, self.T, start, n, self.G, self.ws, self.stream)
        return self.G

    def update(self, G) -> None:
        abi.ttt_cp_update(self.cfg, G, self.ws, self.stream)

    def apply(self, Q, O, start: int, n: int) -> None:
        abi.ttt_cp_apply(self.cfg, Q, self.T, start, n, O, self.ws, self.stream)

    def end(self):
        import torch
        c = self.cfg
        dev = self.G.device
        Wf = [torch.empty((c.B, c.H) + s, dtype=torch.float32, device=dev) for s in abi.weight_shapes(c)]
        abi.ttt_cp_end(c, Wf[0], Wf[1], Wf[2], self.ws, self.stream)
        return Wf

    def status(self) -> int:
        return abi.ttt_status(self.ws, self.stream)


def rank_steps(shard, Q, K, V, lr, O, T_local: int, chunk_local: int, shifted: bool, mask: Sequence[int]):
    """One rank's part of the layer over its shards of every chunk: tokens
    [c * chunk_local, (c + 1) * chunk_local) of the local tensors are its shard
    of chunk c. Shifted mode applies a chunk before its update (LaCT page §3.2),
    single mode after it (§3.1). Yields the partial gradient at every update and
    receives the sum over the ranks."""
    n_chunks = -(-T_local // chunk_local)
    for c in range(n_chunks):
        s = c * chunk_local
        n = min(chunk_local, T_local - s)
        if shifted:
            shard.apply(Q, O, s, n)
        if mask[c]:
            total = yield shard.grad(K, V, lr, s, n)
            shard.update(total)
        if not shifted:
            shard.apply(Q, O, s, n)


def run_rank(steps, all_reduce: Callable) -> None:
    """Drives one rank's generator; all_reduce(G) sums G over the ranks in place."""
    try:
        G = next(steps)
        while True:
            all_reduce(G)
            G = steps.send(G)
    except StopIteration:
        pass


def run_lockstep(all_steps: List) -> None:
    """Drives several ranks' generators in one process: at every update the
    partials are summed (on the device, in rank order) and the sum goes back to
    every rank."""
    pending = []
    for st in all_steps:
        try:
            pending.append(next(st))
        except StopIteration:
            pending.append(None)
    while any(p is not None for p in pending):
        if any(p is None for p in pending):
            raise RuntimeError("ranks disagree on the number of updates")
        total = pending[0].clone()
        for p in pending[1:]:
            total += p
        nxt = []
        for st in all_steps:
            try:
                nxt.append(st.send(total))
            except StopIteration:
                nxt.append(None)
        pending = nxt
