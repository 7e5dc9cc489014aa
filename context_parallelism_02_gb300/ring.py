"""Ring attention over real ranks: the host driver of context parallelism.

Each process holds one rank's shards, in that rank's local row order
(``cp_shard_map``): its queries for the whole run, and one K/V block at a
time.  At ring step k = 0..N-1 it folds the block it holds -- the block of
rank (rank - k) mod N -- into its running (out, lse) with ``flash_block_step``
while that block travels on to rank + 1 and the next one arrives from
rank - 1.  This is the loop of the ring sketch in "Context Parallelism"
("Ring attention": send to rank + 1, receive from rank - 1, run flash_block
on the block held, wait, swap) and step 2 of "Algorithmic Mechanics" in
"Sequence Parallelism in LLMs"; the transfer of step k overlaps the compute
of step k ("Overlapping Compute and Communication": hidden when
T_comp >= T_comm).  N compute steps, N - 1 transfers.

The transfer is a transport object:
  * ``P2PTransport`` -- torch.distributed point-to-point, batched send to
    rank + 1 and receive from rank - 1: NCCL for CUDA tensors (the block lands
    in this GPU's own HBM, in a buffer the driver owns), gloo for CPU tensors;
  * ``HostStagedTransport`` -- CUDA tensors over a CPU-only (gloo) group: the
    block is copied to pinned host memory, exchanged by gloo, and copied into
    the receive buffer on a copy stream, all while the step computes.

All arithmetic of the path runs in libcp's kernels (``flash_block_step``); this
module only orders launches and transfers.  ``step`` can be replaced (the
CPU tests pass one that records what each rank holds).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
import torch.distributed as dist

from . import api


# ----------------------------------------------------------------------------- sharding


def shard_positions(S: int, N: int, layout: int, rank: int) -> torch.Tensor:
    """Global positions of rank ``rank``'s local rows (int64, length S / N)."""
    return torch.from_numpy(api.cp_shard_map(S, N, layout)[rank].astype("int64"))


def shard(x: torch.Tensor, rank: int, N: int, layout: int, dim: int = 1) -> torch.Tensor:
    """Rank ``rank``'s shard of a global-order tensor, in its local row order
    (the input distribution a data loader would do; a copy)."""
    pos = shard_positions(x.shape[dim], N, layout, rank).to(x.device)
    return x.index_select(dim, pos).contiguous()


def unshard(parts, N: int, layout: int, dim: int = 1) -> torch.Tensor:
    """Inverse of :func:`shard`: the N ranks' shards back in global order."""
    S = parts[0].shape[dim] * N
    shape = list(parts[0].shape)
    shape[dim] = S
    out = parts[0].new_empty(shape)
    for r, p in enumerate(parts):
        out.index_copy_(dim, shard_positions(S, N, layout, r).to(p.device), p)
    return out


# ----------------------------------------------------------------------------- transports


def _peers(group):
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    if group is not None:
        nxt, prv = dist.get_global_rank(group, nxt), dist.get_global_rank(group, prv)
    return nxt, prv


class P2PTransport:
    """Send the held block to rank + 1 and receive the next from rank - 1 with
    one batched torch.distributed point-to-point call.

    NCCL (CUDA tensors): the NCCL stream is ordered after the work already
    queued on the current stream (the previous step, which read the receive
    buffer), and :meth:`wait` orders the current stream after the transfer,
    so the host never blocks.  gloo (CPU tensors): :meth:`wait` blocks."""

    def __init__(self, group=None):
        self.group = group
        self.next, self.prev = _peers(group)

    def start(self, send, recv):
        ops = [dist.P2POp(dist.isend, t, self.next, self.group, tag=i) for i, t in enumerate(send)]
        ops += [dist.P2POp(dist.irecv, t, self.prev, self.group, tag=i) for i, t in enumerate(recv)]
        return dist.batch_isend_irecv(ops)

    def wait(self, works):
        for w in works:
            w.wait()


class HostStagedTransport:
    """CUDA blocks over a CPU-only (gloo) process group: device -> pinned host,
    gloo send/receive between the host buffers, host -> device into the
    receive buffer.  The copies run on a copy stream and the exchange on gloo's
    threads, so both overlap the step queued in between."""

    def __init__(self, group=None):
        self.inner = P2PTransport(group)
        self.copy = None
        self.host = {}

    def _pinned(self, key, like):
        t = self.host.get(key)
        if t is None or t.shape != like.shape or t.dtype != like.dtype:
            t = torch.empty(like.shape, dtype=like.dtype, pin_memory=True)
            self.host[key] = t
        return t

    def start(self, send, recv):
        if self.copy is None:
            self.copy = torch.cuda.Stream(send[0].device)
        compute = torch.cuda.current_stream(send[0].device)
        # everything queued so far (the previous step, which read the receive
        # buffer) must finish before the receive buffer is overwritten
        queued = compute.record_event()
        # the held block is complete once the copy stream's last upload is
        self.copy.synchronize()
        hs = [self._pinned(("s", i), t) for i, t in enumerate(send)]
        hr = [self._pinned(("r", i), t) for i, t in enumerate(recv)]
        with torch.cuda.stream(self.copy):
            for h, d in zip(hs, send):
                h.copy_(d, non_blocking=True)
        self.copy.synchronize()
        return self.inner.start(hs, hr), recv, hr, queued, compute

    def wait(self, handle):
        works, recv, hr, queued, compute = handle
        self.inner.wait(works)
        with torch.cuda.stream(self.copy):
            self.copy.wait_event(queued)
            for d, h in zip(recv, hr):
                d.copy_(h, non_blocking=True)
        compute.wait_stream(self.copy)


# ----------------------------------------------------------------------------- driver


def cuda_step(q, k, v, out_acc, lse_acc, out_final, *, rank, source, N, S, layout, causal,
              scale, accumulate):
    """One ring step in libcp (``flash_block_step``) on the current stream."""
    api.flash_block_step(q, k, v, rank, source, N, S, layout, causal, scale, out_acc=out_acc,
                         lse_acc=lse_acc, out_final=out_final, accumulate=accumulate)


@dataclass
class StepTimes:
    """CUDA events around each step's compute (filled by :func:`ring_attention`)."""
    events: list = field(default_factory=list)

    def compute_ms(self):
        return [a.elapsed_time(b) for a, b in self.events]


def ring_attention(q, k, v, *, rank: int, N: int, S: int, layout: int, causal: bool = True,
                   scale: float | None = None, transport=None, step=cuda_step,
                   state_dtype=torch.float32, times: StepTimes | None = None):
    """Ring attention forward for one rank; returns (out, lse).

    q ``[B, C, Hq, D]``, k/v ``[B, C, Hkv, D]`` (C = S / N): this rank's shards
    in local row order.  out ``[B, C, Hq, D]`` (q's dtype) and lse
    ``[B, Hq, C]`` (fp32, natural log) are this rank's rows of the attention
    over all S keys.  ``transport`` moves the K/V blocks around the ring
    (required when N > 1).  k and v are only read: the blocks that arrive go
    into two buffer pairs of the driver's own.
    """
    if N > 1 and transport is None:
        raise ValueError("a ring of N > 1 ranks needs a transport")
    B, C, Hq, D = q.shape
    bufs = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(min(N - 1, 2))]
    out_acc = torch.empty((B, C, Hq, D), dtype=state_dtype, device=q.device)
    lse_acc = torch.empty((B, Hq, C), dtype=state_dtype, device=q.device)
    out = torch.empty_like(q)
    cur = (k, v)
    for s in range(N):
        nxt = bufs[s % 2] if s + 1 < N else None
        handle = transport.start(cur, nxt) if nxt is not None else None
        if times is not None and q.is_cuda:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record()
        step(q, cur[0], cur[1], out_acc, lse_acc, out if s == N - 1 else None, rank=rank,
             source=(rank - s) % N, N=N, S=S, layout=layout, causal=causal, scale=scale,
             accumulate=s > 0)
        if times is not None and q.is_cuda:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record()
            times.events.append((e0, e1))
        if handle is not None:
            transport.wait(handle)
            cur = nxt
    return out, lse_acc


def ring_attention_emulated(q, k, v, N: int, layout: int, causal: bool = True,
                            scale: float | None = None, stream=None):
    """All N ranks of the ring in one process, on global-order tensors: each
    rank's shards are cut once, then every (rank, step) runs flash_block_step
    on the source rank's shard in place (the transfer is free).  Returns
    (out, lse) in global order.  The per-step launches are the ones a device
    of a real ring makes."""
    B, S, Hq, D = q.shape
    qs = [shard(q, r, N, layout) for r in range(N)]
    ks = [shard(k, r, N, layout) for r in range(N)]
    vs = [shard(v, r, N, layout) for r in range(N)]
    outs, lses = [], []
    for r in range(N):
        C = S // N
        out_acc = torch.empty((B, C, Hq, D), dtype=torch.float32, device=q.device)
        lse_acc = torch.empty((B, Hq, C), dtype=torch.float32, device=q.device)
        out = torch.empty_like(qs[r])
        for s in range(N):
            src = (r - s) % N
            api.flash_block_step(qs[r], ks[src], vs[src], r, src, N, S, layout, causal, scale,
                                 out_acc=out_acc, lse_acc=lse_acc,
                                 out_final=out if s == N - 1 else None, accumulate=s > 0,
                                 stream=stream)
        outs.append(out)
        lses.append(lse_acc)
    return unshard(outs, N, layout, dim=1), unshard(lses, N, layout, dim=2)
