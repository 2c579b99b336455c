"""Expert parallelism over several ranks: the host side of the MoonEP page's
contracts ("Step-by-step"), on any torch.distributed process group.

  * ``Plan`` -- the dispatch plan computed by ``moe_ep_plan`` (libmoe, native)
    from the gathered per-rank expert counts: every rank processes exactly
    S*K routed rows; rank r owns experts [rG, rG + G), G = E/R, and keeps
    copies of remote experts in B preload slots (B = E/R for training).
  * ``send_rows`` / ``recv_layout`` -- which routed pairs a source sends to
    every destination, and how a destination lays its rows out: local expert
    by local expert (home experts, then the slots, then remote experts left
    without a slot), source rank by source rank inside an expert, so the local
    grouped GEMM addresses experts by row index through a local cu_seqlens.
  * ``exchange`` -- point-to-point transfer of one buffer per (source,
    destination) pair: the all-to-all of the dispatch and of the combine.
  * ``reduce_grad`` -- the gradients of slot copies go to the home rank of
    their expert, are added to the home gradient in rank order and the slots
    are cleared.

Nothing here computes on rows: the expert FFN of the local rows is the
caller's (on GPUs, ``moe_expert_ffn`` over the local [G + B, H, H'] weights).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import _lib as L


class Plan:
    """The dispatch plan of one layer call.  ``counts`` [R, E]: pairs each
    source rank routes to each expert (every row sums to S*K)."""

    def __init__(self, counts, S: int, K: int, B: int):
        counts = np.asarray(counts, np.int32)
        self.R, self.E = counts.shape
        self.S, self.K, self.B = S, K, B
        self.G = self.E // self.R
        self.counts = counts
        (self.piece_count, self.piece_offset, self.slot_expert, self.local_counts,
         self.remote_reads) = L.moe_ep_plan(self.R, self.E, S, K, B, counts)

    def local_experts(self, d: int):
        """Experts of rank d's rows in local order: home experts, the experts
        in its slots, then remote experts read from their home rank."""
        home = list(range(d * self.G, (d + 1) * self.G))
        slots = [int(e) for e in self.slot_expert[d] if e >= 0]
        placed = set(home) | set(slots)
        rest = [e for e in range(self.E) if e not in placed and self.piece_count[d, :, e].sum() > 0]
        return home + slots + rest

    def local_cu_seqlens(self, d: int):
        """Exclusive scan of the rows per local expert of rank d."""
        rows = [int(self.piece_count[d, :, e].sum()) for e in self.local_experts(d)]
        return np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)


def send_rows(plan: Plan, s: int, idx_s):
    """For source rank s with top-K ids idx_s [S, K]: for every destination d,
    the pair indices (t*K + k) it sends, in d's local row order."""
    flat = np.asarray(idx_s).reshape(-1)
    by_expert = [np.nonzero(flat == e)[0] for e in range(plan.E)]  # stable: (t, k) order
    out = []
    for d in range(plan.R):
        parts = []
        for e in plan.local_experts(d):
            c, o = int(plan.piece_count[d, s, e]), int(plan.piece_offset[d, s, e])
            if c:
                parts.append(by_expert[e][o:o + c])
        out.append(np.concatenate(parts).astype(np.int64) if parts else np.zeros(0, np.int64))
    return out


def recv_layout(plan: Plan, d: int):
    """Rank d's local rows as blocks (source s, expert e, rows), in local row
    order: receiving buffer s is split into consecutive blocks of these sizes."""
    blocks = []
    for e in plan.local_experts(d):
        for s in range(plan.R):
            c = int(plan.piece_count[d, s, e])
            if c:
                blocks.append((s, e, c))
    return blocks


def assemble(plan: Plan, d: int, received):
    """Rank d's local row buffer from the per-source received buffers
    (received[s] holds source s's rows in d's local expert order)."""
    taken = [0] * plan.R
    rows = []
    for s, e, c in recv_layout(plan, d):
        rows.append(received[s][taken[s]:taken[s] + c])
        taken[s] += c
    return torch.cat(rows) if rows else received[0][:0]


def split_back(plan: Plan, d: int, local_rows):
    """Inverse of ``assemble``: rank d's local rows cut back into one buffer per
    source rank (the combine direction of the exchange)."""
    parts = [[] for _ in range(plan.R)]
    r = 0
    for s, e, c in recv_layout(plan, d):
        parts[s].append(local_rows[r:r + c])
        r += c
    return [torch.cat(p) if p else local_rows[:0] for p in parts]


def exchange(send, recv_shapes, group=None):
    """One buffer to and from every rank (send[d] goes to rank d; the buffer
    received from rank s has shape recv_shapes[s]); point-to-point, so it runs
    on backends without an all-to-all (gloo)."""
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    dtype = send[rank].dtype
    recv = [torch.empty(recv_shapes[s], dtype=dtype) for s in range(world)]
    recv[rank] = send[rank].clone()
    reqs = []
    for peer in range(world):
        if peer == rank:
            continue
        if send[peer].numel():
            reqs.append(dist.isend(send[peer].contiguous(), peer, group=group))
        if recv[peer].numel():
            reqs.append(dist.irecv(recv[peer], peer, group=group))
    for q in reqs:
        q.wait()
    return recv


def gather_counts(idx_local, E: int, group=None):
    """counts [R, E] of every rank from the local top-K ids (all-gather)."""
    world = dist.get_world_size(group)
    mine = torch.from_numpy(np.bincount(np.asarray(idx_local).reshape(-1), minlength=E).astype(np.int64))
    out = [torch.empty(E, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(out, mine, group=group)
    return np.stack([o.numpy() for o in out]).astype(np.int32)


def reduce_grad(plan: Plan, grad, group=None):
    """grad [G + B, ...] of this rank (home experts, then the slots): every slot
    holding a copy of a remote expert is sent to that expert's home rank, which
    adds the copies to its home gradient in increasing rank order; the sent
    slots are cleared.  In place; returns grad."""
    rank = dist.get_rank(group)
    G, B = plan.G, plan.B
    reqs = []
    for j in range(B):
        e = int(plan.slot_expert[rank, j])
        if e >= 0:
            reqs.append(dist.isend(grad[G + j].contiguous(), e // G, group=group))
    incoming = []
    for d in range(plan.R):
        if d == rank:
            continue
        for j in range(B):
            e = int(plan.slot_expert[d, j])
            if e >= 0 and e // G == rank:
                buf = torch.empty_like(grad[0])
                reqs.append(dist.irecv(buf, d, group=group))
                incoming.append((d, e, buf))
    for q in reqs:
        q.wait()
    for d, e, buf in sorted(incoming, key=lambda v: (v[0], v[1])):
        grad[e - rank * G] += buf
    for j in range(B):
        if int(plan.slot_expert[rank, j]) >= 0:
            grad[G + j].zero_()
    return grad
