"""Message exchange between ranks of a multi-GPU job.

The SYLVIE guide's worker loop (section 5, step 4; section 11) quantises the
boundary rows a worker owns, exchanges the codes and their (min, scale) with
an all-to-all, dequantises what arrives and aggregates; the backward sends the
boundary copies' gradients back to their owners the same way (section 3), and
the weight gradients are summed with an all-reduce (section 11).

Layout.  The message buffer is ordered by slot s = (receiving partition q,
node u), q first, then u, each row at byte slot_off[s]; meta holds (min,
scale) per slot.  Partitions are contiguous node blocks, so inside receiver
q's segment the slots whose node lies in partition p form one contiguous
slot range.  Partitions are dealt to ranks in contiguous blocks (rank r holds
partitions [P*r//W, P*(r+1)//W)), so everything rank r sends to rank t in the
forward direction -- the rows of slots (q, u) with q held by t and u held by
r -- is one slot range per receiving partition q, and the backward direction
returns exactly those ranges.  Every rank keeps the buffer in the global slot
layout: a rank writes the rows it produces at their own offsets, and the
exchange moves the byte ranges of the other ranks' rows into place, so the
aggregation kernels read a received row exactly where a single-GPU run reads
it.  Nothing is repacked or re-quantised on the way.

Transport.  ``exchange`` takes a ``comm`` object with ``rank``, ``world`` and
``alltoall(out, inp, out_splits, in_splits)`` / ``allreduce_(t)``:
``DistComm`` wraps ``torch.distributed`` (one rank per GPU over NCCL, or gloo
on CPU tensors); ``LocalGroup`` runs W virtual ranks in one process, with the
all-to-all's exact data movement, for tests on one device.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

Ranges = List[Tuple[int, int]]


class ExchangePlan:
    """Slot ranges each rank pair exchanges, from the boundary's host-side
    part_start [P+1], send_start [P+1] and slot_node [S] arrays."""

    def __init__(self, part_start, send_start, slot_node, world: int):
        part_start = np.asarray(part_start, np.int64)
        send_start = np.asarray(send_start, np.int64)
        slot_node = np.asarray(slot_node, np.int64)
        P = part_start.size - 1
        if world < 1 or world > P:
            raise ValueError(f"world size {world} must be between 1 and the partition count {P}")
        self.P, self.world = P, world
        self.n_slots = int(send_start[-1])
        self.rank_parts = [(P * r // world, P * (r + 1) // world) for r in range(world)]
        # cut[q][p] = first slot of receiver q's segment whose node lies in
        # partition p (cut[q][P] = the segment's end)
        self.cut = np.empty((P, P + 1), np.int64)
        for q in range(P):
            a, b = int(send_start[q]), int(send_start[q + 1])
            self.cut[q] = a + np.searchsorted(slot_node[a:b], part_start, side="left")
        # fwd[r][t]: slot ranges whose node rank r owns and whose receiving
        # partition rank t holds (one range per receiving partition)
        self.fwd: List[List[Ranges]] = [[[] for _ in range(world)] for _ in range(world)]
        for r, (p0, p1) in enumerate(self.rank_parts):
            for t, (q0, q1) in enumerate(self.rank_parts):
                for q in range(q0, q1):
                    a, b = int(self.cut[q][p0]), int(self.cut[q][p1])
                    if b > a:
                        self.fwd[r][t].append((a, b))

    def owned(self, rank: int) -> Ranges:
        """Slot ranges whose node this rank owns (the forward rows it writes)."""
        return [rg for t in range(self.world) for rg in self.fwd[rank][t]]

    def received(self, rank: int) -> Tuple[int, int]:
        """The slots this rank's partitions receive: one contiguous range (the
        backward rows it writes)."""
        q0, q1 = self.rank_parts[rank]
        return int(self.cut[q0][0]), int(self.cut[q1 - 1][self.P]) if q1 > q0 else int(self.cut[q0][0])

    def ranges(self, src: int, dst: int, direction: str) -> Ranges:
        """Slot ranges src sends to dst: forward rows go from the node's owner
        to the receiving partition's rank, backward rows the other way."""
        if direction == "fwd":
            return self.fwd[src][dst]
        if direction == "bwd":
            return self.fwd[dst][src]
        raise ValueError(direction)


def _byte_ranges(ranges: Ranges, slot_off) -> Ranges:
    return [(int(slot_off[a]), int(slot_off[b])) for a, b in ranges]


def _gather(buf, ranges: Ranges):
    import torch

    parts = [buf[a:b] for a, b in ranges if b > a]
    if not parts:
        return buf[:0]
    return parts[0] if len(parts) == 1 else torch.cat(parts)


def _scatter(buf, data, ranges: Ranges) -> None:
    at = 0
    for a, b in ranges:
        if b > a:
            buf[a:b].copy_(data[at:at + (b - a)])
            at += b - a


def send_chunks(plan: ExchangePlan, rank: int, packed, meta, slot_off, direction: str):
    """This rank's send buffers (bytes, meta floats) and per-destination sizes,
    in destination-rank order; nothing for itself (its rows are in place)."""
    mflat = meta.reshape(-1)
    by, mt, nb, nm = [], [], [], []
    for dst in range(plan.world):
        rg = plan.ranges(rank, dst, direction) if dst != rank else []
        b = _gather(packed, _byte_ranges(rg, slot_off))
        m = _gather(mflat, [(2 * a, 2 * c) for a, c in rg])
        by.append(b)
        mt.append(m)
        nb.append(int(b.numel()))
        nm.append(int(m.numel()))
    import torch

    return torch.cat(by), torch.cat(mt), nb, nm


def recv_sizes(plan: ExchangePlan, rank: int, slot_off, direction: str):
    nb, nm = [], []
    for src in range(plan.world):
        rg = plan.ranges(src, rank, direction) if src != rank else []
        nb.append(sum(int(slot_off[b]) - int(slot_off[a]) for a, b in rg))
        nm.append(sum(2 * (b - a) for a, b in rg))
    return nb, nm


def place_received(plan: ExchangePlan, rank: int, recv_b, recv_m, packed, meta, slot_off,
                   direction: str) -> None:
    """Copy each source rank's bytes and meta into their slots' places."""
    mflat = meta.reshape(-1)
    ob, om = 0, 0
    for src in range(plan.world):
        if src == rank:
            continue
        rg = plan.ranges(src, rank, direction)
        br = _byte_ranges(rg, slot_off)
        mr = [(2 * a, 2 * b) for a, b in rg]
        nb = sum(b - a for a, b in br)
        nm = sum(b - a for a, b in mr)
        _scatter(packed, recv_b[ob:ob + nb], br)
        _scatter(mflat, recv_m[om:om + nm], mr)
        ob += nb
        om += nm


def exchange(plan: ExchangePlan, comm, packed, meta, slot_off, direction: str) -> None:
    """One all-to-all of message rows (SYLVIE guide section 5 step 4 forward,
    section 3 backward).  Before: this rank has written its own rows -- the
    forward rows of the slots whose node it owns, or the backward rows of the
    slots its partitions receive.  After: the rows the other ranks wrote for
    this rank are in place as well.  ``slot_off`` is a host int64 array."""
    import torch

    r = comm.rank
    send_b, send_m, in_b, in_m = send_chunks(plan, r, packed, meta, slot_off, direction)
    out_b, out_m = recv_sizes(plan, r, slot_off, direction)
    recv_b = torch.empty(sum(out_b), dtype=packed.dtype, device=packed.device)
    recv_m = torch.empty(sum(out_m), dtype=meta.dtype, device=meta.device)
    comm.alltoall(recv_b, send_b, out_b, in_b)
    comm.alltoall(recv_m, send_m, out_m, in_m)
    place_received(plan, r, recv_b, recv_m, packed, meta, slot_off, direction)


class DistComm:
    """torch.distributed transport: one process per rank."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist, self.group = dist, group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def alltoall(self, out, inp, out_splits: Sequence[int], in_splits: Sequence[int]) -> None:
        self.dist.all_to_all_single(out, inp, list(out_splits), list(in_splits), group=self.group)

    def allreduce_(self, t) -> None:
        """Sum over ranks in place (the weight gradients, section 11)."""
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM, group=self.group)


class LocalGroup:
    """W virtual ranks in one process (tests on one device): every rank's
    send buffer is formed first, then each rank receives the chunks
    addressed to it in source-rank order -- the data an all-to-all
    delivers -- and places them as ``exchange`` does."""

    def __init__(self, world: int):
        self.world = world

    def exchange_all(self, plan: ExchangePlan, packed: list, meta: list, slot_off,
                     direction: str) -> None:
        """The all-to-all of ``exchange`` for every virtual rank at once."""
        import torch

        sends = [send_chunks(plan, r, packed[r], meta[r], slot_off, direction)
                 for r in range(self.world)]
        for t in range(self.world):
            out_b, out_m = recv_sizes(plan, t, slot_off, direction)
            cb, cm = [], []
            for r in range(self.world):
                sb, sm, nb, nm = sends[r]
                ob, om = sum(nb[:t]), sum(nm[:t])
                cb.append(sb[ob:ob + nb[t]])
                cm.append(sm[om:om + nm[t]])
            recv_b, recv_m = torch.cat(cb), torch.cat(cm)
            assert recv_b.numel() == sum(out_b) and recv_m.numel() == sum(out_m)
            place_received(plan, t, recv_b, recv_m, packed[t], meta[t], slot_off, direction)

    @staticmethod
    def allreduce_all(ts: list) -> None:
        """Sum of every virtual rank's tensor, written back to each."""
        total = ts[0].clone()
        for x in ts[1:]:
            total += x
        for x in ts:
            x.copy_(total)
