"""The multi-rank message exchange on CPU (no GPU): the exchange plan covers
every slot once, and two gloo ranks -- each holding only the rows it
produces, from the oracle -- end up with exactly the single-process buffer's
rows they read: the forward messages of their partitions' slots and the
backward messages of the slots whose nodes they own (SYLVIE guide, section 5
step 4 and section 3), plus the weight-gradient all-reduce (section 11)."""
import os
import socket
import sys

import numpy as np
import pytest

import oracle as O
from synth import planted_partition_edges
from sparse_aggregation_message_gb300.exchange import ExchangePlan, LocalGroup

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, P, F = 600, 6, 20


def _problem():
    s, d = planted_partition_edges(N, 4000, P, 0.7, 21)
    rp, col, val = O.csr_build(N, s, d)
    b = O.boundary_index(N, rp, col, val, P)
    nb = O.node_bits(N, rp, b, [50], [2, 8], 1)
    sb = nb[b["slot_node"]].astype(np.uint8)
    off = O.slot_offsets(sb, F)
    rng = np.random.default_rng(4)
    H = rng.standard_normal((N, F)).astype(np.float32)
    Gm = rng.standard_normal((N, F)).astype(np.float32)
    fwd, fmeta, _ = O.quant_pack(H, F, b["slot_node"], sb, off, 7)
    bwd, bmeta, _ = O.halo_quant_pack(b, Gm, F, sb, off, 8)
    return b, sb, off, fwd, fmeta, bwd, bmeta


def _rows_mask(ranges, off, S):
    """Byte mask and slot mask of the given slot ranges."""
    bm = np.zeros(int(off[-1]), bool)
    sm = np.zeros(S, bool)
    for a, z in ranges:
        bm[off[a]:off[z]] = True
        sm[a:z] = True
    return bm, sm


@pytest.mark.parametrize("world", [1, 2, 3, 6])
def test_plan_covers_every_slot_once(world):
    b, *_ = _problem()
    plan = ExchangePlan(b["part_start"], b["send_start"], b["slot_node"], world)
    S = b["n_slots"]
    seen = np.zeros(S, np.int64)
    for r in range(world):
        p0, p1 = plan.rank_parts[r]
        for t in range(world):
            q0, q1 = plan.rank_parts[t]
            for a, z in plan.fwd[r][t]:
                seen[a:z] += 1
                nodes = b["slot_node"][a:z]
                assert np.all((nodes >= b["part_start"][p0]) & (nodes < b["part_start"][p1]))
                assert b["send_start"][q0] <= a and z <= b["send_start"][q1]
    assert np.all(seen == 1)
    # the received ranges tile the slots in rank order
    edges = [plan.received(r) for r in range(world)]
    assert edges[0][0] == 0 and edges[-1][1] == S
    assert all(edges[i][1] == edges[i + 1][0] for i in range(world - 1))


def _check_rank(plan, rank, b, off, bufs, fwd, fmeta, bwd, bmeta, direction):
    import torch
    S = b["n_slots"]
    packed, meta = bufs
    if direction == "fwd":
        want = [plan.received(rank)]
        ref_b, ref_m = fwd, fmeta
    else:
        want = plan.owned(rank)
        ref_b, ref_m = bwd, bmeta
    bm, sm = _rows_mask(want, off, S)
    got_b, got_m = packed.numpy(), meta.numpy()
    assert np.array_equal(got_b[bm], ref_b[bm]), f"rank {rank} {direction} bytes"
    assert np.array_equal(got_m[sm].view(np.uint32), ref_m[sm].view(np.uint32)), f"rank {rank} meta"


def _own_rows(plan, rank, off, S, ref_b, ref_m, ranges):
    import torch
    packed = torch.zeros(int(off[-1]), dtype=torch.uint8)
    meta = torch.zeros((S, 2), dtype=torch.float32)
    for a, z in ranges:
        packed[off[a]:off[z]] = torch.from_numpy(ref_b[off[a]:off[z]])
        meta[a:z] = torch.from_numpy(ref_m[a:z])
    return packed, meta


@pytest.mark.parametrize("world", [2, 3])
def test_local_group_exchange(world):
    b, sb, off, fwd, fmeta, bwd, bmeta = _problem()
    plan = ExchangePlan(b["part_start"], b["send_start"], b["slot_node"], world)
    S = b["n_slots"]
    g = LocalGroup(world)
    fb = [_own_rows(plan, r, off, S, fwd, fmeta, plan.owned(r)) for r in range(world)]
    g.exchange_all(plan, [x[0] for x in fb], [x[1] for x in fb], off, "fwd")
    bb = [_own_rows(plan, r, off, S, bwd, bmeta, [plan.received(r)]) for r in range(world)]
    g.exchange_all(plan, [x[0] for x in bb], [x[1] for x in bb], off, "bwd")
    for r in range(world):
        _check_rank(plan, r, b, off, fb[r], fwd, fmeta, bwd, bmeta, "fwd")
        _check_rank(plan, r, b, off, bb[r], fwd, fmeta, bwd, bmeta, "bwd")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    try:
        import torch
        import torch.distributed as dist
        sys.path.insert(0, ROOT)
        from sparse_aggregation_message_gb300.exchange import DistComm, ExchangePlan, exchange
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        b, sb, off, fwd, fmeta, bwd, bmeta = _problem()
        S = b["n_slots"]
        plan = ExchangePlan(b["part_start"], b["send_start"], b["slot_node"], world)
        comm = DistComm()
        fbuf = _own_rows(plan, rank, off, S, fwd, fmeta, plan.owned(rank))
        exchange(plan, comm, fbuf[0], fbuf[1], off, "fwd")
        _check_rank(plan, rank, b, off, fbuf, fwd, fmeta, bwd, bmeta, "fwd")
        bbuf = _own_rows(plan, rank, off, S, bwd, bmeta, [plan.received(rank)])
        exchange(plan, comm, bbuf[0], bbuf[1], off, "bwd")
        _check_rank(plan, rank, b, off, bbuf, fwd, fmeta, bwd, bmeta, "bwd")
        dW = torch.full((3, 4), float(rank + 1))
        comm.allreduce_(dW)
        assert torch.all(dW == sum(range(1, world + 1)))
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e)))


def test_two_gloo_ranks_exchange_messages():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert got == {0: "ok", 1: "ok"}, got
