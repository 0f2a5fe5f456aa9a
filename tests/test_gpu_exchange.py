"""The multi-rank path on one GPU: W virtual ranks over P partitions, each
producing only its own message rows with the slot-range kernels
(gnn_quant_pack_slots for the forward rows of the slots whose nodes it owns,
gnn_halo_quant_pack_slots for the backward rows of the slots its partitions
receive), exchanged by the all-to-all data movement of
sparse_aggregation_message_gb300.exchange.  Each rank's aggregation over its
own rows must equal the single-process path bit for bit, and so must every
message row it reads.  A world-size-1 NCCL group runs the same exchange
code through torch.distributed."""
import os
import socket

import numpy as np
import pytest

from tests.helpers import dev, gpu_graph, host, padded
from synth import planted_partition_edges

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")
from sparse_aggregation_message_gb300.exchange import (DistComm, ExchangePlan,  # noqa: E402
                                                       LocalGroup, exchange)


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


def _setup(n, m, P, F, split):
    s, d = planted_partition_edges(n, m, P, 0.8, 31)
    csr = gpu_graph(n, s, d, split=split)
    b = G.gnn_boundary_index(csr, P, G.BitRule([50, 80], [1, 4, 8]), 1, F)
    if split:
        G.gnn_boundary_long_slots(csr, b, 32)
    return csr, b


def _ref(csr, b, Hd, Gd, F, seeds):
    t = __import__("torch")
    S = b.n_slots
    Q = int(b.slot_off[-1].item())
    fp, fm = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda"), t.zeros((S, 2), device="cuda")
    G.gnn_quant_pack(Hd, F, b.slot_node, S, b.slot_bits, b.slot_off, seeds[0], fp, fm)
    M = t.empty_like(Hd)
    G.gnn_spmm_fwd(csr, b, Hd, F, fp, fm, M=M)
    hp, hm = t.zeros_like(fp), t.zeros_like(fm)
    G.gnn_halo_quant_pack(b, Gd, F, seeds[1], hp, hm)
    dH = t.empty_like(Gd)
    G.gnn_spmm_bwd_local(csr, b, Gd, F, hp, hm, dH)
    G.gnn_sync_check()
    return fp, fm, M, hp, hm, dH


@pytest.mark.parametrize("n,m,P,W,F,split", [(2000, 12000, 8, 4, 64, 0), (3000, 20000, 6, 3, 100, 32),
                                             (1500, 9000, 5, 5, 16, 0), (2500, 15000, 8, 2, 300, 32)])
def test_virtual_ranks_match_single_process(built, n, m, P, W, F, split):
    t = __import__("torch")
    csr, b = _setup(n, m, P, F, split)
    S = b.n_slots
    off = host(b.slot_off)
    part = host(b.part_start)
    plan = ExchangePlan(part, host(b.send_start), host(b.slot_node), W)
    rng = np.random.default_rng(n + F)
    ld = G.ld_for(F)
    Hd = dev(padded(rng.standard_normal((n, F)).astype(np.float32), F, ld))
    Gd = dev(padded(rng.standard_normal((n, F)).astype(np.float32), F, ld))
    fp, fm, M, hp, hm, dH = _ref(csr, b, Hd, Gd, F, (21, 22))
    Q = int(off[-1])
    grp = LocalGroup(W)
    # forward: each rank quantises the slots whose nodes it owns
    bufs = [(t.zeros(max(Q, 16), dtype=t.uint8, device="cuda"), t.zeros((S, 2), device="cuda"))
            for _ in range(W)]
    for r in range(W):
        for a, z in plan.owned(r):
            G.gnn_quant_pack_slots(Hd, F, b.slot_node, a, z, b.slot_bits, b.slot_off, 21, *bufs[r])
    grp.exchange_all(plan, [x[0] for x in bufs], [x[1] for x in bufs], off, "fwd")
    for r in range(W):
        a, z = plan.received(r)
        assert t.equal(bufs[r][0][off[a]:off[z]], fp[off[a]:off[z]]), f"rank {r} forward bytes"
        assert t.equal(bufs[r][1][a:z], fm[a:z]), f"rank {r} forward meta"
        Mr = t.empty_like(Hd)
        G.gnn_spmm_fwd(csr, b, Hd, F, bufs[r][0], bufs[r][1], M=Mr)
        r0, r1 = int(part[plan.rank_parts[r][0]]), int(part[plan.rank_parts[r][1]])
        assert t.equal(Mr[r0:r1], M[r0:r1]), f"rank {r} forward aggregation"
    # backward: each rank forms the messages of the slots its partitions receive
    bufs = [(t.zeros(max(Q, 16), dtype=t.uint8, device="cuda"), t.zeros((S, 2), device="cuda"))
            for _ in range(W)]
    for r in range(W):
        a, z = plan.received(r)
        G.gnn_halo_quant_pack_slots(b, Gd, F, a, z, 22, *bufs[r])
    grp.exchange_all(plan, [x[0] for x in bufs], [x[1] for x in bufs], off, "bwd")
    for r in range(W):
        for a, z in plan.owned(r):
            assert t.equal(bufs[r][0][off[a]:off[z]], hp[off[a]:off[z]]), f"rank {r} backward bytes"
            assert t.equal(bufs[r][1][a:z], hm[a:z]), f"rank {r} backward meta"
        dHr = t.empty_like(Gd)
        G.gnn_spmm_bwd_local(csr, b, Gd, F, bufs[r][0], bufs[r][1], dHr)
        r0, r1 = int(part[plan.rank_parts[r][0]]), int(part[plan.rank_parts[r][1]])
        assert t.equal(dHr[r0:r1], dH[r0:r1]), f"rank {r} backward aggregation"
    G.gnn_sync_check()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_world_one_through_nccl(built):
    """torch.distributed with one NCCL rank: the exchange moves nothing and
    the rank's buffer is the single-process one."""
    t = __import__("torch")
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        n, P, F = 2000, 8, 64
        csr, b = _setup(n, 12000, P, F, 0)
        S = b.n_slots
        off = host(b.slot_off)
        plan = ExchangePlan(host(b.part_start), host(b.send_start), host(b.slot_node), 1)
        rng = np.random.default_rng(5)
        ld = G.ld_for(F)
        Hd = dev(padded(rng.standard_normal((n, F)).astype(np.float32), F, ld))
        Gd = dev(padded(rng.standard_normal((n, F)).astype(np.float32), F, ld))
        fp, fm, M, hp, hm, dH = _ref(csr, b, Hd, Gd, F, (3, 4))
        comm = DistComm()
        p, mt = t.zeros_like(fp), t.zeros_like(fm)
        for a, z in plan.owned(0):
            G.gnn_quant_pack_slots(Hd, F, b.slot_node, a, z, b.slot_bits, b.slot_off, 3, p, mt)
        exchange(plan, comm, p, mt, off, "fwd")
        assert t.equal(p, fp) and t.equal(mt, fm)
        dW = t.full((4, 4), 2.0, device="cuda")
        comm.allreduce_(dW)
        assert t.all(dW == 2.0)
    finally:
        dist.destroy_process_group()
