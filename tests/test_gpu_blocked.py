"""Cluster-blocked aggregation: the plan's structure (every local entry in
exactly one dense tile or in the residual, residual order kept, dense tiles at
least min_entries entries and every other tile below it, tile row offsets
consistent), and the forward and backward against the oracle on dense and
sparse graphs, with and without partitions, split plans and several column
slices; the backward messages equal gnn_spmm_bwd's bit for bit and the gated
bf16 output equals bf16 of the fp32 output under the gate."""
import numpy as np
import pytest

import oracle as O
from synth import erdos_renyi_edges, planted_partition_edges, star_edges
from tests.helpers import assert_close_agg, dev, gpu_graph, host, oracle_boundary, padded

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")

T = 128


def _graphs():
    yield "dense", 4096, *planted_partition_edges(4096, 100000, 4, 0.95, 21)
    yield "star", 3000, *star_edges(3000, 1234)
    yield "er300", 300, *erdos_renyi_edges(300, 0.3, 4)


GRAPHS = {g[0]: g[1:] for g in _graphs()}


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


def _check_plan(bl, n, rp, cr, lc, val, min_entries):
    rows = O.csr_rows(rp)
    cr = np.asarray(cr, np.int64)
    local = np.ones(cr.size, bool) if lc is None else (np.arange(cr.size) - rp[rows]) < lc[rows]
    nb = (n + T - 1) // T
    tile = np.where(local, (rows // T) * nb + np.maximum(cr, 0) // T, -1)
    ids, cnt = np.unique(tile[local], return_counts=True)
    dense_ids = ids[cnt >= min_entries]
    assert bl.n_tiles == dense_ids.size
    in_dense = local & np.isin(tile, dense_ids)
    assert bl.n_entries == int(in_dense.sum())
    a = bl.arrays
    if bl.n_tiles:
        tcb = host(a["tile_cb"])[:bl.n_tiles]
        rbp = host(a["rb_tile_ptr"])
        tid = np.repeat(np.arange(bl.n_rb), np.diff(rbp)) * nb + tcb
        assert np.array_equal(tid, dense_ids)
        tptr = host(a["tile_ptr"])
        trp = host(a["tile_rowptr"])[:bl.n_tiles * (T + 1)].reshape(bl.n_tiles, T + 1)
        ecol = host(a["ent_col"])[:bl.n_entries]
        ev = host(a["ent_val"])[:bl.n_entries]
        for t in range(bl.n_tiles):
            sel = np.flatnonzero(tile == dense_ids[t])
            order = np.lexsort((cr[sel], rows[sel]))
            sel = sel[order]
            assert tptr[t + 1] - tptr[t] == sel.size
            assert np.array_equal(ecol[tptr[t]:tptr[t + 1]], cr[sel] % T)
            assert np.array_equal(ev[tptr[t]:tptr[t + 1]].view(np.uint32), val[sel].view(np.uint32))
            rin = rows[sel] % T
            assert np.array_equal(trp[t], np.searchsorted(rin, np.arange(T + 1), side="left"))
    keep = ~in_dense
    res = bl.residual
    rrp = host(res.rowptr)
    assert np.array_equal(np.diff(rrp), np.bincount(rows[keep], minlength=n))
    assert np.array_equal(host(res.col)[:res.nnz], cr[keep].astype(np.int32))
    assert np.array_equal(host(res.val)[:res.nnz].view(np.uint32), val[keep].view(np.uint32))
    if lc is not None:
        assert np.array_equal(host(a["res_local_cnt"])[:n], np.bincount(rows[keep & local], minlength=n))


CASES = [("dense", 0, 128, 64, 0), ("dense", 4, 128, 256, 64), ("dense", 4, 300, 64, 128),
         ("dense", 0, 602, 1024, 0), ("star", 3, 100, 8, 64), ("er300", 2, 16, 4, 0),
         ("dense", 4, 64, 10 ** 9, 64)]


@pytest.mark.parametrize("name,P,F,min_entries,split", CASES)
def test_blocked(built, name, P, F, min_entries, split):
    t = __import__("torch")
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, split=split)
    rp, col, val = O.csr_build(n, src, dst)
    b, ob, Q, S = None, None, 16, 1
    if P:
        b = G.gnn_boundary_index(csr, P, G.BitRule([50], [2, 8]), 1, F)
        if split:
            G.gnn_boundary_long_slots(csr, b, 32)
        ob = oracle_boundary(n, rp, col, val, P, [50], [2, 8], 1, F)
        Q, S = max(int(ob["slot_off"][-1]), 16), max(ob["n_slots"], 1)
    bl = G.gnn_blocked_build(csr, b, min_entries, split_len=split)
    G.gnn_sync_check()
    if P:
        _check_plan(bl, n, rp, ob["col_remap"], ob["local_cnt"], ob["val_remap"], min_entries)
    else:
        _check_plan(bl, n, rp, col, None, val, min_entries)
    if name == "dense" and min_entries <= 256:
        assert bl.n_entries > csr.nnz // 2  # the dense case really is blocked

    rng = np.random.default_rng(n + F)
    ld, ldb = G.ld_for(F), G.ldb_for(F)
    H = rng.standard_normal((n, F)).astype(np.float32)
    Hd = dev(padded(H, F, ld))
    packed = t.zeros(Q, dtype=t.uint8, device="cuda")
    meta = t.zeros((S, 2), device="cuda")
    if P:
        G.gnn_quant_pack(Hd, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, 3, packed, meta)
    M = t.full((n, ld), float("nan"), device="cuda")
    Mb = t.full((n, ldb), float("nan"), dtype=t.bfloat16, device="cuda")
    G.gnn_spmm_fwd_blocked(csr, b, bl, Hd, F, packed, meta, M=M, Mb=Mb)
    G.gnn_sync_check()
    ref, Tm = O.spmm_fwd(n, rp, col, val, H, F, ob, ob["slot_bits"] if P else None, 3)
    Mh = host(M)[:, :F]
    assert_close_agg(Mh, ref, Tm, f"blocked forward {name}")
    mbh = host(Mb.view(t.int16)).view(np.uint16)
    want = np.zeros((n, ldb), np.uint16)
    want[:, :F] = (O.bf16_round(Mh).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(mbh, want)

    # backward: messages as gnn_spmm_bwd's, dH within tolerance, gated bf16 consistent
    Gm = dev(padded(rng.standard_normal((n, F)).astype(np.float32), F, ld))
    Hm = np.maximum(rng.standard_normal((n, F)), 0).astype(np.float32)
    pw1, mw1 = t.zeros_like(packed), t.zeros_like(meta)
    pw2, mw2 = t.zeros_like(packed), t.zeros_like(meta)
    dH1 = t.empty((n, ld), device="cuda")
    G.gnn_spmm_bwd(csr, b, Gm, F, 5, pw1, mw1, dH1)
    dH2 = t.full((n, ld), float("nan"), device="cuda")
    dZ = t.full((n, G.ldz_for(F)), float("nan"), dtype=t.bfloat16, device="cuda")
    G.gnn_spmm_bwd_blocked(csr, b, bl, Gm, F, 5, pw2, mw2, H_mask=dev(padded(Hm, F, ld)), dH=dH2,
                           dZ=dZ)
    G.gnn_sync_check()
    assert t.equal(pw1, pw2) and t.equal(mw1, mw2)
    Gh = host(Gm)[:, :F]
    dref, Td = O.spmm_bwd(n, rp, col, val, Gh, F, ob, ob["slot_bits"] if P else None, 5)
    dh2 = host(dH2)[:, :F]
    assert_close_agg(dh2, dref, Td, f"blocked backward {name}")
    wz = np.zeros((n, G.ldz_for(F)), np.uint16)
    wz[:, :F] = (O.bf16_round(np.where(Hm > 0, dh2, np.float32(0))).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(host(dZ.view(t.int16)).view(np.uint16), wz)
