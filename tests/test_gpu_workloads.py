"""The five synthetic workloads at full size, in the launch configuration
bench.py times (row-split plan of 128 entries, long-slot list of 128
entries, slot offsets per layer width).

Per workload: CSR, boundary index, widths and offsets bit-exact against the
oracle in full; quantised messages (forward and backward) bit-exact on a
seeded sample of slots; forward and backward aggregation on a seeded sample of
rows plus the longest (split) rows, within |d| <= 1e-5*sum|terms| + 1e-7; the
first layer's transform on the sampled rows against fp64 products of the same
bf16 inputs."""
import os

import numpy as np
import pytest

import oracle as O
from synth import make_workload
from synth.graphs import CONFIGS, make_weight_bf16
from tests.helpers import assert_close_agg, dev, host, oracle_boundary

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")

SPLIT_LEN = 128
LONG_SLOT_LEN = 128
N_SAMPLE_ROWS = 2048
N_SAMPLE_SLOTS = 4096

WORKLOADS = os.environ.get("GNN_TEST_WORKLOADS", "tiny,yelp,products,reddit,scale").split(",")


def _bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_parity(name):
    import torch as t

    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = make_workload(name)
    n, P, dims = wl.n, wl.P, wl.dims
    rng = np.random.default_rng(wl.seed + 99)

    # ---- a1: CSR (full)
    csr = G.gnn_csr_build(n, dev(wl.src), dev(wl.dst))
    csr = G.gnn_csr_split(csr, SPLIT_LEN)
    rp, col, val = O.csr_build(n, wl.src, wl.dst)
    assert csr.nnz == col.size
    assert np.array_equal(host(csr.rowptr), rp)
    assert np.array_equal(host(csr.col), col)
    assert np.array_equal(host(csr.val).view(np.uint32), val.view(np.uint32))
    del wl

    # ---- a2: boundary, widths, offsets (full), at the first base width
    F0 = dims[0]
    cfg = CONFIGS[name]
    cfg_pct, cfg_bits, base = cfg["rule"]["pct"], cfg["rule"]["bits"], cfg["base_bits"][0]
    bnd = G.gnn_boundary_index(csr, P, G.BitRule(cfg_pct, cfg_bits), base, F0)
    ob = oracle_boundary(n, rp, col, val, P, cfg_pct, cfg_bits, base, F0)
    assert (bnd.n_slots, bnd.nnz_cut) == (ob["n_slots"], ob["nnz_cut"])
    for k in ("part_start", "send_start", "slot_node", "col_remap", "local_cnt", "slot_rowptr",
              "slot_col", "own_ptr", "own_slot", "node_bits", "slot_bits", "slot_off"):
        got = host(bnd.arrays[k])
        assert np.array_equal(got, np.asarray(ob[k]).astype(got.dtype)), k
    assert np.array_equal(host(bnd.slot_val).view(np.uint32), ob["slot_val"].view(np.uint32))
    assert np.array_equal(host(bnd.val_remap).view(np.uint32), ob["val_remap"].view(np.uint32))
    S = bnd.n_slots
    sb = ob["slot_bits"]
    G.gnn_boundary_long_slots(csr, bnd, LONG_SLOT_LEN)

    # sampled rows: random plus the longest rows (those are split into pieces)
    deg = np.diff(rp)
    longest = np.argsort(-deg, kind="stable")[:32]
    rows = np.unique(np.concatenate([rng.choice(n, min(n, N_SAMPLE_ROWS), replace=False), longest]))
    slots = np.unique(rng.choice(S, min(S, N_SAMPLE_SLOTS), replace=False)) if S else np.zeros(0, np.int64)

    for li, F in enumerate(sorted(set(dims[:-1]), reverse=True)):
        ld = G.ld_for(F)
        off = ob["slot_off"] if F == F0 else O.slot_offsets(sb, F)
        off_d = bnd.slot_off if F == F0 else G.gnn_slot_offsets(bnd.slot_bits, S, F)
        assert np.array_equal(host(off_d), off)
        Q = int(off[-1])
        # layer inputs: N(0,1) features for the first width, ReLU'd N(0,1) otherwise
        g = t.Generator(device="cuda")
        g.manual_seed(1000 + F)
        Hd = t.zeros((n, ld), device="cuda")
        Hd[:, :F] = t.randn((n, F), generator=g, device="cuda")
        if F != F0:
            Hd.clamp_(min=0)
        seed_f, seed_b = 2 * li, 2 * li + 1
        packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
        meta = t.zeros((max(S, 1), 2), device="cuda")
        G.gnn_quant_pack(Hd, F, bnd.slot_node, S, bnd.slot_bits, off_d, seed_f, packed, meta)
        M = t.empty((n, ld), device="cuda")
        G.gnn_spmm_fwd(csr, bnd, Hd, F, packed, meta, M=M, slot_off=off_d)
        G.gnn_sync_check()
        # forward messages on sampled slots
        ph, mh = host(packed), host(meta)
        Hrows = host(Hd[t.from_numpy(ob["slot_node"][slots]).long().cuda()])[:, :F] if S else None
        if S:
            codes, wmeta = O.quantize(Hrows, sb[slots], slots, seed_f)
            assert np.array_equal(mh[slots].view(np.uint32), wmeta.view(np.uint32))
            for b in np.unique(sb[slots]):
                sel = slots[sb[slots] == b]
                rb = int(O.rowbytes(b, F))
                got = ph[off[sel][:, None] + np.arange(rb)[None, :]]
                want = O.pack(codes[sb[slots] == b], np.full(sel.size, b), F,
                              np.arange(sel.size) * rb, sel.size * rb).reshape(sel.size, rb)
                assert np.array_equal(got, want), f"packed bytes F={F} b={b}"
        # forward aggregation on sampled rows (the oracle quantises what they read)
        need = np.unique(np.concatenate([col[rp[r]:rp[r + 1]] for r in rows] + [rows]))
        Hh = np.zeros((n, F), np.float32)
        Hh[need] = host(Hd[t.from_numpy(need).long().cuda()])[:, :F]
        ref, T = O.spmm_fwd(n, rp, col, val, Hh, F, ob, sb, seed_f, rows=rows)
        assert_close_agg(host(M[t.from_numpy(rows).long().cuda()])[:, :F], ref, T, f"{name} fwd F={F}")

        # backward: G = the forward output (any dense matrix serves)
        dH = t.empty((n, ld), device="cuda")
        pw = t.zeros_like(packed)
        mw = t.zeros_like(meta)
        G.gnn_spmm_bwd(csr, bnd, M, F, seed_b, pw, mw, dH, slot_off=off_d)
        G.gnn_sync_check()
        ob_F = dict(ob)
        ob_F["slot_off"] = off
        # rows the sampled slots' partials and the sampled rows' owned slots read
        own = np.concatenate([ob["own_slot"][ob["own_ptr"][r]:ob["own_ptr"][r + 1]] for r in rows])
        chk = np.unique(np.concatenate([slots, own])).astype(np.int64)
        srp, scol = ob["slot_rowptr"], ob["slot_col"]
        needv = np.unique(np.concatenate([scol[srp[s]:srp[s + 1]] for s in chk] + [need])) if chk.size else need
        Gh = np.zeros((n, F), np.float32)
        Gh[needv] = host(M[t.from_numpy(needv).long().cuda()])[:, :F]
        if S:
            part = O.slot_partials(ob, Gh, F, slots)
            codes, wmeta = O.quantize(part, sb[slots], slots, seed_b)
            assert np.array_equal(host(mw)[slots].view(np.uint32), wmeta.view(np.uint32))
            pwh = host(pw)
            for b in np.unique(sb[slots]):
                sel = slots[sb[slots] == b]
                rb = int(O.rowbytes(b, F))
                got = pwh[off[sel][:, None] + np.arange(rb)[None, :]]
                want = O.pack(codes[sb[slots] == b], np.full(sel.size, b), F,
                              np.arange(sel.size) * rb, sel.size * rb).reshape(sel.size, rb)
                assert np.array_equal(got, want), f"backward packed bytes F={F} b={b}"
        dref, T2 = O.spmm_bwd(n, rp, col, val, Gh, F, ob, sb, seed_b, rows=rows)
        assert_close_agg(host(dH[t.from_numpy(rows).long().cuda()])[:, :F], dref, T2, f"{name} bwd F={F}")
        del pw, mw, dH

        # the transform of this width on the sampled rows, teacher-forced on Mb
        Fo = dims[1]
        Mb = t.empty((n, G.ldb_for(F)), dtype=t.bfloat16, device="cuda")
        packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
        meta = t.zeros((max(S, 1), 2), device="cuda")
        G.gnn_quant_pack(Hd, F, bnd.slot_node, S, bnd.slot_bits, off_d, seed_f, packed, meta)
        G.gnn_spmm_fwd(csr, bnd, Hd, F, packed, meta, Mb=Mb, slot_off=off_d)
        W = make_weight_bf16(F, Fo, 1234, li)
        Ho = t.empty((n, G.ld_for(Fo)), device="cuda")
        G.gnn_dense_fwd(Mb, n, F, dev(W.view(np.int16)), Fo, True, Ho)
        G.gnn_sync_check()
        A = _bits_to_f32(host(Mb[t.from_numpy(rows).long().cuda()].view(t.int16)).view(np.uint16))[:, :F]
        B = _bits_to_f32(W)
        _, Href = O.dense_fwd(A, B, True)
        got = host(Ho[t.from_numpy(rows).long().cuda()])[:, :Fo]
        scale = O.gemm_abs(A, B)
        assert np.all(np.abs(got - Href) <= 1e-4 * scale + 1e-6), f"{name} transform F={F}"
        del Hd, M, Mb, Ho, packed, meta
        t.cuda.empty_cache()
