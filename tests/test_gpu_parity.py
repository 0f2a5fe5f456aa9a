"""Parity of the CUDA path (called through the C ABI via the binding) with
the oracle on seeded inputs: bit-exact for indices, widths, offsets, codes,
packed bytes and meta; |d| <= 1e-5*sum|terms| + 1e-7 for aggregations."""
import numpy as np
import pytest

import oracle as O
from synth import (circulant_edges, erdos_renyi_edges, planted_partition_edges, star_edges)
from tests.helpers import assert_close_agg, dev, gpu_graph, host, oracle_boundary, padded

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")


def _graphs():
    yield "er1", 1, *erdos_renyi_edges(1, 0.0, 1)
    yield "er2", 2, np.array([0], np.int32), np.array([1], np.int32)
    yield "er5", 5, *erdos_renyi_edges(5, 0.6, 2)
    yield "er64", 64, *erdos_renyi_edges(64, 0.1, 3)
    yield "er300", 300, *erdos_renyi_edges(300, 0.05, 4)
    yield "planted", 4096, *planted_partition_edges(4096, 16384, 4, 0.9, 5)
    yield "star", 3000, *star_edges(3000, 1234)
    yield "empty", 50, np.zeros(0, np.int32), np.zeros(0, np.int32)
    yield "circ15", 256, *circulant_edges(256, 15)


GRAPHS = {g[0]: g[1:] for g in _graphs()}


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


# ------------------------------------------------------------------ a1: CSR
@pytest.mark.parametrize("name", list(GRAPHS))
def test_csr_build_bit_exact(built, name):
    n, src, dst = GRAPHS[name]
    # feed duplicates and reversed copies too
    s2 = np.concatenate([src, dst[: len(dst) // 3]]).astype(np.int32)
    d2 = np.concatenate([dst, src[: len(src) // 3]]).astype(np.int32)
    csr = gpu_graph(n, s2, d2)
    rp, col, val = O.csr_build(n, s2, d2)
    assert csr.nnz == col.size and csr.symmetric
    assert np.array_equal(host(csr.rowptr), rp)
    assert np.array_equal(host(csr.col), col)
    assert np.array_equal(host(csr.val).view(np.uint32), val.view(np.uint32))


@pytest.mark.parametrize("flags", [0, O.FLAG_SELF_LOOPS, O.FLAG_SYMMETRIZE | O.FLAG_SELF_LOOPS,
                                   O.FLAG_DEDUP, O.FLAGS_GCN])
def test_csr_build_flags(built, flags):
    rng = np.random.default_rng(flags)
    n = 40
    src = rng.integers(0, n, 300).astype(np.int32)
    dst = rng.integers(0, n, 300).astype(np.int32)
    csr = gpu_graph(n, src, dst, flags)
    rp, col, val = O.csr_build(n, src, dst, flags)
    assert np.array_equal(host(csr.rowptr), rp)
    assert np.array_equal(host(csr.col), col)
    assert np.array_equal(host(csr.val).view(np.uint32), val.view(np.uint32))
    assert csr.symmetric == bool(flags & O.FLAG_SYMMETRIZE)


def test_csr_build_rejects_out_of_range_endpoint(built):
    with pytest.raises(G.GnnError) as e:
        gpu_graph(10, np.array([0, 3], np.int32), np.array([1, 10], np.int32))
    assert e.value.status == 1


@pytest.mark.parametrize("name,split", [("star", 64), ("planted", 32), ("er300", 32), ("er1", 32),
                                        ("empty", 32)])
def test_csr_split_plan(built, name, split):
    """Long rows (more than `split` entries) are cut into consecutive pieces
    of `split` entries, in row order."""
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, split=split)
    rp, _, _ = O.csr_build(n, src, dst)
    deg = np.diff(rp)
    long_rows = np.nonzero(deg > split)[0]
    assert csr.n_long == long_rows.size
    assert np.array_equal(host(csr.split["long_rows"])[: long_rows.size], long_rows)
    pieces = [(r, b) for r in long_rows for b in range(rp[r], rp[r + 1], split)]
    assert csr.n_pieces == len(pieces)
    pp = np.concatenate([[0], np.cumsum([(deg[r] + split - 1) // split for r in long_rows])])
    assert np.array_equal(host(csr.split["piece_ptr"]), pp)
    if pieces:
        assert np.array_equal(host(csr.split["piece_row"])[: len(pieces)], [p[0] for p in pieces])
        assert np.array_equal(host(csr.split["piece_beg"])[: len(pieces)], [p[1] for p in pieces])


@pytest.mark.parametrize("name,P,T", [("star", 3, 32), ("star", 5, 100), ("planted", 4, 32),
                                      ("er300", 3, 32)])
def test_boundary_long_slot_list(built, name, P, T):
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst)
    b = G.gnn_boundary_index(csr, P, G.BitRule([50], [2, 8]), 1, 8)
    G.gnn_boundary_long_slots(csr, b, T)
    rp, col, val = O.csr_build(n, src, dst)
    ob = O.boundary_index(n, rp, col, val, P)
    want = np.nonzero(np.diff(ob["slot_rowptr"]) > T)[0]
    assert b.n_long_slots == want.size
    if want.size:
        assert np.array_equal(host(b.arrays["long_slots"])[: want.size], want)


# ------------------------------------------------------------------ a2: boundary
BND_CASES = [("er64", 4, [90], [2, 8], 1, 16), ("er300", 7, [25, 50, 75], [1, 2, 4, 8], 1, 37),
             ("planted", 4, [90], [2, 8], 1, 16), ("star", 3, [80], [4, 8], 2, 5),
             ("er5", 8, [50], [1, 8], 4, 3), ("er300", 1, [90], [2, 8], 1, 8),
             ("circ15", 16, [95], [1, 8], 8, 300), ("empty", 4, [90], [2, 8], 1, 16),
             ("planted", 4, [90], [32, 32], 1, 9)]


@pytest.mark.parametrize("name,P,pct,bits,base,F", BND_CASES)
def test_boundary_index_bit_exact(built, name, P, pct, bits, base, F):
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst)
    b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), base, F)
    rp, col, val = O.csr_build(n, src, dst)
    ob = oracle_boundary(n, rp, col, val, P, pct, bits, base, F)
    assert (b.n_slots, b.nnz_cut) == (ob["n_slots"], ob["nnz_cut"])
    for k in ("part_start", "send_start", "slot_node", "col_remap", "local_cnt", "slot_rowptr",
              "slot_col", "own_ptr", "own_slot", "node_bits", "slot_bits", "slot_off"):
        got = host(b.arrays[k])
        want = np.asarray(ob[k])
        assert np.array_equal(got, want.astype(got.dtype)), k
    assert np.array_equal(host(b.slot_val).view(np.uint32), ob["slot_val"].view(np.uint32))
    assert np.array_equal(host(b.val_remap).view(np.uint32), ob["val_remap"].view(np.uint32))
    # base-width change recomputes widths and offsets only
    G.gnn_boundary_set_bits(csr, b, G.BitRule(pct, bits), 8, F + 3)
    nb8 = O.node_bits(n, rp, ob, pct, bits, 8)
    assert np.array_equal(host(b.node_bits), nb8)
    sb8 = nb8[ob["slot_node"]] if ob["n_slots"] else np.zeros(0, np.uint8)
    assert np.array_equal(host(b.slot_off), O.slot_offsets(sb8, F + 3))


# ------------------------------------------------------------------ a3: quantise + pack
def _messy_rows(R, F, seed):
    rng = np.random.default_rng(seed)
    X = (rng.standard_normal((R, F)) * rng.uniform(0.01, 100, (R, 1))).astype(np.float32)
    X[0] = 3.25                       # constant row
    if R > 1:
        X[1] = 0.0
        X[1, ::2] = -0.0              # signed zeros
    if R > 2:
        X[2] = np.round(X[2])         # integers
    if R > 3:
        X[3] = np.abs(X[3])           # min > 0
    if R > 4:
        X[4, :] = 1e-39 * np.arange(F, dtype=np.float32)  # subnormals
    return X


@pytest.mark.parametrize("F", [1, 3, 5, 16, 37, 100, 128, 129, 256, 300, 602, 1024])
def test_quant_pack_bit_exact(built, F):
    R = 257
    rng = np.random.default_rng(F)
    X = _messy_rows(R + 40, F, F)
    ld = G.ld_for(F)
    row_idx = rng.permutation(R + 40)[:R].astype(np.int32)
    bits = rng.choice([1, 2, 4, 8, 32], R).astype(np.uint8)
    off = O.slot_offsets(bits, F)
    seed = 0xC0FFEE + F
    want_buf, want_meta, _ = O.quant_pack(X, F, row_idx, bits, off[:-1], seed, int(off[-1]))
    t = __import__("torch")
    Xd = dev(padded(X, F, ld))
    packed = t.full((int(off[-1]),), 0xAB, dtype=t.uint8, device="cuda")
    meta = t.full((R, 2), float("nan"), dtype=t.float32, device="cuda")
    G.gnn_quant_pack(Xd, F, dev(row_idx), R, dev(bits), dev(off), seed, packed, meta)
    G.gnn_sync_check()
    assert np.array_equal(host(packed), want_buf)
    assert np.array_equal(host(meta).view(np.uint32), want_meta.view(np.uint32))
    # identity row map, then the receive side
    packed2 = t.zeros_like(packed)
    meta2 = t.zeros_like(meta)
    G.gnn_quant_pack(Xd, F, None, R, dev(bits), dev(off), seed, packed2, meta2)
    want2, wmeta2, codes2 = O.quant_pack(X, F, np.arange(R), bits, off[:-1], seed, int(off[-1]))
    assert np.array_equal(host(packed2), want2)
    out = t.full((R, ld), float("nan"), dtype=t.float32, device="cuda")
    G.gnn_dequant_unpack(packed2, meta2, dev(off), dev(bits), R, F, out)
    deq = O.dequantize(O.unpack(want2, bits, F, off[:-1]), wmeta2, bits)
    got = host(out)
    assert np.array_equal(got[:, :F].view(np.uint32), deq.view(np.uint32))
    assert np.all(got[:, F:ld] == 0)


def test_quant_pack_zero_rows_is_noop(built):
    t = __import__("torch")
    X = t.zeros((4, 4), device="cuda")
    G.gnn_quant_pack(X, 4, None, 0, None, None, 1, None, None)


# ------------------------------------------------------------------ a4: forward aggregation
def _features(n, F, seed):
    return np.random.default_rng(seed).standard_normal((n, F)).astype(np.float32)


@pytest.mark.parametrize("name,F,split", [("er1", 4, 0), ("er5", 3, 0), ("er64", 16, 0),
                                          ("er300", 37, 0), ("planted", 16, 0), ("star", 100, 0),
                                          ("star", 602, 0), ("empty", 8, 0), ("er300", 300, 0),
                                          ("er300", 1024, 0), ("star", 100, 64), ("star", 16, 32),
                                          ("star", 602, 100), ("planted", 16, 32), ("er300", 300, 32)])
def test_spmm_fwd_plain(built, name, F, split):
    t = __import__("torch")
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, split=split)
    rp, col, val = O.csr_build(n, src, dst)
    H = _features(n, F, 7)
    ld, ldb = G.ld_for(F), G.ldb_for(F)
    M = t.full((n, ld), float("nan"), device="cuda")
    Mb = t.full((n, ldb), float("nan"), dtype=t.bfloat16, device="cuda")
    G.gnn_spmm_fwd(csr, None, dev(padded(H, F, ld)), F, M=M, Mb=Mb)
    G.gnn_sync_check()
    ref, T = O.spmm_fwd(n, rp, col, val, H, F)
    got = host(M)
    assert_close_agg(got[:, :F], ref, T, f"spmm_fwd {name} F={F}")
    assert np.all(got[:, F:] == 0)
    mb = host(Mb.view(t.int16)).view(np.uint16)
    want_b = (O.bf16_round(got[:, :F]).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(mb[:, :F], want_b)
    assert np.all(mb[:, F:] == 0)


def _partitioned_setup(name, P, pct, bits, base, F, seed, split=0, long_slots=0):
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, split=split)
    b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), base, F)
    if long_slots:
        G.gnn_boundary_long_slots(csr, b, long_slots)
    rp, col, val = O.csr_build(n, src, dst)
    ob = oracle_boundary(n, rp, col, val, P, pct, bits, base, F)
    return n, csr, b, rp, col, val, ob


PART_CASES = [("planted", 4, [90], [2, 8], 1, 16, 0), ("er300", 7, [25, 50, 75], [1, 2, 4, 8], 1, 37, 0),
              ("star", 3, [80], [4, 8], 1, 300, 0), ("er64", 5, [50], [1, 8], 2, 602, 0),
              ("er300", 3, [90], [2, 8], 1, 129, 0), ("er5", 8, [50], [1, 8], 1, 3, 0),
              ("star", 3, [80], [4, 8], 1, 300, 64), ("star", 5, [50], [1, 8], 1, 16, 32),
              ("planted", 4, [90], [2, 8], 1, 16, 32), ("er300", 7, [25, 50, 75], [1, 2, 4, 8], 1, 602, 32)]


@pytest.mark.parametrize("name,P,pct,bits,base,F,split", PART_CASES)
def test_spmm_fwd_partitioned(built, name, P, pct, bits, base, F, split):
    t = __import__("torch")
    n, csr, b, rp, col, val, ob = _partitioned_setup(name, P, pct, bits, base, F, 0, split)
    H = _features(n, F, 11)
    ld = G.ld_for(F)
    Hd = dev(padded(H, F, ld))
    seed = 2 * 1
    Q = int(ob["slot_off"][-1])
    packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
    meta = t.zeros((max(b.n_slots, 1), 2), dtype=t.float32, device="cuda")
    G.gnn_quant_pack(Hd, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, seed, packed, meta)
    M = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_fwd(csr, b, Hd, F, packed, meta, M=M)
    G.gnn_sync_check()
    wbuf, wmeta, _ = O.quant_pack(H, F, ob["slot_node"], ob["slot_bits"], ob["slot_off"][:-1], seed, Q)
    assert np.array_equal(host(packed)[:Q], wbuf)
    assert np.array_equal(host(meta)[: b.n_slots].view(np.uint32), wmeta.view(np.uint32))
    ref, T = O.spmm_fwd(n, rp, col, val, H, F, ob, ob["slot_bits"], seed)
    assert_close_agg(host(M)[:, :F], ref, T, f"spmm_fwd partitioned {name}")


def test_spmm_fwd_passthrough_equals_plain(built):
    """Width 32 sends exact rows, so the partitioned forward reproduces the
    plain one up to the order of the fp32 additions (the partitioned layout
    adds a row's local entries before its remote ones)."""
    t = __import__("torch")
    n, csr, b, rp, col, val, ob = _partitioned_setup("planted", 4, [90], [32, 32], 1, 24, 0)
    H = dev(padded(_features(n, 24, 3), 24, 24))
    Q = int(ob["slot_off"][-1])
    packed = t.zeros(Q, dtype=t.uint8, device="cuda")
    meta = t.zeros((b.n_slots, 2), device="cuda")
    G.gnn_quant_pack(H, 24, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, 5, packed, meta)
    M1 = t.empty((n, 24), device="cuda")
    M0 = t.empty((n, 24), device="cuda")
    G.gnn_spmm_fwd(csr, b, H, 24, packed, meta, M=M1)
    G.gnn_spmm_fwd(csr, None, H, 24, M=M0)
    _, T = O.spmm_fwd(n, rp, col, val, host(H), 24)
    err = np.abs(host(M1).astype(np.float64) - host(M0))
    assert np.all(err <= 2e-5 * T + 2e-7)


@pytest.mark.parametrize("P", [1, 4])
def test_regular_graph_constant_features_fixed_point(built, P):
    """d-regular graph, d+1 = 16: constant features come back bit-exactly.
    Unpartitioned, every column may hold its own constant; with quantised
    partitions each row must be constant too (then its scale is 0 and the
    message is exact)."""
    t = __import__("torch")
    n, F = 256, 8
    src, dst = circulant_edges(n, 15)
    csr = gpu_graph(n, src, dst)
    if P == 1:
        H = np.tile(np.array([0.75, -3.0, 0.0, 1e-3, 7.5, -0.125, 2.0, 5.0], np.float32), (n, 1))
    else:
        H = np.full((n, F), -2.375, np.float32)
    Hd = dev(H)
    M = t.empty((n, F), device="cuda")
    if P == 1:
        G.gnn_spmm_fwd(csr, None, Hd, F, M=M)
    else:
        b = G.gnn_boundary_index(csr, P, G.BitRule([50], [1, 2]), 1, F)
        Q = int(host(b.slot_off)[-1])
        packed = t.zeros(Q, dtype=t.uint8, device="cuda")
        meta = t.zeros((b.n_slots, 2), device="cuda")
        G.gnn_quant_pack(Hd, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, 9, packed, meta)
        G.gnn_spmm_fwd(csr, b, Hd, F, packed, meta, M=M)
    assert np.array_equal(host(M), H)


# ------------------------------------------------------------------ a7/a8: backward aggregation
@pytest.mark.parametrize("name,F,split", [("er64", 16, 0), ("planted", 16, 0), ("star", 300, 0),
                                          ("er300", 129, 0), ("star", 300, 64), ("er300", 129, 32)])
def test_spmm_bwd_plain(built, name, F, split):
    t = __import__("torch")
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, split=split)
    rp, col, val = O.csr_build(n, src, dst)
    Gm = _features(n, F, 21)
    ld = G.ld_for(F)
    dH = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_bwd(csr, None, dev(padded(Gm, F, ld)), F, 0, None, None, dH)
    G.gnn_sync_check()
    ref, T = O.spmm_bwd(n, rp, col, val, Gm, F)
    assert_close_agg(host(dH)[:, :F], ref, T, f"spmm_bwd {name}")


@pytest.mark.parametrize("name,P,pct,bits,base,F,split", PART_CASES)
def test_spmm_bwd_partitioned(built, name, P, pct, bits, base, F, split):
    """With a split plan the long slots (more than 32 entries) are also summed
    by whole blocks; the messages must not change."""
    t = __import__("torch")
    n, csr, b, rp, col, val, ob = _partitioned_setup(name, P, pct, bits, base, F, 0, split,
                                                     long_slots=32 if split else 0)
    Gm = _features(n, F, 31)
    ld = G.ld_for(F)
    Q = int(ob["slot_off"][-1])
    seed = 2 * 1 + 1
    pw = t.full((max(Q, 16),), 0xCD, dtype=t.uint8, device="cuda")
    mw = t.zeros((max(b.n_slots, 1), 2), device="cuda")
    dH = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_bwd(csr, b, dev(padded(Gm, F, ld)), F, seed, pw, mw, dH)
    G.gnn_sync_check()
    wbuf, wmeta, _ = O.halo_quant_pack(ob, Gm, F, ob["slot_bits"], ob["slot_off"], seed)
    assert np.array_equal(host(pw)[:Q], wbuf)
    assert np.array_equal(host(mw)[: b.n_slots].view(np.uint32), wmeta.view(np.uint32))
    ref, T = O.spmm_bwd(n, rp, col, val, Gm, F, ob, ob["slot_bits"], seed)
    assert_close_agg(host(dH)[:, :F], ref, T, f"spmm_bwd partitioned {name}")


def test_adjoint_identity_on_gpu(built):
    """<A H, G> = <H, A^T G> with the GPU's plain forward and backward."""
    t = __import__("torch")
    n, src, dst = GRAPHS["planted"]
    csr = gpu_graph(n, src, dst)
    F = 32
    H = _features(n, F, 1)
    Gm = _features(n, F, 2)
    M = t.empty((n, F), device="cuda")
    dH = t.empty((n, F), device="cuda")
    G.gnn_spmm_fwd(csr, None, dev(H), F, M=M)
    G.gnn_spmm_bwd(csr, None, dev(Gm), F, 0, None, None, dH)
    lhs = float(np.sum(host(M).astype(np.float64) * Gm))
    rhs = float(np.sum(H.astype(np.float64) * host(dH)))
    scale = float(np.sum(np.abs(host(M)) * np.abs(Gm)))
    assert abs(lhs - rhs) <= 1e-5 * scale
