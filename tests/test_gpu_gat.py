"""Attention aggregator (GAT, one head) on the GPU against oracle/gat.py.

Teacher-forced stage by stage: the position maps bit-exact; Y against fp64
products of the same bf16 inputs; the forward messages of the GPU's Y
bit-exact; the attention within a bound from the fp32 score sums; H_out
within the aggregation bound given the GPU's attention; the score gradients g
within a bound from the fp32 dot products; the backward messages bit-exact
given the GPU's attention and g; the attention-vector gradients and dW /
dH_in within their bounds given the same."""
import numpy as np
import pytest

import oracle as O
from oracle import gat
from synth import planted_partition_edges, star_edges
from tests.helpers import assert_close_agg, dev, gpu_graph, host, oracle_boundary, padded

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")

GAMMA = 2.0 ** -24


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


def _bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rand_w(F_in, F_out, seed):
    rng = np.random.default_rng(seed)
    lim = np.sqrt(6.0 / (F_in + F_out))
    w = O.bf16_round(rng.uniform(-lim, lim, (F_in, F_out)).astype(np.float32))
    return (w.view(np.uint32) >> 16).astype(np.uint16)


def _graph(name, n):
    if name == "planted":
        return planted_partition_edges(n, 4 * n, 4, 0.9, 5)
    return star_edges(n, 1234)


CASES = [("planted", 4096, 100, 64, 4, [90], [2, 8], 0),
         ("star", 3000, 300, 256, 3, [80], [4, 8], 64),
         ("planted", 4096, 64, 128, 0, None, None, 32)]


@pytest.mark.parametrize("name,n,F_in,F_out,P,pct,bits,split", CASES)
def test_gat_layer(built, name, n, F_in, F_out, P, pct, bits, split):
    t = __import__("torch")
    src, dst = _graph(name, n)
    csr = gpu_graph(n, src, dst, split=split)
    rp, col, val = O.csr_build(n, src, dst)
    if P:
        b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), 1, F_out)
        if split:
            G.gnn_boundary_long_slots(csr, b, 32)
        ob = oracle_boundary(n, rp, col, val, P, pct, bits, 1, F_out)
        S, Q, sb = b.n_slots, int(ob["slot_off"][-1]), ob["slot_bits"]
        cr = ob["col_remap"]
    else:
        b, ob, S, Q, sb, cr = None, None, 0, 16, None, col
    tpos, spos = G.gnn_gat_index(csr, b)
    G.gnn_sync_check()
    assert np.array_equal(host(tpos)[:csr.nnz], gat.transpose_positions(n, rp, cr))
    if P and ob["nnz_cut"]:
        assert np.array_equal(host(spos)[:ob["nnz_cut"]], gat.slot_positions(rp, ob))

    rng = np.random.default_rng(n + F_out)
    H = rng.standard_normal((n, F_in)).astype(np.float32)
    Wb = _rand_w(F_in, F_out, 3)
    a_l = (0.3 * rng.standard_normal(F_out)).astype(np.float32)
    a_r = (0.3 * rng.standard_normal(F_out)).astype(np.float32)
    ld, ldb, ldo = G.ld_for(F_in), G.ldb_for(F_in), G.ld_for(F_out)
    packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
    meta = t.zeros((max(S, 1), 2), device="cuda")
    Hb = t.empty((n, ldb), dtype=t.bfloat16, device="cuda")
    Y = t.empty((n, ldo), device="cuda")
    alpha = t.empty(csr.nnz, device="cuda")
    Ho = t.empty((n, ldo), device="cuda")
    Wd, ald, ard = dev(Wb.view(np.int16)), dev(a_l), dev(a_r)
    G.gnn_gat_layer_fwd(csr, b, dev(padded(H, F_in, ld)), F_in, Wd, F_out, ald, ard, True, 31,
                        packed, meta, Hb, Y, alpha, Ho)
    G.gnn_sync_check()
    A = _bits_to_f32(host(Hb.view(t.int16)).view(np.uint16)[:, :F_in])
    B = _bits_to_f32(Wb)
    _, Yref = O.dense_fwd(A, B, False)
    Yg = host(Y)[:, :F_out]
    assert np.all(np.abs(Yg - Yref) <= 1e-4 * O.gemm_abs(A, B) + 1e-6)
    Ydeq = None
    if P:
        wbuf, wmeta, codes = O.quant_pack(Yg, F_out, ob["slot_node"], sb, ob["slot_off"][:-1], 31, Q)
        assert np.array_equal(host(packed)[:Q], wbuf)
        assert np.array_equal(host(meta)[:S].view(np.uint32), wmeta.view(np.uint32))
        Ydeq = O.dequantize(codes, wmeta, sb)
    # attention: bound from the fp32 score sums (F terms each) and expf
    fw = gat.forward(n, rp, col, Yg, F_out, a_l, a_r, bnd=ob, Ydeq=Ydeq)
    ag = host(alpha).astype(np.float64)
    rows = fw["rows"]
    X = fw["X_rows"]
    sl_abs = np.abs(Yg).astype(np.float64) @ np.abs(a_l.astype(np.float64))
    src_abs = np.abs(X) @ np.abs(a_r.astype(np.float64))
    dpre = 2 * F_out * GAMMA * (sl_abs[rows] + src_abs) + 1e-7
    dmax = np.zeros(n)
    np.maximum.at(dmax, rows, dpre)
    assert np.all(np.abs(ag - fw["alpha"]) <= fw["alpha"] * (4 * (dpre + dmax[rows]) + 1e-5) + 1e-8)
    assert np.allclose(np.add.reduceat(ag, rp[:-1]), 1.0, atol=1e-5)
    # H_out given the GPU's attention
    Zref = np.zeros((n, F_out))
    np.add.at(Zref, rows, ag[:, None] * X)
    T = np.zeros((n, F_out))
    np.add.at(T, rows, np.abs(ag)[:, None] * np.abs(X))
    assert_close_agg(host(Ho)[:, :F_out], np.maximum(Zref, 0), T, "gat forward")

    # ---- backward
    Hog = host(Ho)[:, :F_out]
    dHo = rng.standard_normal((n, F_out)).astype(np.float32)
    dZ = np.where(Hog > 0, dHo, np.float32(0)).astype(np.float32)
    pw = t.zeros_like(packed)
    mw = t.zeros_like(meta)
    dW = t.empty((F_in, F_out), device="cuda")
    dal = t.empty(F_out, device="cuda")
    dar = t.empty(F_out, device="cuda")
    dHi = t.empty((n, ld), device="cuda")
    g = t.empty(csr.nnz, device="cuda")
    G.gnn_gat_layer_bwd(csr, b, tpos, spos, dev(padded(dHo, F_out, ldo)), Ho, True, Hb, Y, alpha,
                        packed, meta, Wd, ald, ard, F_in, F_out, 32, pw, mw, dW, dal, dar, dHi, g)
    G.gnn_sync_check()
    gg = host(g).astype(np.float64)
    # g given the GPU's attention: bound from the fp32 dot products
    fw_t = dict(fw, alpha=ag)
    bs = gat.backward_scores(n, rp, fw_t, dZ, F_out)
    Bk = 2 * F_out * GAMMA * np.einsum("kf,kf->k", np.abs(dZ.astype(np.float64))[rows], np.abs(X))
    Cv = np.zeros(n)
    np.add.at(Cv, rows, ag * Bk + 64 * GAMMA * ag * np.abs(bs["dalpha"]))
    near0 = np.abs(fw["pre"]) < 1e-4
    tol = 2 * ag * (Bk + Cv[rows]) + 1e-9
    ok = (np.abs(gg - bs["g"]) <= tol) | near0
    assert np.all(ok), f"{int((~ok).sum())} score gradients out of bound"
    # backward messages given the GPU's attention and g, bit-exact
    if P:
        P32, r32 = gat.slot_messages_bwd(rp, ob, dZ, F_out, a_r, host(alpha), host(g))
        bcodes, bmeta = O.quantize(P32, sb, np.arange(S), 32)
        bbuf = O.pack(bcodes, sb, F_out, ob["slot_off"][:-1], Q)
        assert np.array_equal(host(pw)[:Q], bbuf)
        assert np.array_equal(host(mw)[:S].view(np.uint32), bmeta.view(np.uint32))
        bdeq = O.dequantize(bcodes, bmeta, sb).astype(np.float64)
    # dY, da_l, da_r given the GPU's attention, g and messages (fp64)
    cr64 = np.asarray(cr, np.int64)
    local = cr64 >= 0
    dY = np.zeros((n, F_out))
    np.add.at(dY, cr64[local], ag[local, None] * dZ.astype(np.float64)[rows[local]])
    ds_r = np.zeros(n)
    np.add.at(ds_r, cr64[local], gg[local])
    ds_l = np.zeros(n)
    np.add.at(ds_l, rows, gg)
    dY += np.outer(ds_r, a_r) + np.outer(ds_l, a_l)
    da_r = ds_r @ Yg.astype(np.float64)
    if P:
        np.add.at(dY, ob["slot_node"].astype(np.int64), bdeq)
        da_r += r32.astype(np.float64) @ Ydeq.astype(np.float64)
    da_l = ds_l @ Yg.astype(np.float64)
    sc_l = np.abs(ds_l) @ np.abs(Yg).astype(np.float64)
    sc_r = np.abs(ds_r) @ np.abs(Yg).astype(np.float64) + (
        np.abs(r32).astype(np.float64) @ np.abs(Ydeq) if P else 0)
    assert np.all(np.abs(host(dal) - da_l) <= 1e-5 * sc_l + 1e-7)
    assert np.all(np.abs(host(dar) - da_r) <= 1e-5 * sc_r + 1e-7)
    # dense backward of dY (bf16 rounding of dY: the bf16-path bound)
    dW_ref = A.T.astype(np.float64) @ dY
    assert np.all(np.abs(host(dW) - dW_ref) <= 2e-2 * O.gemm_abs(A.T, np.abs(dY)) + 1e-5)
    dH_ref = dY @ B.T.astype(np.float64)
    assert np.all(np.abs(host(dHi)[:, :F_in] - dH_ref) <= 2e-2 * O.gemm_abs(np.abs(dY), B.T) + 1e-5)
