"""Transform-first layers (A (H W) = (A H) W, aggregation at width F_out):
bf16 copy of the input bit-exact, the transform against fp64 products of the
same bf16 inputs, the messages of Y bit-exact, the activated aggregation
within |d| <= 1e-5*sum|terms| + 1e-7 (ReLU is 1-Lipschitz), the backward
messages bit-exact, and dW / dH_in equal to the standalone dense backward of
the same dY; plus agreement with the aggregate-first layer on the same
inputs within the bf16-path bound."""
import numpy as np
import pytest

import oracle as O
from synth import planted_partition_edges, star_edges
from tests.helpers import assert_close_agg, dev, gpu_graph, host, oracle_boundary, padded

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")


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


CASES = [("planted", 4096, 100, 64, 4, [90], [2, 8], 0, True),
         ("star", 3000, 602, 128, 3, [80], [4, 8], 64, True),
         ("planted", 4096, 300, 32, 4, [25, 50, 75], [1, 2, 4, 8], 32, False)]


@pytest.mark.parametrize("name,n,F_in,F_out,P,pct,bits,split,relu", CASES)
def test_tf_layer(built, name, n, F_in, F_out, P, pct, bits, split, relu):
    t = __import__("torch")
    src, dst = _graph(name, n)
    csr = gpu_graph(n, src, dst, split=split)
    b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), 1, F_out)
    if split:
        G.gnn_boundary_long_slots(csr, b, split)
    rp, col, val = O.csr_build(n, src, dst)
    ob = oracle_boundary(n, rp, col, val, P, pct, bits, 1, F_out)
    S, Q, sb = b.n_slots, int(ob["slot_off"][-1]), ob["slot_bits"]
    rng = np.random.default_rng(n + F_in)
    H = rng.standard_normal((n, F_in)).astype(np.float32)
    Wb = _rand_w(F_in, F_out, 7)
    Wd = dev(Wb.view(np.int16))
    ld, ldb, ldo = G.ld_for(F_in), G.ldb_for(F_in), G.ld_for(F_out)
    packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
    meta = t.zeros((max(S, 1), 2), device="cuda")
    Hb = t.full((n, ldb), float("nan"), dtype=t.bfloat16, device="cuda")
    Y = t.full((n, ldo), float("nan"), device="cuda")
    Ho = t.full((n, ldo), float("nan"), device="cuda")
    G.gnn_layer_fwd_tf(csr, b, dev(padded(H, F_in, ld)), F_in, Wd, F_out, relu, 21, packed, meta,
                       Hb, Y, Ho)
    G.gnn_sync_check()
    # Hb = bf16(H), zero-padded
    hb = host(Hb.view(t.int16)).view(np.uint16)
    want = np.zeros((n, ldb), np.uint16)
    want[:, :F_in] = (O.bf16_round(H).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(hb, want)
    # Y against fp64 products of the same bf16 inputs
    A = _bits_to_f32(hb[:, :F_in])
    B = _bits_to_f32(Wb)
    _, Yref = O.dense_fwd(A, B, False)
    Yg = host(Y)[:, :F_out]
    assert np.all(np.abs(Yg - Yref) <= 1e-4 * O.gemm_abs(A, B) + 1e-6)
    # messages of the GPU's Y, bit-exact
    wbuf, wmeta, _ = O.quant_pack(Yg, F_out, ob["slot_node"], sb, ob["slot_off"][:-1], 21, Q)
    assert np.array_equal(host(packed)[:Q], wbuf)
    assert np.array_equal(host(meta)[:S].view(np.uint32), wmeta.view(np.uint32))
    # H_out = act(A Y)
    ref, T = O.spmm_fwd(n, rp, col, val, Yg, F_out, ob, sb, 21)
    if relu:
        ref = np.maximum(ref, 0.0)
    Hog = host(Ho)[:, :F_out]
    assert_close_agg(Hog, ref, T, "tf forward")

    # ---- backward
    dHo = rng.standard_normal((n, F_out)).astype(np.float32)
    dW = t.full((F_in, F_out), float("nan"), device="cuda")
    dHi = t.full((n, ld), float("nan"), device="cuda")
    pw = t.zeros_like(packed)
    mw = t.zeros_like(meta)
    dHo_d = dev(padded(dHo, F_out, ldo))
    G.gnn_layer_bwd_tf(csr, b, dHo_d, Ho, relu, Hb, Wd, F_in, F_out, 22, pw, mw, dW, dHi)
    # dZ exactly, then the same backward aggregation standalone (deterministic)
    dZ = np.where(Hog > 0, dHo, np.float32(0.0)).astype(np.float32) if relu else dHo
    dY = t.empty((n, ldo), device="cuda")
    pw2 = t.zeros_like(packed)
    mw2 = t.zeros_like(meta)
    G.gnn_spmm_bwd(csr, b, dev(padded(dZ, F_out, ldo)), F_out, 22, pw2, mw2, dY)
    dM2 = t.empty((n, ld), device="cuda")
    dW2 = t.empty((F_in, F_out), device="cuda")
    G.gnn_dense_bwd(Hb, n, F_in, Wd, F_out, dY, None, False, dM2, dW2)
    G.gnn_sync_check()
    assert t.equal(pw, pw2) and t.equal(mw, mw2)
    assert t.equal(dW, dW2)
    assert t.equal(dHi[:, :F_in], dM2[:, :F_in])
    bbuf, bmeta, _ = O.halo_quant_pack(ob, dZ, F_out, sb, ob["slot_off"], 22)
    assert np.array_equal(host(pw)[:Q], bbuf)
    dYref, T2 = O.spmm_bwd(n, rp, col, val, dZ, F_out, ob, sb, 22)
    dYg = host(dY)[:, :F_out]
    assert_close_agg(dYg, dYref, T2, "tf backward aggregation")
    dM_ref, dW_ref, dZb = O.dense_bwd(A, B, dYg, None, False)
    assert np.all(np.abs(host(dW) - dW_ref) <= 1e-4 * O.gemm_abs(A.T, dZb) + 1e-6)
    assert np.all(np.abs(host(dHi)[:, :F_in] - dM_ref) <= 1e-4 * O.gemm_abs(dZb, B.T) + 1e-6)
    # the first layer does without dH_in
    dW3 = t.empty((F_in, F_out), device="cuda")
    G.gnn_layer_bwd_tf(csr, b, dHo_d, Ho, relu, Hb, Wd, F_in, F_out, 22, pw, mw, dW3, None)
    G.gnn_sync_check()
    assert t.equal(dW3, dW)


def test_tf_matches_aggregate_first(built):
    """Without partitions both orders compute ReLU(A H W); they differ only in
    where bf16 rounding falls (H, or A H), so they agree within the
    bf16-path bound 2e-2 * sum|A||H||W|."""
    t = __import__("torch")
    n, F_in, F_out = 4096, 200, 48
    src, dst = _graph("planted", n)
    csr = gpu_graph(n, src, dst)
    rp, col, val = O.csr_build(n, src, dst)
    rng = np.random.default_rng(9)
    H = rng.standard_normal((n, F_in)).astype(np.float32)
    Wb = _rand_w(F_in, F_out, 8)
    Wd = dev(Wb.view(np.int16))
    Hd = dev(padded(H, F_in, G.ld_for(F_in)))
    Ho_tf = t.empty((n, G.ld_for(F_out)), device="cuda")
    Hb = t.empty((n, G.ldb_for(F_in)), dtype=t.bfloat16, device="cuda")
    Y = t.empty((n, G.ld_for(F_out)), device="cuda")
    G.gnn_layer_fwd_tf(csr, None, Hd, F_in, Wd, F_out, True, 0, None, None, Hb, Y, Ho_tf)
    Ho_af = t.empty((n, G.ld_for(F_out)), device="cuda")
    Mb = t.empty((n, G.ldb_for(F_in)), dtype=t.bfloat16, device="cuda")
    G.gnn_layer_fwd(csr, None, Hd, F_in, Wd, F_out, True, 0, None, None, Mb, Ho_af)
    G.gnn_sync_check()
    import scipy.sparse as sp
    Ad = sp.csr_matrix((np.abs(val).astype(np.float64), col, rp), shape=(n, n))
    scale = (Ad @ np.abs(H).astype(np.float64)) @ np.abs(_bits_to_f32(Wb)).astype(np.float64)
    d = np.abs(host(Ho_tf)[:, :F_out].astype(np.float64) - host(Ho_af)[:, :F_out])
    assert np.all(d <= 2e-2 * scale + 1e-6)
