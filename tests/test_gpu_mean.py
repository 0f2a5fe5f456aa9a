"""The GraphSAGE mean aggregator (weights 1/d_v) on the same quantised path:
CSR weights and their A^T weights bit-exact, the boundary's reordered A^T
weights bit-exact, forward and backward aggregation (plain and partitioned,
with and without split plans and long slots) against the oracle, messages
bit-exact."""
import numpy as np
import pytest

import oracle as O
from tests.helpers import assert_close_agg, dev, gpu_graph, host, oracle_boundary, padded
from tests.test_gpu_parity import GRAPHS

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")

MEAN = O.FLAGS_GCN | O.FLAG_MEAN


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


def _features(n, F, seed):
    return np.random.default_rng(seed).standard_normal((n, F)).astype(np.float32)


@pytest.mark.parametrize("name", ["er5", "er64", "er300", "planted", "star", "empty"])
def test_mean_csr_bit_exact(built, name):
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, flags=MEAN)
    rp, col, val = O.csr_build(n, src, dst, MEAN)
    assert not csr.symmetric
    assert np.array_equal(host(csr.rowptr), rp)
    assert np.array_equal(host(csr.col), col)
    assert np.array_equal(host(csr.val).view(np.uint32), val.view(np.uint32))
    vt = O.transpose_values(n, rp, col, val)
    assert csr.val_t is not None
    assert np.array_equal(host(csr.val_t).view(np.uint32), vt.view(np.uint32))


def test_mean_without_symmetrize_has_no_transpose(built):
    n, src, dst = GRAPHS["er64"]
    csr = gpu_graph(n, src, dst, flags=O.FLAG_DEDUP | O.FLAG_SELF_LOOPS | O.FLAG_MEAN)
    assert csr.val_t is None and not csr.symmetric
    t = __import__("torch")
    Gm = t.zeros((n, 8), device="cuda")
    with pytest.raises(G.GnnError):
        G.gnn_spmm_bwd(csr, None, Gm, 8, 0, None, None, t.empty_like(Gm))


@pytest.mark.parametrize("name,F,split", [("er64", 16, 0), ("star", 300, 0), ("star", 300, 64),
                                          ("er300", 129, 32), ("planted", 100, 0)])
def test_mean_plain_fwd_bwd(built, name, F, split):
    t = __import__("torch")
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, flags=MEAN, split=split)
    rp, col, val = O.csr_build(n, src, dst, MEAN)
    ld = G.ld_for(F)
    H = _features(n, F, 3)
    M = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_fwd(csr, None, dev(padded(H, F, ld)), F, M=M)
    dH = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_bwd(csr, None, dev(padded(H, F, ld)), F, 0, None, None, dH)
    G.gnn_sync_check()
    ref, T = O.spmm_fwd(n, rp, col, val, H, F)
    assert_close_agg(host(M)[:, :F], ref, T, "mean forward")
    ref, T = O.spmm_bwd(n, rp, col, val, H, F)
    assert_close_agg(host(dH)[:, :F], ref, T, "mean backward")


CASES = [("planted", 4, [90], [2, 8], 16, 0), ("er300", 7, [25, 50, 75], [1, 2, 4, 8], 37, 0),
         ("star", 3, [80], [4, 8], 300, 64), ("er300", 3, [90], [2, 8], 129, 32),
         ("er64", 5, [50], [1, 8], 602, 0)]


@pytest.mark.parametrize("name,P,pct,bits,F,split", CASES)
def test_mean_partitioned(built, name, P, pct, bits, F, split):
    t = __import__("torch")
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, flags=MEAN, split=split)
    b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), 1, F)
    if split:
        G.gnn_boundary_long_slots(csr, b, 32)
    rp, col, val = O.csr_build(n, src, dst, MEAN)
    vt = O.transpose_values(n, rp, col, val)
    ob = oracle_boundary(n, rp, col, val, P, pct, bits, 1, F, val_t=vt)
    assert np.array_equal(host(b.val_remap).view(np.uint32), ob["val_remap"].view(np.uint32))
    assert np.array_equal(host(b.val_remap_t).view(np.uint32), ob["val_remap_t"].view(np.uint32))
    assert np.array_equal(host(b.slot_val).view(np.uint32), ob["slot_val"].view(np.uint32))
    S, Q, sb = b.n_slots, int(ob["slot_off"][-1]), ob["slot_bits"]
    ld = G.ld_for(F)
    H = _features(n, F, 5)
    Hd = dev(padded(H, F, ld))
    packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
    meta = t.zeros((max(S, 1), 2), device="cuda")
    G.gnn_quant_pack(Hd, F, b.slot_node, S, b.slot_bits, b.slot_off, 4, packed, meta)
    M = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_fwd(csr, b, Hd, F, packed, meta, M=M)
    pw = t.zeros_like(packed)
    mw = t.zeros_like(meta)
    dH = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_spmm_bwd(csr, b, Hd, F, 5, pw, mw, dH)
    G.gnn_sync_check()
    ref, T = O.spmm_fwd(n, rp, col, val, H, F, ob, sb, 4)
    assert_close_agg(host(M)[:, :F], ref, T, "mean forward partitioned")
    wbuf, wmeta, _ = O.halo_quant_pack(ob, H, F, sb, ob["slot_off"], 5)
    assert np.array_equal(host(pw)[:Q], wbuf)
    assert np.array_equal(host(mw)[:S].view(np.uint32), wmeta.view(np.uint32))
    ref, T = O.spmm_bwd(n, rp, col, val, H, F, ob, sb, 5)
    assert_close_agg(host(dH)[:, :F], ref, T, "mean backward partitioned")
    # a boundary without the A^T weights is refused for the backward
    b.arrays.pop("val_remap_t")
    with pytest.raises(G.GnnError):
        G.gnn_spmm_bwd(csr, b, Hd, F, 5, pw, mw, dH)
