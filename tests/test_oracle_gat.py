"""Pins of the attention-aggregator oracle (oracle/gat.py): brute-force
attention on tiny graphs, the backward against central finite differences of
a linear loss, the partitioned forms reducing to the plain ones when the
messages are raw fp32 rows, and softmax invariants."""
import numpy as np
import pytest

import oracle as O
from oracle import gat
from synth import erdos_renyi_edges, planted_partition_edges


def _setup(n, p, seed, F):
    src, dst = erdos_renyi_edges(n, p, seed)
    rp, col, val = O.csr_build(n, src, dst)
    rng = np.random.default_rng(seed)
    Y = rng.standard_normal((n, F))
    a_l = rng.standard_normal(F) * 0.5
    a_r = rng.standard_normal(F) * 0.5
    return rp, col, Y, a_l, a_r, rng


@pytest.mark.parametrize("n,p,seed", [(6, 0.5, 1), (12, 0.3, 2)])
def test_attention_bruteforce(n, p, seed):
    F = 3
    rp, col, Y, a_l, a_r, _ = _setup(n, p, seed, F)
    fw = gat.forward(n, rp, col, Y, F, a_l, a_r)
    for v in range(n):
        nb = [int(u) for u in col[rp[v]:rp[v + 1]]]
        assert v in nb  # the self-loop
        e = []
        for u in nb:
            x = float(Y[v] @ a_l + Y[u] @ a_r)
            e.append(x if x > 0 else 0.2 * x)
        w = np.exp(np.array(e) - max(e))
        alpha = w / w.sum()
        assert np.allclose(fw["alpha"][rp[v]:rp[v + 1]], alpha, rtol=1e-13, atol=0)
        z = sum(a * Y[u] for a, u in zip(alpha, nb))
        assert np.allclose(fw["Z"][v], z, rtol=1e-12, atol=1e-14)


def test_softmax_invariants():
    n, F = 40, 4
    rp, col, Y, a_l, a_r, _ = _setup(n, 0.2, 3, F)
    fw = gat.forward(n, rp, col, Y, F, a_l, a_r)
    sums = np.add.reduceat(fw["alpha"], rp[:-1])
    assert np.allclose(sums, 1.0, atol=1e-14) and np.all(fw["alpha"] >= 0)
    # a_l shifts every score of a row equally only through LeakyReLU; with
    # a_l = 0 and a constant Y the attention is uniform
    fw2 = gat.forward(n, rp, col, np.ones((n, F)), F, np.zeros(F), a_r)
    assert np.allclose(fw2["alpha"], np.repeat(1.0 / np.diff(rp), np.diff(rp)))


@pytest.mark.parametrize("seed", [4, 5])
def test_backward_finite_differences(seed):
    """L = sum(Gz * Z): dY, da_l, da_r against central differences."""
    n, F = 9, 3
    rp, col, Y, a_l, a_r, rng = _setup(n, 0.45, seed, F)
    Gz = rng.standard_normal((n, F))

    def loss(Y_, al, ar):
        return float(np.sum(Gz * gat.forward(n, rp, col, Y_, F, al, ar)["Z"]))

    fw = gat.forward(n, rp, col, Y, F, a_l, a_r)
    bw = gat.backward_plain(n, rp, col, Y, F, a_l, a_r, fw, Gz)
    h = 1e-6
    num = np.zeros_like(Y)
    for i in range(n):
        for j in range(F):
            Yp, Ym = Y.copy(), Y.copy()
            Yp[i, j] += h
            Ym[i, j] -= h
            num[i, j] = (loss(Yp, a_l, a_r) - loss(Ym, a_l, a_r)) / (2 * h)
    assert np.allclose(bw["dY"], num, rtol=1e-6, atol=1e-7)
    for which, got in (("l", bw["da_l"]), ("r", bw["da_r"])):
        nd = np.zeros(F)
        for j in range(F):
            d = np.zeros(F)
            d[j] = h
            if which == "l":
                nd[j] = (loss(Y, a_l + d, a_r) - loss(Y, a_l - d, a_r)) / (2 * h)
            else:
                nd[j] = (loss(Y, a_l, a_r + d) - loss(Y, a_l, a_r - d)) / (2 * h)
        assert np.allclose(got, nd, rtol=1e-6, atol=1e-7), which


@pytest.mark.parametrize("P", [2, 4])
def test_partitioned_reduces_to_plain_with_raw_messages(P):
    """Raw 32-bit messages dequantise to the fp32 rows exactly, so the
    partitioned forward equals the plain one and the partitioned backward
    differs only by the fp32 rounding of the messages."""
    n, F = 60, 5
    src, dst = planted_partition_edges(n, 240, 4, 0.7, 6)
    rp, col, val = O.csr_build(n, src, dst)
    rng = np.random.default_rng(P)
    Y = rng.standard_normal((n, F)).astype(np.float32).astype(np.float64)
    a_l = rng.standard_normal(F).astype(np.float32)
    a_r = rng.standard_normal(F).astype(np.float32)
    b = O.boundary_index(n, rp, col, val, P)
    S = b["n_slots"]
    sb = np.full(S, 32, np.uint8)
    Ydeq = Y[b["slot_node"]]
    fwp = gat.forward(n, rp, col, Y, F, a_l, a_r, bnd=b, Ydeq=Ydeq)
    fw0 = gat.forward(n, rp, col, Y, F, a_l, a_r)
    assert np.allclose(fwp["Z"], fw0["Z"], rtol=1e-12, atol=1e-13)
    dZ = rng.standard_normal((n, F)).astype(np.float32)
    bw0 = gat.backward_plain(n, rp, col, Y, F, a_l, a_r, fw0, dZ)
    bs = gat.backward_scores(n, rp, fwp, dZ, F)
    bwp = gat.backward_partitioned(n, rp, Y, F, a_l, a_r, b, fwp, dZ, sb, 7,
                                   fwp["alpha"].astype(np.float32), bs["g"].astype(np.float32), Ydeq)
    scale = np.abs(bw0["dY"]).max()
    assert np.allclose(bwp["dY"], bw0["dY"], rtol=0, atol=1e-5 * scale)
    assert np.allclose(bwp["da_l"], bw0["da_l"], rtol=1e-12, atol=1e-12)
    assert np.allclose(bwp["da_r"], bw0["da_r"], rtol=1e-5, atol=1e-5 * scale)
    # a wrong message (its score term dropped) is caught
    assert not np.allclose(bwp["P"] - (bwp["r"][:, None] * a_r).astype(np.float32), bwp["P"])


def test_positions():
    n = 30
    src, dst = planted_partition_edges(n, 90, 3, 0.6, 8)
    rp, col, val = O.csr_build(n, src, dst)
    b = O.boundary_index(n, rp, col, val, 3)
    cr = b["col_remap"].astype(np.int64)
    rows = O.csr_rows(rp)
    tp = gat.transpose_positions(n, rp, cr)
    for k in range(cr.size):
        if cr[k] >= 0:
            assert rows[tp[k]] == cr[k] and cr[tp[k]] == rows[k]
        else:
            assert tp[k] == -1
    sp_ = gat.slot_positions(rp, b)
    for s in range(b["n_slots"]):
        for j in range(b["slot_rowptr"][s], b["slot_rowptr"][s + 1]):
            k = sp_[j]
            assert rows[k] == b["slot_col"][j] and ~cr[k] == s
