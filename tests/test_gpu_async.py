"""Asynchronous epochs (SYLVIE guide section 10): a layer aggregates with the
previous epoch's boundary messages while the current epoch's are quantised
and packed on a second stream.

Checked against the oracle with the stale matrix passed as the message
source: the messages each call packs are bit-exact, the aggregation is within
|d| <= 1e-5 * sum|terms| + 1e-7 (plus bf16 rounding where the output is
bf16), and the split backward calls reproduce the fused one bit for bit."""
import numpy as np
import pytest

import oracle as O
from synth import planted_partition_edges, star_edges
from tests.helpers import assert_close_agg, dev, gpu_graph, host, oracle_boundary, padded

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")

CASES = [("planted", 4096, 16, 16, 4, [90], [2, 8], 0),
         ("planted", 4096, 100, 64, 4, [25, 50, 75], [1, 2, 4, 8], 64),
         ("star", 3000, 300, 128, 3, [80], [4, 8], 64)]


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


def _graph(name, n):
    if name == "planted":
        return planted_partition_edges(n, 4 * n, 4, 0.9, 5)
    return star_edges(n, 1234)


def _bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rand_w(F_in, F_out, seed):
    rng = np.random.default_rng(seed)
    lim = np.sqrt(6.0 / (F_in + F_out))
    w = O.bf16_round(rng.uniform(-lim, lim, (F_in, F_out)).astype(np.float32))
    return (w.view(np.uint32) >> 16).astype(np.uint16)


def _setup(name, n, F_in, P, pct, bits, split):
    src, dst = _graph(name, n)
    csr = gpu_graph(n, src, dst, split=split)
    b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), 1, F_in)
    if split:
        G.gnn_boundary_long_slots(csr, b, split)
    rp, col, val = O.csr_build(n, src, dst)
    ob = oracle_boundary(n, rp, col, val, P, pct, bits, 1, F_in)
    return csr, b, rp, col, val, ob


@pytest.mark.parametrize("name,n,F,F_out,P,pct,bits,split", CASES)
def test_bwd_split_calls_equal_fused(built, name, n, F, F_out, P, pct, bits, split):
    t = __import__("torch")
    csr, b, rp, col, val, ob = _setup(name, n, F, P, pct, bits, split)
    Q = int(ob["slot_off"][-1])
    ld = G.ld_for(F)
    Gm = dev(padded(np.random.default_rng(3).standard_normal((n, F)).astype(np.float32), F, ld))
    outs = []
    for fused in (True, False):
        pk = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
        mt = t.zeros((max(b.n_slots, 1), 2), device="cuda")
        dH = t.full((n, ld), float("nan"), device="cuda")
        if fused:
            G.gnn_spmm_bwd(csr, b, Gm, F, 9, pk, mt, dH)
        else:
            G.gnn_halo_quant_pack(b, Gm, F, 9, pk, mt)
            G.gnn_spmm_bwd_local(csr, b, Gm, F, pk, mt, dH)
        G.gnn_sync_check()
        outs.append((host(pk), host(mt), host(dH)))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))
    assert np.array_equal(outs[0][2].view(np.uint32), outs[1][2].view(np.uint32))


@pytest.mark.parametrize("name,n,F,F_out,P,pct,bits,split", CASES)
def test_layer_async_two_epochs(built, name, n, F, F_out, P, pct, bits, split):
    """Epoch 0 synchronous, epoch 1 asynchronous: the forward aggregation of
    epoch 1 reads H1 for local sources and the messages of H0 for remote
    ones; epoch 1's messages of H1 are packed meanwhile.  Same for the
    backward pass with dM0 / dM1."""
    t = __import__("torch")
    csr, b, rp, col, val, ob = _setup(name, n, F, P, pct, bits, split)
    S, Q = b.n_slots, int(ob["slot_off"][-1])
    sb = ob["slot_bits"]
    ld, ldb, ldo = G.ld_for(F), G.ldb_for(F), G.ld_for(F_out)
    rng = np.random.default_rng(n + F)
    H0 = rng.standard_normal((n, F)).astype(np.float32)
    H1 = (H0 + 0.5 * rng.standard_normal((n, F))).astype(np.float32)
    Wb = _rand_w(F, F_out, 5)
    Wd = dev(Wb.view(np.int16))
    aux = t.cuda.Stream()

    def bufs():
        return (t.zeros(max(Q, 16), dtype=t.uint8, device="cuda"),
                t.zeros((max(S, 1), 2), device="cuda"))

    # ---- epoch 0 (synchronous): messages of H0 with seed 10
    p0, m0 = bufs()
    Mb0 = t.empty((n, ldb), dtype=t.bfloat16, device="cuda")
    Ho0 = t.empty((n, ldo), device="cuda")
    G.gnn_layer_fwd(csr, b, dev(padded(H0, F, ld)), F, Wd, F_out, True, 10, p0, m0, Mb0, Ho0)
    # ---- epoch 1 (asynchronous): aggregate with p0/m0, pack H1 with seed 12
    p1, m1 = bufs()
    Mb1 = t.full((n, ldb), float("nan"), dtype=t.bfloat16, device="cuda")
    Ho1 = t.full((n, ldo), float("nan"), device="cuda")
    H1d = dev(padded(H1, F, ld))
    G.gnn_layer_fwd_async(csr, b, H1d, F, Wd, F_out, True, 12, p0, m0, p1, m1, Mb1, Ho1, aux)
    # a consumer on the main stream sees the new messages complete
    Mchk = t.empty((n, ld), device="cuda")
    G.gnn_spmm_fwd(csr, b, H1d, F, p1, m1, M=Mchk)
    G.gnn_sync_check()

    wbuf, wmeta, _ = O.quant_pack(H1, F, ob["slot_node"], sb, ob["slot_off"][:-1], 12, Q)
    assert np.array_equal(host(p1)[:Q], wbuf), "epoch-1 forward messages"
    assert np.array_equal(host(m1)[:S].view(np.uint32), wmeta.view(np.uint32))
    ref, T = O.spmm_fwd(n, rp, col, val, H1, F, ob, sb, 10, H_msg=H0)
    mb = _bits_to_f32(host(Mb1.view(t.int16)).view(np.uint16))[:, :F]
    assert np.all(np.abs(mb - ref) <= 1e-5 * T + 1e-7 + 2.0 ** -8 * np.abs(ref)), "stale forward"
    # the same aggregation through the synchronous entry point, bit for bit
    Mb_sync = t.empty((n, ldb), dtype=t.bfloat16, device="cuda")
    G.gnn_spmm_fwd(csr, b, H1d, F, p0, m0, Mb=Mb_sync)
    G.gnn_sync_check()
    assert t.equal(Mb1.view(t.int16), Mb_sync.view(t.int16))
    ref_new, T_new = O.spmm_fwd(n, rp, col, val, H1, F, ob, sb, 12)
    assert_close_agg(host(Mchk)[:, :F], ref_new, T_new, "consumer of the new messages")
    if S:
        # the stale and fresh aggregations differ where remote sources are read
        assert not np.allclose(ref, ref_new)
    # transform of epoch 1 on the GPU's Mb
    _, Href = O.dense_fwd(mb, _bits_to_f32(Wb), True)
    err = np.abs(host(Ho1)[:, :F_out] - Href)
    assert np.all(err <= 1e-4 * O.gemm_abs(mb, _bits_to_f32(Wb)) + 1e-6)

    # ---- backward: epoch 0 synchronous with seed 11, epoch 1 async with seed 13
    dHo0 = dev(rng.standard_normal((n, ldo)).astype(np.float32))
    dHo1 = dev(rng.standard_normal((n, ldo)).astype(np.float32))
    q0, n0 = bufs()
    dW0 = t.empty((F, F_out), device="cuda")
    dHi0 = t.empty((n, ld), device="cuda")
    G.gnn_layer_bwd(csr, b, dHo0, Ho0, True, Mb0, Wd, F, F_out, 11, q0, n0, dW0, dHi0)
    q1, n1 = bufs()
    dW1 = t.full((F, F_out), float("nan"), device="cuda")
    dHi1 = t.full((n, ld), float("nan"), device="cuda")
    G.gnn_layer_bwd_async(csr, b, dHo1, Ho1, True, Mb1, Wd, F, F_out, 13, q0, n0, q1, n1, dW1,
                          dHi1, aux)
    # dM of each epoch from the standalone dense backward (deterministic)
    dMs = []
    for dHo, Ho, Mb in ((dHo0, Ho0, Mb0), (dHo1, Ho1, Mb1)):
        dM = t.empty((n, ld), device="cuda")
        dWx = t.empty((F, F_out), device="cuda")
        G.gnn_dense_bwd(Mb, n, F, Wd, F_out, dHo, Ho, True, dM, dWx)
        dMs.append((host(dM)[:, :F], dWx))
    G.gnn_sync_check()
    assert t.equal(dW1, dMs[1][1])
    dM0, dM1 = dMs[0][0], dMs[1][0]
    bbuf, bmeta, _ = O.halo_quant_pack(ob, dM1, F, sb, ob["slot_off"], 13)
    assert np.array_equal(host(q1)[:Q], bbuf), "epoch-1 backward messages"
    assert np.array_equal(host(n1)[:S].view(np.uint32), bmeta.view(np.uint32))
    dref, T2 = O.spmm_bwd(n, rp, col, val, dM1, F, ob, sb, 11, G_msg=dM0)
    assert_close_agg(host(dHi1)[:, :F], dref, T2, "stale backward")


def test_async_requires_message_buffers(built):
    t = __import__("torch")
    csr, b, rp, col, val, ob = _setup("planted", 4096, 16, 4, [90], [2, 8], 0)
    n, F = 4096, 16
    Mb = t.empty((n, G.ldb_for(F)), dtype=t.bfloat16, device="cuda")
    Ho = t.empty((n, G.ld_for(16)), device="cuda")
    H = t.zeros((n, G.ld_for(F)), device="cuda")
    W = dev(_rand_w(F, 16, 1).view(np.int16))
    with pytest.raises(G.GnnError):
        G.gnn_layer_fwd_async(csr, b, H, F, W, 16, True, 1, None, None, None, None, Mb, Ho,
                              t.cuda.Stream())
