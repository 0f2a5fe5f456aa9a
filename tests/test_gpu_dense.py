"""Parity of the tcgen05 dense transform and of whole layers with the oracle.

Dense results are compared with fp64 products of the same bf16 inputs:
|d| <= 2e-2 * sum_k |a_ik b_kj| + 1e-6 (the stated bf16-path bound), and
also against the much tighter bound fp32 accumulation of exact bf16 products
obeys, 1e-4 * sum_k |a_ik b_kj| + 1e-6, so a wrong tile layout cannot hide."""
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


def _bf16_bits(x):
    return (O.bf16_round(x).view(np.uint32) >> 16).astype(np.uint16)


def _bits_to_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def _check_gemm(got, ref, scale, what):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= 2e-2 * scale + 1e-6), f"{what}: outside the bf16-path bound"
    worst = float(np.max(err / (scale + 1e-30))) if err.size else 0.0
    assert np.all(err <= 1e-4 * scale + 1e-6), f"{what}: normalised error {worst:.3g} > 1e-4"


def _rand_mb(n, F_in, seed):
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((n, F_in)).astype(np.float32)
    ldb = G.ldb_for(F_in)
    bits = np.zeros((n, ldb), np.uint16)
    bits[:, :F_in] = _bf16_bits(M)
    return bits


def _rand_w(F_in, F_out, seed):
    rng = np.random.default_rng(seed)
    lim = np.sqrt(6.0 / (F_in + F_out))
    return _bf16_bits(rng.uniform(-lim, lim, (F_in, F_out)).astype(np.float32))


DENSE_CASES = [(1, 16, 16), (127, 16, 16), (128, 100, 256), (1000, 300, 256), (4099, 602, 128),
               (300, 256, 256), (257, 37, 64), (2000, 1024, 32)]


@pytest.mark.parametrize("n,F_in,F_out", DENSE_CASES)
@pytest.mark.parametrize("relu", [0, 1])
def test_dense_fwd(built, n, F_in, F_out, relu):
    t = __import__("torch")
    Mb = _rand_mb(n, F_in, n + F_in)
    W = _rand_w(F_in, F_out, F_out)
    ldo = G.ld_for(F_out)
    H = t.full((n, ldo), float("nan"), device="cuda")
    G.gnn_dense_fwd(dev(Mb.view(np.int16)), n, F_in, dev(W.view(np.int16)), F_out, relu, H)
    G.gnn_sync_check()
    A = _bits_to_f32(Mb[:, :F_in])
    B = _bits_to_f32(W)
    Z, Hn = O.dense_fwd(A, B, relu)
    _check_gemm(host(H)[:, :F_out], Hn, O.gemm_abs(A, B), f"dense_fwd n={n} {F_in}x{F_out}")


@pytest.mark.parametrize("n,F_in,F_out", DENSE_CASES + [(70000, 300, 256)])
def test_dense_bwd(built, n, F_in, F_out):
    t = __import__("torch")
    Mb = _rand_mb(n, F_in, 7 + n)
    W = _rand_w(F_in, F_out, 3)
    rng = np.random.default_rng(11)
    dHo = rng.standard_normal((n, F_out)).astype(np.float32)
    Ho = np.maximum(rng.standard_normal((n, F_out)).astype(np.float32), 0)
    ldm = G.ld_for(F_in)
    dM = t.full((n, ldm), float("nan"), device="cuda")
    dW = t.full((F_in, F_out), float("nan"), device="cuda")
    G.gnn_dense_bwd(dev(Mb.view(np.int16)), n, F_in, dev(W.view(np.int16)), F_out, dev(dHo), dev(Ho),
                    True, dM, dW)
    G.gnn_sync_check()
    A = _bits_to_f32(Mb[:, :F_in])
    B = _bits_to_f32(W)
    dM_ref, dW_ref, dZb = O.dense_bwd(A, B, dHo, Ho, relu=True)
    _check_gemm(host(dM)[:, :F_in], dM_ref, O.gemm_abs(dZb, B.T), f"dM n={n}")
    assert np.all(host(dM)[:, F_in:] == 0)
    _check_gemm(host(dW), dW_ref, O.gemm_abs(A.T, dZb), f"dW n={n}")


def test_dense_bwd_is_deterministic(built):
    t = __import__("torch")
    n, F_in, F_out = 50000, 300, 256
    Mb = dev(_rand_mb(n, F_in, 1).view(np.int16))
    W = dev(_rand_w(F_in, F_out, 2).view(np.int16))
    dHo = t.randn(n, F_out, device="cuda")
    outs = []
    for _ in range(2):
        dM = t.empty((n, F_in + 0), device="cuda")
        dW = t.empty((F_in, F_out), device="cuda")
        G.gnn_dense_bwd(Mb, n, F_in, W, F_out, dHo, None, False, dM, dW)
        outs.append((dM.clone(), dW.clone()))
    assert t.equal(outs[0][0], outs[1][0]) and t.equal(outs[0][1], outs[1][1])


# ------------------------------------------------------------------ whole layers
LAYER_CASES = [("planted", 4096, 16, 16, 4, [90], [2, 8], 0),
               ("planted", 4096, 100, 256, 4, [25, 50, 75], [1, 2, 4, 8], 64),
               ("star", 3000, 300, 128, 3, [80], [4, 8], 64)]


def _graph(name):
    if name == "planted":
        return planted_partition_edges(4096, 16384, 4, 0.9, 5)
    return star_edges(3000, 1234)


@pytest.mark.parametrize("name,n,F_in,F_out,P,pct,bits,split", LAYER_CASES)
def test_layer_fwd_bwd(built, name, n, F_in, F_out, P, pct, bits, split):
    t = __import__("torch")
    src, dst = _graph(name)
    csr = gpu_graph(n, src, dst, split=split)
    b = G.gnn_boundary_index(csr, P, G.BitRule(pct, bits), 1, F_in)
    rp, col, val = O.csr_build(n, src, dst)
    ob = oracle_boundary(n, rp, col, val, P, pct, bits, 1, F_in)
    rng = np.random.default_rng(n + F_in)
    H = rng.standard_normal((n, F_in)).astype(np.float32)
    Wb = _rand_w(F_in, F_out, 5)
    ld, ldb, ldo = G.ld_for(F_in), G.ldb_for(F_in), G.ld_for(F_out)
    Q = int(ob["slot_off"][-1])
    packed = t.zeros(max(Q, 16), dtype=t.uint8, device="cuda")
    meta = t.zeros((max(b.n_slots, 1), 2), device="cuda")
    Mb = t.full((n, ldb), float("nan"), dtype=t.bfloat16, device="cuda")
    Ho = t.full((n, ldo), float("nan"), device="cuda")
    Hd = dev(padded(H, F_in, ld))
    Wd = dev(Wb.view(np.int16))
    G.gnn_layer_fwd(csr, b, Hd, F_in, Wd, F_out, True, 4, packed, meta, Mb, Ho)
    G.gnn_sync_check()
    # forward: messages bit-exact, aggregation within tolerance (plus bf16 rounding)
    wbuf, _, _ = O.quant_pack(H, F_in, ob["slot_node"], ob["slot_bits"], ob["slot_off"][:-1], 4, Q)
    assert np.array_equal(host(packed)[:Q], wbuf)
    Mref, T = O.spmm_fwd(n, rp, col, val, H, F_in, ob, ob["slot_bits"], 4)
    mb = _bits_to_f32(host(Mb.view(t.int16)).view(np.uint16))
    err = np.abs(mb[:, :F_in] - Mref)
    assert np.all(err <= 1e-5 * T + 1e-7 + 2.0 ** -8 * np.abs(Mref)), "Mb outside tolerance"
    assert np.all(mb[:, F_in:] == 0)
    # transform, teacher-forced on the GPU's Mb
    A = mb[:, :F_in]
    B = _bits_to_f32(Wb)
    _, Href = O.dense_fwd(A, B, True)
    _check_gemm(host(Ho)[:, :F_out], Href, O.gemm_abs(A, B), "layer H_out")
    # backward
    dHo = dev(rng.standard_normal((n, ldo)).astype(np.float32))
    dW = t.full((F_in, F_out), float("nan"), device="cuda")
    dHi = t.full((n, ld), float("nan"), device="cuda")
    pw = t.zeros_like(packed)
    mw = t.zeros_like(meta)
    G.gnn_layer_bwd(csr, b, dHo, Ho, True, Mb, Wd, F_in, F_out, 5, pw, mw, dW, dHi)
    # the same dense backward standalone gives the dM the layer used (deterministic)
    dM = t.empty((n, ld), device="cuda")
    dW2 = t.empty((F_in, F_out), device="cuda")
    G.gnn_dense_bwd(Mb, n, F_in, Wd, F_out, dHo, Ho, True, dM, dW2)
    G.gnn_sync_check()
    assert t.equal(dW, dW2)
    dM_ref, dW_ref, dZb = O.dense_bwd(A, B, host(dHo)[:, :F_out], host(Ho)[:, :F_out], True)
    _check_gemm(host(dW), dW_ref, O.gemm_abs(A.T, dZb), "layer dW")
    _check_gemm(host(dM)[:, :F_in], dM_ref, O.gemm_abs(dZb, B.T), "layer dM")
    dMh = host(dM)[:, :F_in]
    bbuf, _, _ = O.halo_quant_pack(ob, dMh, F_in, ob["slot_bits"], ob["slot_off"], 5)
    assert np.array_equal(host(pw)[:Q], bbuf), "backward messages differ"
    dref, T2 = O.spmm_bwd(n, rp, col, val, dMh, F_in, ob, ob["slot_bits"], 5)
    assert_close_agg(host(dHi)[:, :F_in], dref, T2, "layer dH_in")


def test_layer_bwd_first_layer_skips_aggregation(built):
    t = __import__("torch")
    src, dst = _graph("planted")
    n, F_in, F_out = 4096, 16, 16
    csr = gpu_graph(n, src, dst)
    Mb = dev(_rand_mb(n, F_in, 3).view(np.int16))
    W = dev(_rand_w(F_in, F_out, 4).view(np.int16))
    dHo = t.randn(n, F_out, device="cuda")
    dW = t.empty((F_in, F_out), device="cuda")
    G.gnn_layer_bwd(csr, None, dHo, None, False, Mb, W, F_in, F_out, 1, None, None, dW, None)
    G.gnn_sync_check()
    assert t.isfinite(dW).all()
