"""The backward aggregation with the lower layer's ReLU gate fused into its
store (gnn_spmm_bwd_masked) and the dense backward that reads its bf16 output
(gnn_dense_bwd_z): the gated bf16 rows equal bf16(dH * 1[H > 0]) of the
plain backward's dH bit for bit, zero-padded to the 64-column stride; the
messages are the plain backward's; and the dense backward from that dZ equals
gnn_dense_bwd from (dH, H) bit for bit."""
import numpy as np
import pytest

import oracle as O
from tests.helpers import dev, gpu_graph, host, oracle_boundary, padded
from tests.test_gpu_parity import GRAPHS

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return G


def _f32(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def _bf16_bits(x):
    return (O.bf16_round(x).view(np.uint32) >> 16).astype(np.uint16)


CASES = [("er64", 0, 16, 0), ("planted", 4, 16, 32), ("star", 3, 300, 64), ("er300", 7, 100, 32),
         ("planted", 4, 256, 0), ("star", 0, 128, 64), ("er300", 3, 129, 0)]


@pytest.mark.parametrize("name,P,F,split", CASES)
@pytest.mark.parametrize("gate", [True, False])
def test_masked_backward(built, name, P, F, split, gate):
    t = __import__("torch")
    n, src, dst = GRAPHS[name]
    csr = gpu_graph(n, src, dst, split=split)
    b = None
    Q, S = 16, 1
    if P:
        b = G.gnn_boundary_index(csr, P, G.BitRule([50], [2, 8]), 1, F)
        if split:
            G.gnn_boundary_long_slots(csr, b, 32)
        S = max(b.n_slots, 1)
        Q = max(int(host(b.slot_off)[-1]), 16)
    rng = np.random.default_rng(n + F)
    ld, ldz = G.ld_for(F), G.ldz_for(F)
    Gm = dev(padded(rng.standard_normal((n, F)).astype(np.float32), F, ld))
    Hm = np.maximum(rng.standard_normal((n, F)), 0).astype(np.float32)
    Hm_d = dev(padded(Hm, F, ld))
    pw1, mw1 = t.zeros(Q, dtype=t.uint8, device="cuda"), t.zeros((S, 2), device="cuda")
    pw2, mw2 = t.zeros_like(pw1), t.zeros_like(mw1)
    dH = t.empty((n, ld), device="cuda")
    G.gnn_spmm_bwd(csr, b, Gm, F, 5, pw1, mw1, dH)
    dZ = t.full((n, ldz), float("nan"), dtype=t.bfloat16, device="cuda")
    G.gnn_spmm_bwd_masked(csr, b, Gm, F, 5, pw2, mw2, Hm_d if gate else None, dZ)
    G.gnn_sync_check()
    assert t.equal(pw1, pw2) and t.equal(mw1, mw2)
    dh = host(dH)[:, :F]
    want = np.zeros((n, ldz), np.uint16)
    want[:, :F] = _bf16_bits(np.where(Hm > 0, dh, np.float32(0)) if gate else dh)
    assert np.array_equal(host(dZ.view(t.int16)).view(np.uint16), want)
    # the two halves called apart give the same bytes
    if b is not None:
        pw3, mw3 = t.zeros_like(pw1), t.zeros_like(mw1)
        dZ3 = t.full((n, ldz), float("nan"), dtype=t.bfloat16, device="cuda")
        G.gnn_halo_quant_pack(b, Gm, F, 5, pw3, mw3)
        G.gnn_spmm_bwd_local_masked(csr, b, Gm, F, pw3, mw3, Hm_d if gate else None, dZ3)
        G.gnn_sync_check()
        assert t.equal(pw1, pw3) and t.equal(mw1, mw3) and t.equal(dZ, dZ3)
    # against the oracle directly: dZ = bf16(fp32 sum * gate); the fp32 sum is
    # within 1e-5*T + 1e-7 of the fp64 one, bf16 rounding adds half an ulp
    # (at most 2^-8 relative: bf16 keeps 8 significant bits)
    rp, col, val = O.csr_build(n, src, dst)
    Gh = host(Gm)[:, :F]
    if b is not None:
        ob = oracle_boundary(n, rp, col, val, P, [50], [2, 8], 1, F)
        ref, T = O.spmm_bwd(n, rp, col, val, Gh, F, ob, ob["slot_bits"], 5)
    else:
        ref, T = O.spmm_bwd(n, rp, col, val, Gh, F)
    gmask = (Hm > 0) if gate else np.ones_like(Hm, bool)
    got = _f32(host(dZ.view(t.int16)).view(np.uint16))
    assert np.all(got[:, F:] == 0)
    g = got[:, :F].astype(np.float64)
    assert np.all(g[~gmask] == 0)
    bound = 2.0 ** -8 * np.abs(ref) + 1.1e-5 * T + 2e-7
    assert np.all(np.abs(g - ref)[gmask] <= bound[gmask])
    # the dense backward of the layer below, from dZ or from (dH, H)
    F_in = 48
    Mb = np.zeros((n, G.ldb_for(F_in)), np.uint16)
    Mb[:, :F_in] = _bf16_bits(rng.standard_normal((n, F_in)).astype(np.float32))
    W = _bf16_bits((0.1 * rng.standard_normal((F_in, F))).astype(np.float32)) if F % 16 == 0 else None
    if W is None:
        return
    Mbd, Wd = dev(Mb.view(np.int16)), dev(W.view(np.int16))
    dM1, dW1 = t.empty((n, G.ld_for(F_in)), device="cuda"), t.empty((F_in, F), device="cuda")
    dM2, dW2 = t.empty_like(dM1), t.empty_like(dW1)
    G.gnn_dense_bwd(Mbd, n, F_in, Wd, F, dH, Hm_d if gate else None, gate, dM1, dW1)
    G.gnn_dense_bwd_z(Mbd, n, F_in, Wd, F, dZ, dM2, dW2)
    G.gnn_sync_check()
    assert t.equal(dM1[:, :F_in], dM2[:, :F_in]) and t.equal(dW1, dW2)
    # against the oracle's dense backward on the oracle's own dZ (its fp64
    # aggregation, gated and rounded to bf16): an input may sit one bf16 step
    # away from the GPU's, well inside the transform's tolerance
    dZo = O.bf16_round(np.where(gmask, ref, 0.0).astype(np.float32)).astype(np.float64)
    Mbf = _f32(Mb[:, :F_in])
    Wf = _f32(W)
    dM_ref, dW_ref, _ = O.dense_bwd(Mbf, Wf, dZo, None, False)
    sM = O.gemm_abs(dZo, Wf.T)
    sW = O.gemm_abs(Mbf.T, dZo)
    assert np.all(np.abs(host(dM2)[:, :F_in] - dM_ref) <= 2e-2 * sM + 1e-6)
    assert np.all(np.abs(host(dW2) - dW_ref) <= 2e-2 * sW + 1e-6)
