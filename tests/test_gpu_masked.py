"""The backward aggregation with the lower layer's ReLU gate fused into its
store (gnn_spmm_bwd_masked) and the dense backward that reads its bf16 output
(gnn_dense_bwd_z): the gated bf16 rows equal bf16(dH * 1[H > 0]) of the
plain backward's dH bit for bit, zero-padded to the 64-column stride; the
messages are the plain backward's; and the dense backward from that dZ equals
gnn_dense_bwd from (dH, H) bit for bit."""
import numpy as np
import pytest

import oracle as O
from tests.helpers import dev, gpu_graph, host, padded
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
