"""Kernels the library selects only for graphs with 16M slots or more: the
ring kernel of the backward messages (also used for rows of four or more
16-byte chunks per lane) and the node-grouped quantiser of the forward
messages.  The small graphs of the other tests do not reach them, so this
file builds the library once more with both slot thresholds at zero (a
build variant under the package's _build/ directory), routes the binding
through it, and repeats the partitioned backward against the oracle at 2, 3,
5 and 8 chunks per lane, with split rows and long slots, one attention layer
(whose backward messages carry the score term), and the forward messages of
gnn_quant_pack_owned against the oracle and gnn_quant_pack -- messages
bit-exact, aggregations within the aggregation bound."""
import numpy as np
import pytest

import oracle as O
from tests import test_gpu_gat as GAT
from tests.helpers import dev, host, padded
from tests import test_gpu_parity as PAR

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")


@pytest.fixture(scope="module")
def ring_everywhere():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_aggregation_message_gb300 import _abi, builder

    G.load()
    path = builder.build(extra=["-DGNN_RING_MIN_SLOTS=0", "-DGNN_OWNED_MIN_SLOTS=0"],
                         variant="large_graph_kernels")
    old = _abi.use_lib(_abi.open_lib(path))
    yield G
    _abi.use_lib(old)


# (name, P, pct, bits, base, F, split): F = 129, 200, 300, 602, 1024 give 2,
# 2, 3, 5 and 8 chunks per lane in the backward-message kernel
RING_CASES = [("planted", 4, [90], [2, 8], 1, 129, 0), ("star", 3, [80], [4, 8], 1, 200, 64),
              ("er300", 7, [25, 50, 75], [1, 2, 4, 8], 1, 300, 32),
              ("star", 5, [50], [1, 8], 1, 602, 32), ("er300", 3, [90], [2, 8], 1, 1024, 0)]


@pytest.mark.parametrize("name,P,pct,bits,base,F,split", RING_CASES)
def test_backward_messages_through_ring(ring_everywhere, name, P, pct, bits, base, F, split):
    PAR.test_spmm_bwd_partitioned(ring_everywhere, name, P, pct, bits, base, F, split)


def test_attention_backward_messages_through_ring(ring_everywhere):
    GAT.test_gat_layer(ring_everywhere, "star", 3000, 300, 256, 3, [80], [4, 8], 64)


@pytest.mark.parametrize("name,P,pct,bits,base,F,split",
                         PAR.PART_CASES + RING_CASES[-1:] + [("planted", 4, [90], [32, 32], 1, 24, 0)])
def test_node_grouped_forward_messages(ring_everywhere, name, P, pct, bits, base, F, split):
    t = __import__("torch")
    n, csr, b, rp, col, val, ob = PAR._partitioned_setup(name, P, pct, bits, base, F, 0, split)
    H = PAR._features(n, F, 13)
    Hd = dev(padded(H, F, G.ld_for(F)))
    Q = int(ob["slot_off"][-1])
    S = max(b.n_slots, 1)
    p1 = t.full((max(Q, 16),), 0xAB, dtype=t.uint8, device="cuda")
    m1 = t.full((S, 2), float("nan"), device="cuda")
    p2, m2 = p1.clone(), m1.clone()
    G.gnn_quant_pack_owned(b, Hd, F, 77, p1, m1)
    G.gnn_quant_pack(Hd, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, 77, p2, m2)
    G.gnn_sync_check()
    want, wmeta, _ = O.quant_pack(H, F, ob["slot_node"], ob["slot_bits"], ob["slot_off"][:-1], 77, Q)
    assert np.array_equal(host(p1)[:Q], want)
    assert np.array_equal(host(m1)[: b.n_slots].view(np.uint32), wmeta.view(np.uint32))
    assert np.array_equal(host(p1), host(p2))
    assert np.array_equal(host(m1).view(np.uint32), host(m2).view(np.uint32))
