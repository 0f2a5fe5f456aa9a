"""The ring kernel of the backward messages at every row layout it serves.

The library sends a backward-message launch through the ring kernel when the
launch has 16M slots or more (or rows of four or more 16-byte chunks per
lane); the small graphs of the other tests reach it only at the widest
layouts.  This file builds the library once more with that slot threshold at
zero (a build variant under the package's _build/ directory), routes the
binding through it, and repeats the partitioned backward against the oracle
at 2, 3, 5 and 8 chunks per lane, with split rows and long slots, and one
attention layer, whose backward messages carry the score term -- messages
bit-exact, aggregations within the aggregation bound."""
import pytest

from tests import test_gpu_gat as GAT
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
    path = builder.build(extra=["-DGNN_RING_MIN_SLOTS=0"], variant="ring_min0")
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
