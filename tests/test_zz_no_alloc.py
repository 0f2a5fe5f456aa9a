"""The forward aggregation entry point that allocates nothing.

Some callers cannot allocate device memory while they run -- a serving loop
that reserved all of its memory at start-up, or a plugin that a host
framework hands only input and output pointers.  gnn_spmm_fwd_noalloc takes
its scratch (the partial rows of long, split rows) from a fixed array inside
the library.  These tests call it through the C ABI and compare it with
gnn_spmm_fwd (which takes a caller workspace) on two calls in a row, and check
that a request larger than the array is refused before anything runs.  This
file is collected last so a failure here stops a -x run only after every
other test has run."""
import ctypes

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


def test_noalloc_forward_matches_workspace_forward_twice(built):
    t = __import__("torch")
    n, F, P = 3000, 100, 3
    src, dst = star_edges(n, 1234)
    # add some community structure so ordinary rows mix with the split hub row
    s2, d2 = planted_partition_edges(n, 6000, 3, 0.9, 2)
    src, dst = np.concatenate([src, s2]), np.concatenate([dst, d2])
    csr = gpu_graph(n, src, dst, split=64)
    assert csr.n_pieces > 0  # the scratch is really used
    b = G.gnn_boundary_index(csr, P, G.BitRule([50], [2, 8]), 1, F)
    rp, col, val = O.csr_build(n, src, dst)
    ob = oracle_boundary(n, rp, col, val, P, [50], [2, 8], 1, F)
    ld = G.ld_for(F)
    Q = int(ob["slot_off"][-1])
    for call_no, seed in enumerate([3, 4]):  # two calls in a row, different inputs
        H = np.random.default_rng(seed).standard_normal((n, F)).astype(np.float32)
        Hd = dev(padded(H, F, ld))
        packed = t.zeros(Q, dtype=t.uint8, device="cuda")
        meta = t.zeros((b.n_slots, 2), device="cuda")
        G.gnn_quant_pack(Hd, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, seed, packed, meta)
        M_ws = t.full((n, ld), float("nan"), device="cuda")
        M_na = t.full((n, ld), float("nan"), device="cuda")
        G.gnn_spmm_fwd(csr, b, Hd, F, packed, meta, M=M_ws)
        G.gnn_spmm_fwd_noalloc(csr, b, Hd, F, packed, meta, M=M_na)
        G.gnn_sync_check()
        ref, T = O.spmm_fwd(n, rp, col, val, H, F, ob, ob["slot_bits"], seed)
        got_ws, got_na = host(M_ws), host(M_na)
        # against the existing entry point, within the aggregation tolerance
        err = np.abs(got_na[:, :F].astype(np.float64) - got_ws[:, :F])
        assert np.all(err <= 1e-5 * T + 1e-7), f"call {call_no}: no-alloc differs from gnn_spmm_fwd"
        assert_close_agg(got_na[:, :F], ref, T, f"no-alloc call {call_no}")


def test_noalloc_refuses_a_plan_larger_than_its_array(built):
    from sparse_aggregation_message_gb300 import _abi
    lib = _abi.load()
    # a split plan whose partial rows need 64 MiB at F=1024 (n_pieces=16384)
    c = _abi.GnnCsr(4, 1, 4, 16, 16, 16, 64, 1, 16384, 16, 16, 16, 16)
    st = lib.gnn_spmm_fwd_noalloc(ctypes.byref(c), None, ctypes.c_void_p(16), 1024, 1024, None,
                                  None, ctypes.c_void_p(16), 1024, None, 0, None)
    assert st == 2
    assert b"static buffer" in lib.gnn_last_error()
