"""One small pass of the hot path on cuda:0 checked against the oracle: the
4096-node planted-partition workload (4 partitions, widths 8/2 by importance),
boundary index, forward quantise-pack + aggregation, backward halo
quantise-pack + aggregation."""
from __future__ import annotations

import numpy as np


def run() -> None:
    import torch

    import oracle as O
    import sparse_aggregation_message_gb300 as G
    from synth import make_workload
    from tests.helpers import assert_close_agg, dev, host, oracle_boundary, padded

    assert torch.cuda.is_available(), "smoke needs cuda:0"
    torch.cuda.set_device(0)
    wl = make_workload("tiny")
    n, F = wl.n, wl.dims[0]
    csr = G.gnn_csr_build(n, dev(wl.src), dev(wl.dst))
    rp, col, val = O.csr_build(n, wl.src, wl.dst)
    assert np.array_equal(host(csr.col), col) and np.array_equal(host(csr.rowptr), rp)
    rule = G.BitRule(wl.rule_pct, wl.rule_bits)
    b = G.gnn_boundary_index(csr, wl.P, rule, 1, F)
    ob = oracle_boundary(n, rp, col, val, wl.P, wl.rule_pct, wl.rule_bits, 1, F)
    assert np.array_equal(host(b.col_remap), ob["col_remap"])
    assert np.array_equal(host(b.slot_off), ob["slot_off"])
    rng = np.random.default_rng(wl.seed + 1)
    H = rng.standard_normal((n, F)).astype(np.float32)
    Gm = rng.standard_normal((n, F)).astype(np.float32)
    ld = G.ld_for(F)
    Q = int(ob["slot_off"][-1])
    packed = torch.zeros(Q, dtype=torch.uint8, device="cuda")
    meta = torch.zeros((b.n_slots, 2), device="cuda")
    Hd = dev(padded(H, F, ld))
    G.gnn_quant_pack(Hd, F, b.slot_node, b.n_slots, b.slot_bits, b.slot_off, 2, packed, meta)
    M = torch.empty((n, ld), device="cuda")
    G.gnn_spmm_fwd(csr, b, Hd, F, packed, meta, M=M)
    pw = torch.zeros(Q, dtype=torch.uint8, device="cuda")
    mw = torch.zeros((b.n_slots, 2), device="cuda")
    dH = torch.empty((n, ld), device="cuda")
    G.gnn_spmm_bwd(csr, b, dev(padded(Gm, F, ld)), F, 3, pw, mw, dH)
    G.gnn_sync_check()
    wbuf, _, _ = O.quant_pack(H, F, ob["slot_node"], ob["slot_bits"], ob["slot_off"][:-1], 2, Q)
    assert np.array_equal(host(packed), wbuf), "forward packed bytes differ"
    ref, T = O.spmm_fwd(n, rp, col, val, H, F, ob, ob["slot_bits"], 2)
    assert_close_agg(host(M)[:, :F], ref, T, "smoke forward")
    bbuf, _, _ = O.halo_quant_pack(ob, Gm, F, ob["slot_bits"], ob["slot_off"], 3)
    assert np.array_equal(host(pw), bbuf), "backward packed bytes differ"
    ref, T = O.spmm_bwd(n, rp, col, val, Gm, F, ob, ob["slot_bits"], 3)
    assert_close_agg(host(dH)[:, :F], ref, T, "smoke backward")
    print("smoke ok: tiny workload, forward and backward match the oracle")


if __name__ == "__main__":
    run()
