"""Shared test helpers: move seeded inputs to the GPU, run the library through
its binding, and fetch oracle results for the same inputs."""
from __future__ import annotations

import numpy as np

import oracle as O

TOL_REL = 1e-5   # aggregation: |d| <= 1e-5 * sum|terms| + 1e-7
TOL_ABS = 1e-7


def torch():
    import torch as t
    return t


def dev(x, dtype=None):
    t = torch()
    a = t.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        a = a.to(dtype)
    return a.cuda()


def host(t):
    return t.detach().cpu().numpy()


def padded(X, F, ld):
    out = np.zeros((X.shape[0], ld), np.float32)
    out[:, :F] = X[:, :F]
    return out


def gpu_graph(n, src, dst, flags=O.FLAGS_GCN, split=0):
    """CSR on the GPU; split > 0 attaches a row-split plan (rows longer than
    `split` entries cut into pieces)."""
    import sparse_aggregation_message_gb300 as G
    t = torch()
    s = dev(np.asarray(src, np.int32))
    d = dev(np.asarray(dst, np.int32))
    csr = G.gnn_csr_build(n, s, d, flags)
    if split:
        csr = G.gnn_csr_split(csr, split)
    t.cuda.synchronize()
    return csr


def oracle_boundary(n, rowptr, col, val, P, pct, bits, base, F, val_t=None):
    b = O.boundary_index(n, rowptr, col, val, P, val_t)
    nb = O.node_bits(n, rowptr, b, pct, bits, base)
    sb = nb[b["slot_node"]] if b["n_slots"] else np.zeros(0, np.uint8)
    b["node_bits"] = nb
    b["slot_bits"] = sb.astype(np.uint8)
    b["slot_off"] = O.slot_offsets(sb, F)
    return b


def assert_close_agg(got, ref, T, where=""):
    """|got - ref| <= 1e-5 * T + 1e-7 element-wise (T = sum of |terms|)."""
    err = np.abs(got.astype(np.float64) - ref)
    bound = TOL_REL * T + TOL_ABS
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{where}: {bad.sum()} elements out of bound; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} T {T[tuple(i)]!r}")
