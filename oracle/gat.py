"""Oracle of the attention aggregator: a GAT layer on the boundary-quantised
path, forward and backward.

TEST INFRASTRUCTURE ONLY -- imported by tests, never by the library.

Source: the SYLVIE guide, section 2 (GAT weights the neighbour aggregation by
attention coefficients alpha_vu) and section 12 (its GAT runs use one head).
The pages give no formula; the reading taken is the single-head graph
attention layer of Velickovic et al. (ICLR 2018) on the transformed rows:
  Y = H W,  s_l = Y a_l,  s_r = Y a_r,
  e_vu = LeakyReLU(s_l[v] + s_r[u]) (slope 0.2) over u in N(v) + {v},
  alpha_v. = softmax(e_v.),  Z_v = sum_u alpha_vu Y_u,  H' = act(Z).
Partitions (section 3): a remote source u is known to v's partition only by
its dequantised message Y~_u (the quantised row of Y), so its score is
s~_r = a_r . Y~_u, computed by the receiver.  The backward (section 3: the
gradients travel back along the same dependencies) sends each boundary copy
its gradient d(loss)/dY~_u = sum_{v in q} alpha_vu dZ_v + a_r sum_{v in q} g_vu
(g the gradient at the pre-activation score), quantised like the forward
messages, and the owner adds it to dY_u (straight through the quantiser).

Everything accumulates in fp64 except where a fixed fp32 order is stated:
the backward message, whose codes are compared bit for bit, is the halo
partial of section 3 (start +0, entries by ascending v, each product and sum
rounded to fp32) followed by the score term, each element rounded
fl(P + fl(r_s * a_r)).
"""
from __future__ import annotations

import numpy as np

from . import oracle as O

SLOPE = 0.2
F32 = np.float32


def lrelu(x):
    return np.where(x > 0, x, SLOPE * x)


def lrelu_grad(x):
    return np.where(x > 0, 1.0, SLOPE)


def _entries(n, rowptr):
    return O.csr_rows(rowptr)


def forward(n, rowptr, col, Y, F, a_l, a_r, bnd=None, Ydeq=None):
    """Scores, attention and Z.  Without bnd the entries are the CSR's (col);
    with bnd they follow col_remap (local ids, then ~slot), and Ydeq[s] is the
    dequantised message of slot s.  Returns dict(pre, alpha, Z, s_l, s_r,
    s_slot, X_rows) with X_rows[k] the row entry k aggregates (fp64)."""
    Yd = np.asarray(Y, np.float64)[:, :F]
    a_l = np.asarray(a_l, np.float64)
    a_r = np.asarray(a_r, np.float64)
    s_l = Yd @ a_l
    s_r = Yd @ a_r
    rows = _entries(n, rowptr)
    if bnd is None:
        src = np.asarray(col, np.int64)
        src_score = s_r[src]
        X_rows = Yd[src]
        s_slot = None
    else:
        cr = np.asarray(bnd["col_remap"], np.int64)
        remote = cr < 0
        slot = np.where(remote, ~cr, 0)
        Yq = np.asarray(Ydeq, np.float64)[:, :F] if Ydeq is not None and len(Ydeq) else \
            np.zeros((0, F))
        s_slot = Yq @ a_r if Yq.size else np.zeros(0)
        src_score = np.where(remote, s_slot[slot] if s_slot.size else 0.0, s_r[np.where(remote, 0, cr)])
        X_rows = np.where(remote[:, None], Yq[slot] if Yq.size else 0.0, Yd[np.where(remote, 0, cr)])
    pre = s_l[rows] + src_score
    e = lrelu(pre)
    alpha = np.zeros_like(e)
    for v in range(n):
        b, t = rowptr[v], rowptr[v + 1]
        if t > b:
            m = e[b:t].max()
            w = np.exp(e[b:t] - m)
            alpha[b:t] = w / w.sum()
    Z = np.zeros((n, F))
    np.add.at(Z, rows, alpha[:, None] * X_rows)
    return dict(pre=pre, alpha=alpha, Z=Z, s_l=s_l, s_r=s_r, s_slot=s_slot, X_rows=X_rows,
                rows=rows)


def backward_scores(n, rowptr, fw, dZ, F):
    """Per entry k of row v: dalpha_k = dZ_v . x_k, the softmax backward
    de_k = alpha_k (dalpha_k - sum_j alpha_j dalpha_j) and g_k = de_k *
    LeakyReLU'(pre_k); ds_l[v] = sum_k g_k."""
    dZd = np.asarray(dZ, np.float64)[:, :F]
    rows = fw["rows"]
    dalpha = np.einsum("kf,kf->k", dZd[rows], fw["X_rows"])
    c = np.zeros(n)
    np.add.at(c, rows, fw["alpha"] * dalpha)
    de = fw["alpha"] * (dalpha - c[rows])
    g = de * lrelu_grad(fw["pre"])
    ds_l = np.zeros(n)
    np.add.at(ds_l, rows, g)
    return dict(dalpha=dalpha, g=g, ds_l=ds_l)


def backward_plain(n, rowptr, col, Y, F, a_l, a_r, fw, dZ):
    """Without partitions: dY = A_alpha^T dZ + ds_r a_r + ds_l a_l, and the
    attention-vector gradients."""
    bs = backward_scores(n, rowptr, fw, dZ, F)
    dZd = np.asarray(dZ, np.float64)[:, :F]
    rows = fw["rows"]
    src = np.asarray(col, np.int64)
    dY = np.zeros((n, F))
    np.add.at(dY, src, fw["alpha"][:, None] * dZd[rows])
    ds_r = np.zeros(n)
    np.add.at(ds_r, src, bs["g"])
    a_l = np.asarray(a_l, np.float64)
    a_r = np.asarray(a_r, np.float64)
    dY += np.outer(ds_r, a_r) + np.outer(bs["ds_l"], a_l)
    Yd = np.asarray(Y, np.float64)[:, :F]
    return dict(dY=dY, da_l=bs["ds_l"] @ Yd, da_r=ds_r @ Yd, **bs)


def slot_messages_bwd(rowptr, bnd, dZ, F, a_r, alpha32, g32):
    """The backward message of every slot in the fixed fp32 order: start +0,
    entries v ascending, P = fl(P + fl(alpha_vs * dZ_v)); r = fixed-order fp32
    sum of g_vs; then P = fl(P + fl(r * a_r)).  alpha32 / g32 are the fp32
    attention and score gradients of the entries (col_remap order)."""
    S = bnd["n_slots"]
    srp, scol = bnd["slot_rowptr"], bnd["slot_col"]
    spos = slot_positions(rowptr, bnd)
    dZ32 = np.asarray(dZ, F32)[:, :F]
    a_r32 = np.asarray(a_r, F32)
    P = np.zeros((S, F), F32)
    r = np.zeros(S, F32)
    for s in range(S):
        for j in range(srp[s], srp[s + 1]):
            k = spos[j]
            P[s] = (P[s] + (F32(alpha32[k]) * dZ32[scol[j]]).astype(F32)).astype(F32)
            r[s] = F32(r[s] + F32(g32[k]))
        P[s] = (P[s] + (r[s] * a_r32).astype(F32)).astype(F32)
    return P, r


def slot_positions(rowptr, bnd):
    """For every slot-CSR entry (slot s, row v): the position, in col_remap
    order, of row v's remote entry that reads slot s."""
    cr = np.asarray(bnd["col_remap"], np.int64)
    n = bnd["n"]
    srp, scol = bnd["slot_rowptr"], bnd["slot_col"]
    S = bnd["n_slots"]
    pos = {}
    for v in range(n):
        for k in range(rowptr[v], rowptr[v + 1]):
            if cr[k] < 0:
                pos[(int(~cr[k]), v)] = k
    out = np.zeros(srp[-1] if S else 0, np.int64)
    for s in range(S):
        for j in range(srp[s], srp[s + 1]):
            out[j] = pos[(s, int(scol[j]))]
    return out


def transpose_positions(n, rowptr, cr):
    """For every local entry k of row u (col_remap order) reading v: the
    position of row v's local entry reading u; -1 for remote entries."""
    cr = np.asarray(cr, np.int64)
    rows = O.csr_rows(rowptr)
    pos = {}
    for k in range(cr.size):
        if cr[k] >= 0:
            pos[(int(rows[k]), int(cr[k]))] = k
    out = np.full(cr.size, -1, np.int64)
    for k in range(cr.size):
        if cr[k] >= 0:
            out[k] = pos[(int(cr[k]), int(rows[k]))]
    return out


def backward_partitioned(n, rowptr, Y, F, a_l, a_r, bnd, fw, dZ, slot_bits, seed, alpha32, g32,
                         Ydeq):
    """With partitions: the backward messages (fixed fp32 order, quantised with
    key s), the owner's dY (local transposed terms, own score terms and the
    dequantised messages it owns), and the attention-vector gradients (the
    remote score terms use the receiver's Y~)."""
    bs = backward_scores(n, rowptr, fw, dZ, F)
    cr = np.asarray(bnd["col_remap"], np.int64)
    rows = fw["rows"]
    dZd = np.asarray(dZ, np.float64)[:, :F]
    local = cr >= 0
    dY = np.zeros((n, F))
    np.add.at(dY, cr[local], fw["alpha"][local, None] * dZd[rows[local]])
    ds_r = np.zeros(n)
    np.add.at(ds_r, cr[local], bs["g"][local])
    a_l64 = np.asarray(a_l, np.float64)
    a_r64 = np.asarray(a_r, np.float64)
    dY += np.outer(ds_r, a_r64) + np.outer(bs["ds_l"], a_l64)
    P, r = slot_messages_bwd(rowptr, bnd, dZ, F, a_r, alpha32, g32)
    S = bnd["n_slots"]
    codes, meta = O.quantize(P, slot_bits, np.arange(S), seed)
    deq = O.dequantize(codes, meta, slot_bits).astype(np.float64)
    np.add.at(dY, np.asarray(bnd["slot_node"], np.int64), deq)
    Yd = np.asarray(Y, np.float64)[:, :F]
    Yq = np.asarray(Ydeq, np.float64)[:, :F]
    da_r = ds_r @ Yd + (r.astype(np.float64) @ Yq if S else 0.0)
    return dict(dY=dY, da_l=bs["ds_l"] @ Yd, da_r=da_r, P=P, r=r, codes=codes, meta=meta,
                deq=deq, **bs)
