"""Oracle: a plain CPU statement of the boundary-quantised GCN aggregation.

TEST INFRASTRUCTURE ONLY -- imported by tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  Arithmetic follows the
definitions directly; numpy/scipy primitives (sort, unique, sparse matmul)
serve as steps.  Floating point accumulates in fp64 except where a definition
fixes fp32 (the quantiser, dequantisation and the backward halo partial sums).

Sources (all from the SYLVIE guide "SYLVIE: 3D-adaptive and Universal System
for Large-scale Graph Neural Network Training"):
  * section 2 (message-passing GNN): the GCN layer
    z_v = sum_{u in N(v) + {v}} 1/sqrt(d_v d_u) W h_u,  h_v = sigma(z_v);
  * section 3 (inner / boundary nodes): which embeddings cross partitions,
    forward embeddings and backward embedding gradients;
  * section 6 (message quantisation): scale = (max - min)/(2^b - 1),
    q = stochastic_round((h - min)/scale), h~ = scale*q + min;
  * section 7 (data-dimension adaptivity): global in-degree, importance by
    percentile rank in the boundary pool (max degree -> 1, ties equal), the
    weight-gradient formula;
  * section 9 (combining node bits with the base width): the worked example;
  * section 11 (end-to-end pseudocode): the order quantise -> exchange ->
    dequantise -> aggregate, mirrored in the backward pass.

Readings where the pages are silent (all listed in the design notes):
degrees include the self-loop; one message slot per (boundary node, receiving
partition) pair; the hash is the MurmurHash3 32-bit finaliser composition
hash32(seed, s, j) = fmix32(fmix32(seed ^ fmix32(s)) ^ j); codes are packed
LSB-first into little-endian 32-bit words, each row padded to 16 bytes; the
backward halo partial sums run in a fixed fp32 order (ascending v).

Pins: every function here is checked by tests/test_oracle_pins.py against
published values, closed forms, invariants or brute force.
"""
from __future__ import annotations

import numpy as np
import scipy.sparse as sp

F32 = np.float32
U32 = np.uint32

FLAG_SYMMETRIZE = 1
FLAG_DEDUP = 2
FLAG_SELF_LOOPS = 4
FLAG_MEAN = 8
FLAGS_GCN = FLAG_SYMMETRIZE | FLAG_DEDUP | FLAG_SELF_LOOPS


# --------------------------------------------------------------------------
# hashing: MurmurHash3 32-bit finaliser (Appleby, SMHasher, public domain)
# --------------------------------------------------------------------------
def fmix32(h):
    h = np.asarray(h, dtype=np.uint64) & 0xFFFFFFFF
    h = h ^ (h >> 16)
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h = h ^ (h >> 13)
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h = h ^ (h >> 16)
    return h.astype(U32)


def hash32(seed, s, j):
    """hash32(seed, s, j) = fmix32(fmix32(seed ^ fmix32(s)) ^ j), broadcasting."""
    k = fmix32(np.uint64(seed & 0xFFFFFFFF) ^ fmix32(s).astype(np.uint64))
    return fmix32(k.astype(np.uint64) ^ (np.asarray(j, dtype=np.uint64) & 0xFFFFFFFF))


def sr_uniform(seed, s, j):
    """The stochastic-rounding offset u = (hash32 >> 8) * 2^-24 in [0, 1), fp32."""
    return (hash32(seed, s, j) >> U32(8)).astype(F32) * F32(2.0 ** -24)


# --------------------------------------------------------------------------
# a1: CSR with GCN normalisation (section 2)
# --------------------------------------------------------------------------
def csr_build(n, src, dst, flags=FLAGS_GCN):
    """Rows are destinations v, columns sources u.  Optionally symmetrise,
    deduplicate and give every node exactly one self-loop.  val = fp32 of
    1/sqrt(d_v * d_u) computed in fp64, d = row length (self-loop included);
    with FLAG_MEAN the GraphSAGE mean weight 1/d_v instead (section 2 names
    GraphSAGE's aggregator as the alternative; the mean over N(v) + {v} is
    the reading taken)."""
    src = np.asarray(src, np.int64)
    dst = np.asarray(dst, np.int64)
    rows, cols = dst, src
    if flags & FLAG_SYMMETRIZE:
        rows, cols = np.concatenate([dst, src]), np.concatenate([src, dst])
    if flags & FLAG_SELF_LOOPS:
        keep = rows != cols
        ids = np.arange(n, dtype=np.int64)
        rows = np.concatenate([rows[keep], ids])
        cols = np.concatenate([cols[keep], ids])
    key = rows * n + cols
    key = _distinct_sorted(key) if flags & FLAG_DEDUP else np.sort(key)
    rows, cols = key // n, key % n
    rowptr = np.zeros(n + 1, np.int64)
    rowptr[1:] = np.cumsum(np.bincount(rows, minlength=n))
    deg = np.diff(rowptr).astype(np.float64)
    if flags & FLAG_MEAN:
        val = (1.0 / deg[rows]).astype(F32)
    else:
        val = (1.0 / np.sqrt(deg[rows] * deg[cols])).astype(F32)
    return rowptr, cols.astype(np.int32), val


def transpose_values(n, rowptr, col, val):
    """A^T on A's own pattern (which must be symmetric): entry e = (v, u)
    receives the value of entry (u, v)."""
    rows = csr_rows(rowptr)
    key = rows * n + col.astype(np.int64)
    tkey = col.astype(np.int64) * n + rows
    at = np.searchsorted(key, tkey)
    assert np.all(at < key.size) and np.array_equal(key[np.minimum(at, key.size - 1)], tkey), \
        "pattern is not symmetric"
    return np.asarray(val)[at]


def _distinct_sorted(a):
    """Sorted distinct values of an integer array (sort, drop repeats)."""
    a = np.sort(np.asarray(a))
    if a.size < 2:
        return a
    return a[np.concatenate([[True], a[1:] != a[:-1]])]


def csr_rows(rowptr):
    return np.repeat(np.arange(rowptr.size - 1, dtype=np.int64), np.diff(rowptr))


# --------------------------------------------------------------------------
# a2: partitions, boundary slots and per-node bit widths (sections 3, 7, 9)
# --------------------------------------------------------------------------
def partition_starts(n, P):
    """Contiguous node blocks: start[p] = floor(p*n/P)."""
    return (np.arange(P + 1, dtype=np.int64) * n) // P


def part_of(x, starts):
    """p with start[p] <= x < start[p+1] (the non-empty block holding x)."""
    return np.searchsorted(starts, np.asarray(x, np.int64), side="right") - 1


def boundary_index(n, rowptr, col, val, P, val_t=None):
    """Slots are the pairs (q, u) where a node of partition q aggregates u and
    u is not in q; ordered by q then u.  Each row's entries are listed with
    local sources first (their ids) and remote ones after (~slot), both in CSR
    order, with the weights in the same order (and the A^T weights val_t, when
    given, as val_remap_t).  Returns a dict of the arrays."""
    starts = partition_starts(n, P)
    rows = csr_rows(rowptr)
    col64 = col.astype(np.int64)
    pv = part_of(rows, starts)
    pu = part_of(col64, starts)
    cut = pv != pu
    slot_keys = _distinct_sorted(pv[cut] * n + col64[cut])
    S = slot_keys.size
    slot_q = slot_keys // n
    slot_node = (slot_keys % n).astype(np.int32)
    send_start = np.searchsorted(slot_q, np.arange(P + 1), side="left").astype(np.int64)
    s_of_edge = np.searchsorted(slot_keys, pv[cut] * n + col64[cut])
    remap_csr = col.astype(np.int32).copy()
    remap_csr[cut] = ~s_of_edge.astype(np.int32)
    # each row's entries: local sources first, then remote slots, each group
    # in CSR order (a stable partition of the row)
    order = np.lexsort((np.arange(rows.size), cut, rows))
    col_remap = remap_csr[order]
    val_remap = val[order]
    extra = {} if val_t is None else dict(val_remap_t=np.asarray(val_t)[order])
    local_cnt = np.bincount(rows[~cut], minlength=n).astype(np.int32)
    ev = rows[cut]
    order = np.lexsort((ev, s_of_edge))
    slot_col = ev[order].astype(np.int32)
    slot_val = val[cut][order]
    slot_rowptr = np.zeros(S + 1, np.int64)
    slot_rowptr[1:] = np.cumsum(np.bincount(s_of_edge, minlength=S))
    own_slot = np.lexsort((np.arange(S), slot_node)).astype(np.int32)
    own_ptr = np.zeros(n + 1, np.int64)
    own_ptr[1:] = np.cumsum(np.bincount(slot_node, minlength=n))
    return dict(P=P, n=n, n_slots=S, nnz_cut=int(cut.sum()), part_start=starts,
                send_start=send_start, slot_node=slot_node, col_remap=col_remap,
                val_remap=val_remap, local_cnt=local_cnt,
                slot_rowptr=slot_rowptr, slot_col=slot_col, slot_val=slot_val,
                own_ptr=own_ptr, own_slot=own_slot, **extra)


def importance_counts(deg, pool):
    """c_u = #{w in pool : d_w <= d_u} and n = |pool|.  Importance is c_u/n:
    the max-degree node gets 1, equal degrees get equal importance, and it is
    unchanged by relabelling nodes (section 7)."""
    d_pool = np.sort(np.asarray(deg)[pool])
    c = np.searchsorted(d_pool, deg, side="right")
    return c.astype(np.int64), int(d_pool.size)


def mask_bits(c, n, pct, bits):
    """Discretise importance into levels: level = #{i : 100*c > pct[i]*n};
    mask bits = bits[level].  (A top-Q% rule is pct=[100-Q].)"""
    c = np.asarray(c, np.int64)
    level = np.zeros(c.shape, np.int64)
    for p in pct:
        level += (100 * c > int(p) * n)
    return np.asarray(bits, np.int64)[level]


def combine_and_clip(mask, base):
    """Per-node width = min(8, mask_bits * base) (section 9); 32 passes through."""
    mask = np.asarray(mask, np.int64)
    return np.where(mask == 32, 32, np.minimum(8, mask * int(base)))


def node_bits(n, rowptr, bnd, pct, bits, base):
    pool = np.diff(bnd["own_ptr"]) > 0
    deg = np.diff(rowptr)
    c, npool = importance_counts(deg, pool)
    nb = combine_and_clip(mask_bits(c, npool, pct, bits), base)
    return np.where(pool, nb, 0).astype(np.uint8)


def rowbytes(b, F):
    b = np.asarray(b, np.int64)
    return np.where(b == 32, 16 * ((4 * F + 15) // 16), 16 * ((F * b + 127) // 128))


def slot_offsets(slot_bits, F):
    off = np.zeros(len(slot_bits) + 1, np.int64)
    off[1:] = np.cumsum(rowbytes(slot_bits, F))
    return off


# --------------------------------------------------------------------------
# a3: stochastic integer quantisation, packing, dequantisation (section 6)
# --------------------------------------------------------------------------
def quantize(X, bits, keys, seed):
    """Quantise each row of X (fp32, [R, F]) with its own width.  Returns
    codes (uint32 [R, F]) and meta (fp32 [R, 2] = (min, scale)).  All steps
    are IEEE fp32 round-to-nearest: scale = (max - min)/(2^b - 1);
    t = (x - min)/scale; code = min(2^b - 1, floor(t + u)), u from hash32 with
    row key ``keys[r]`` and column j.  A constant row has scale 0 and codes 0.
    Zero min/max are stored as +0.  Width 32 stores the fp32 bits, meta (0,0)."""
    X = np.asarray(X, F32)
    R, F = X.shape
    bits = np.asarray(bits, np.int64)
    keys = np.asarray(keys, np.int64)
    codes = np.zeros((R, F), U32)
    meta = np.zeros((R, 2), F32)
    j = np.arange(F, dtype=np.int64)
    for b in np.unique(bits):
        rows = np.nonzero(bits == b)[0]
        x = X[rows]
        if b == 32:
            codes[rows] = x.view(U32)
            continue
        top = F32(2 ** int(b) - 1)
        mn = x.min(axis=1)
        mx = x.max(axis=1)
        mn[mn == 0] = F32(0.0)
        mx[mx == 0] = F32(0.0)
        flat = mx == mn
        scale = np.where(flat, F32(0.0), (mx - mn) / top).astype(F32)
        safe = np.where(flat, F32(1.0), scale).astype(F32)
        t = (x - mn[:, None]) / safe[:, None]
        u = sr_uniform(seed, keys[rows][:, None], j[None, :])
        c = np.minimum(np.floor(t + u), top).astype(U32)
        c[flat] = 0
        codes[rows] = c
        meta[rows, 0] = mn
        meta[rows, 1] = scale
    return codes, meta


def dequantize(codes, meta, bits):
    """h~ = scale * code + min, fp32 multiply then fp32 add; width 32 returns
    the stored fp32 values."""
    codes = np.asarray(codes, U32)
    bits = np.asarray(bits, np.int64)
    out = (meta[:, 1:2] * codes.astype(F32)) + meta[:, 0:1]
    wide = bits == 32
    if wide.any():
        out[wide] = codes[wide].view(F32)
    return out.astype(F32)


def pack(codes, bits, F, off, total=None):
    """Row r's code j occupies bits [b*(j % (32/b)), +b) of little-endian
    32-bit word floor(j*b/32) starting at byte off[r]; the row is zero-padded
    to rowbytes(b, F) = 16*ceil(F*b/128) bytes.  Width 32 stores raw fp32."""
    codes = np.asarray(codes, U32)
    bits = np.asarray(bits, np.int64)
    off = np.asarray(off, np.int64)
    if total is None:
        total = int((off[:bits.size] + rowbytes(bits, F)).max(initial=0))
    buf = np.zeros(total, np.uint8)
    for b in np.unique(bits):
        rows = np.nonzero(bits == b)[0]
        rb = int(rowbytes(b, F))
        nw = rb // 4
        if b == 32:
            words = np.zeros((rows.size, nw), U32)
            words[:, :F] = codes[rows]
        else:
            per = 32 // int(b)
            c = np.zeros((rows.size, nw * per), np.uint64)
            c[:, :F] = codes[rows]
            c = c.reshape(rows.size, nw, per)
            shifts = (np.arange(per, dtype=np.uint64) * np.uint64(b))[None, None, :]
            words = np.bitwise_or.reduce(c << shifts, axis=2).astype(U32)
        by = words.astype("<u4").view(np.uint8).reshape(rows.size, rb)
        buf[off[rows][:, None] + np.arange(rb)[None, :]] = by
    return buf


def unpack(buf, bits, F, off):
    """Inverse of ``pack``: codes (uint32 [R, F])."""
    bits = np.asarray(bits, np.int64)
    off = np.asarray(off, np.int64)
    R = bits.size
    codes = np.zeros((R, F), U32)
    for b in np.unique(bits):
        rows = np.nonzero(bits == b)[0]
        rb = int(rowbytes(b, F))
        by = buf[off[rows][:, None] + np.arange(rb)[None, :]]
        words = by.reshape(rows.size, rb).copy().view("<u4").astype(np.uint64)
        if b == 32:
            codes[rows] = words[:, :F].astype(U32)
            continue
        per = 32 // int(b)
        j = np.arange(F)
        w = words[:, j // per]
        sh = ((j % per) * int(b)).astype(np.uint64)
        codes[rows] = ((w >> sh[None, :]) & np.uint64((1 << int(b)) - 1)).astype(U32)
    return codes


def quant_pack(X, F, row_idx, bits, off, seed, total=None):
    """Quantise rows X[row_idx[r], :F] (row key r) and pack them: the message
    buffer and its meta, as the sender of section 11 produces them."""
    rows = np.asarray(X)[np.asarray(row_idx, np.int64), :F]
    codes, meta = quantize(rows, bits, np.arange(len(bits)), seed)
    return pack(codes, bits, F, off, total), meta, codes


# --------------------------------------------------------------------------
# a4: forward aggregation with dequantised remote rows (sections 2, 3, 6, 11)
# --------------------------------------------------------------------------
def _slot_messages(X, F, slot_node, slots, slot_bits, seed):
    """Dequantised message rows for ``slots`` (each quantised with key s)."""
    rows = np.asarray(X)[slot_node[slots].astype(np.int64), :F]
    codes, meta = quantize(rows, slot_bits[slots], slots, seed)
    return dequantize(codes, meta, slot_bits[slots])


def spmm_fwd(n, rowptr, col, val, H, F, bnd=None, slot_bits=None, seed=0, rows=None, H_msg=None):
    """M[v] = sum_e val[e] * x_e, where x_e = H[u] for a local source u and the
    dequantised message of slot (part(v), u) for a remote one.  Accumulates in
    fp64; also returns T[v] = sum_e |val[e] * x_e| (for error bounds).
    ``rows`` selects output rows (default all).  ``H_msg``: the matrix the
    messages are formed from (default H); in an asynchronous epoch (section
    10) it is the previous epoch's layer input and ``seed`` that epoch's."""
    rows = np.arange(n, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    lens = rowptr[rows + 1] - rowptr[rows]
    e = _expand_ranges(rowptr[rows], lens)
    out_row = np.repeat(np.arange(rows.size), lens)
    w = (val if bnd is None else bnd["val_remap"])[e].astype(np.float64)
    if bnd is None:
        src_id = col[e].astype(np.int64)
        uniq, inv = np.unique(src_id, return_inverse=True)
        X = np.asarray(H)[uniq, :F].astype(np.float64)
    else:
        cr = bnd["col_remap"][e].astype(np.int64)
        remote = cr < 0
        key = np.where(remote, n + ~cr, cr)
        uniq, inv = np.unique(key, return_inverse=True)
        loc = uniq[uniq < n]
        slots = uniq[uniq >= n] - n
        X = np.zeros((uniq.size, F), np.float64)
        X[: loc.size] = np.asarray(H)[loc, :F]
        if slots.size:
            Xm = H if H_msg is None else H_msg
            X[loc.size:] = _slot_messages(Xm, F, bnd["slot_node"], slots, slot_bits, seed)
    A = sp.csr_matrix((w, (out_row, inv)), shape=(rows.size, uniq.size))
    M = A @ X
    T = abs(A) @ np.abs(X)
    return M, T


def _expand_ranges(starts, lens):
    total = int(lens.sum())
    if total == 0:
        return np.zeros(0, np.int64)
    base = np.repeat(starts - np.concatenate([[0], np.cumsum(lens)[:-1]]), lens)
    return base + np.arange(total, dtype=np.int64)


# --------------------------------------------------------------------------
# a7 / a8: backward halo partials and local transpose aggregation (section 3)
# --------------------------------------------------------------------------
def slot_partials(bnd, G, F, slots=None):
    """Gradient partial of each halo copy, P_s = sum_{v in q} A_vu G[v], in the
    fixed fp32 order: start +0, entries by ascending v, product rounded to fp32
    then sum rounded to fp32."""
    S = bnd["n_slots"]
    slots = np.arange(S, dtype=np.int64) if slots is None else np.asarray(slots, np.int64)
    srp, scol, sval = bnd["slot_rowptr"], bnd["slot_col"], bnd["slot_val"]
    lens = srp[slots + 1] - srp[slots]
    order = np.argsort(-lens, kind="stable")
    acc = np.zeros((slots.size, F), F32)
    G = np.asarray(G)
    for k in range(int(lens.max(initial=0))):
        m = int(np.count_nonzero(lens[order] > k))
        idx = order[:m]
        ent = srp[slots[idx]] + k
        prod = (sval[ent][:, None] * G[scol[ent].astype(np.int64), :F]).astype(F32)
        acc[idx] = (acc[idx] + prod).astype(F32)
    return acc


def spmm_bwd(n, rowptr, col, val, G, F, bnd=None, slot_bits=None, seed=0, rows=None, G_msg=None):
    """dH = A^T G.  With partitions (A's pattern symmetric): dH[u] = sum of
    A_vu G[v] over local v -- A_vu is val_remap_t when the boundary has it,
    else A is symmetric and val_remap serves -- plus the dequantised halo
    partials of every slot u owns
    (each quantised with key s and ``seed``).  fp64 accumulation; returns
    (dH, T) for ``rows`` (default all).  ``G_msg``: the matrix the halo
    partials are formed from (default G; the previous epoch's in an
    asynchronous epoch, section 10)."""
    rows = np.arange(n, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    if bnd is None:
        A = sp.csr_matrix((val.astype(np.float64), col.astype(np.int64), rowptr), shape=(n, n))
        At = A.T.tocsr()[rows]
        Gd = np.asarray(G)[:, :F].astype(np.float64)
        return At @ Gd, abs(At) @ np.abs(Gd)
    lens = rowptr[rows + 1] - rowptr[rows]
    e = _expand_ranges(rowptr[rows], lens)
    out_row = np.repeat(np.arange(rows.size), lens)
    cr = bnd["col_remap"][e]
    loc = cr >= 0
    src = cr[loc].astype(np.int64)
    uniq, inv = np.unique(src, return_inverse=True)
    wt = bnd["val_remap_t"] if "val_remap_t" in bnd else bnd["val_remap"]
    A = sp.csr_matrix((wt[e][loc].astype(np.float64), (out_row[loc], inv)),
                      shape=(rows.size, uniq.size))
    Xl = np.asarray(G)[uniq, :F].astype(np.float64)
    dH = A @ Xl
    T = abs(A) @ np.abs(Xl)
    own_ptr, own_slot = bnd["own_ptr"], bnd["own_slot"]
    olens = own_ptr[rows + 1] - own_ptr[rows]
    if olens.sum():
        oi = _expand_ranges(own_ptr[rows], olens)
        slots = own_slot[oi].astype(np.int64)
        orow = np.repeat(np.arange(rows.size), olens)
        part = slot_partials(bnd, G if G_msg is None else G_msg, F, slots)
        codes, meta = quantize(part, slot_bits[slots], slots, seed)
        deq = dequantize(codes, meta, slot_bits[slots]).astype(np.float64)
        np.add.at(dH, orow, deq)
        np.add.at(T, orow, np.abs(deq))
    return dH, T


def halo_quant_pack(bnd, G, F, slot_bits, slot_off, seed):
    """Backward messages: slot partials quantised with key s and packed."""
    S = bnd["n_slots"]
    part = slot_partials(bnd, G, F)
    codes, meta = quantize(part, slot_bits, np.arange(S), seed)
    return pack(codes, slot_bits, F, slot_off), meta, codes


# --------------------------------------------------------------------------
# a5 / a6: dense transform and its backward (sections 2 and 7)
# --------------------------------------------------------------------------
def bf16_round(x):
    """fp32 -> nearest bf16 value (ties to even), returned as fp32.  Finite
    inputs only."""
    u = np.asarray(x, F32).view(U32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(U32).view(F32)


def dense_fwd(Mb, W, relu):
    """Z = Mb W in fp64 on bf16 inputs; H' = ReLU(Z) when ``relu``."""
    Z = np.asarray(Mb, np.float64) @ np.asarray(W, np.float64)
    return Z, (np.maximum(Z, 0.0) if relu else Z)


def dense_bwd(Mb, W, dH_out, H_out, relu):
    """dZ = dH' * 1[Z > 0] (1[Z>0] = 1[ReLU(Z)>0]), rounded to bf16; then
    dM = dZ W^T and dW = Mb^T dZ in fp64 (section 7's weight gradient with the
    aggregation already applied in Mb)."""
    dZ = np.asarray(dH_out, F32)
    if relu:
        dZ = np.where(np.asarray(H_out) > 0, dZ, F32(0.0)).astype(F32)
    dZb = bf16_round(dZ).astype(np.float64)
    Wd = np.asarray(W, np.float64)
    return dZb @ Wd.T, np.asarray(Mb, np.float64).T @ dZb, dZb


def gemm_abs(A, B):
    """sum_k |A_ik B_kj|: the scale for GEMM error bounds."""
    return np.abs(np.asarray(A, np.float64)) @ np.abs(np.asarray(B, np.float64))
