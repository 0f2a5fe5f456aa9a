"""Pins for the oracle: published values, closed forms, invariants and brute
force on tiny inputs.  Each check is chosen so that a plausible slip in the
oracle (a dropped term, a wrong index or sign, a transposed operand, an
off-by-one in the packing) fails at least one of them."""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O
from synth import circulant_edges, erdos_renyi_edges, star_edges, planted_partition_edges

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------ hashing
def test_fmix32_published_vectors():
    for key, seed, want in _golden_lines("murmur3_x86_32.txt"):
        seed, want = int(seed, 16), int(want, 16)
        if key == "-":
            got = int(O.fmix32(seed ^ 0))
        else:
            # one all-zero 4-byte block: the block mix leaves h = rotl(seed,13)*5+c
            h = ((seed << 13) | (seed >> 19)) & 0xFFFFFFFF
            h = (h * 5 + 0xE6546B64) & 0xFFFFFFFF
            got = int(O.fmix32(h ^ 4))
        assert got == want, (key, hex(got), hex(want))


def test_sr_uniform_is_uniform():
    # chi-square of u over 256 equal bins, 2^18 draws: 255 dof, mean 255,
    # sd ~22.6; 400 is > 6 sd.
    s = np.repeat(np.arange(512), 512)
    j = np.tile(np.arange(512), 512)
    u = O.sr_uniform(12345, s, j)
    assert u.dtype == np.float32 and u.min() >= 0 and u.max() < 1
    h = np.bincount((u * 256).astype(np.int64), minlength=256)
    e = u.size / 256
    chi2 = ((h - e) ** 2 / e).sum()
    assert chi2 < 400, chi2


# ------------------------------------------------------------------ CSR
def _dense_adj(n, src, dst):
    A = np.zeros((n, n), bool)
    for a, b in zip(src, dst):
        if a != b:
            A[a, b] = A[b, a] = True
    for i in range(n):
        A[i, i] = True
    return A


@pytest.mark.parametrize("n,p,seed", [(1, 0.0, 0), (7, 0.5, 1), (40, 0.2, 2), (64, 0.05, 3)])
def test_csr_bruteforce(n, p, seed):
    src, dst = erdos_renyi_edges(n, p, seed)
    # duplicate and reversed copies must not change the result
    src2 = np.concatenate([src, dst[: len(dst) // 2]])
    dst2 = np.concatenate([dst, src[: len(src) // 2]])
    rowptr, col, val = O.csr_build(n, src2, dst2)
    A = _dense_adj(n, src, dst)
    for v in range(n):
        cols = [u for u in range(n) if A[v, u]]
        assert list(col[rowptr[v]:rowptr[v + 1]]) == cols
    deg = A.sum(1)
    for v in range(n):
        for k in range(rowptr[v], rowptr[v + 1]):
            u = col[k]
            want = np.float32(1.0 / math.sqrt(float(deg[v]) * float(deg[u])))
            assert val[k] == want


def test_csr_flags_without_symmetrize():
    # directed edges u->v land in row v only; no dedup keeps repeats
    rowptr, col, val = O.csr_build(3, [0, 0, 1], [1, 1, 2], flags=O.FLAG_SELF_LOOPS)
    assert list(rowptr) == [0, 1, 4, 6]
    assert list(col) == [0, 0, 0, 1, 1, 2]


@pytest.mark.parametrize("n,d", [(64, 3), (256, 15), (512, 63), (300, 8)])
def test_regular_graph_constant_features_fixed_point(n, d):
    """d-regular graph with self-loops: every weight is 1/(d+1), so a constant
    feature column is reproduced; bit-exactly when d+1 is a power of two."""
    src, dst = circulant_edges(n, d)
    rowptr, col, val = O.csr_build(n, src, dst)
    assert np.all(np.diff(rowptr) == d + 1)
    H = np.full((n, 4), 0.75, np.float32)
    H[:, 1] = -3.0
    M, T = O.spmm_fwd(n, rowptr, col, val, H, 4)
    if (d + 1) & d == 0:
        assert np.array_equal(M, H.astype(np.float64))
    else:
        assert np.allclose(M, H, rtol=1e-6, atol=0)


# ------------------------------------------------------------------ aggregation
def _dense_ahat(n, rowptr, col, val):
    A = np.zeros((n, n))
    for v in range(n):
        for k in range(rowptr[v], rowptr[v + 1]):
            A[v, col[k]] = float(val[k])
    return A


@pytest.mark.parametrize("n,p,seed", [(5, 0.6, 4), (33, 0.15, 5), (64, 0.1, 6)])
def test_spmm_dense_bruteforce_and_adjoint(n, p, seed):
    src, dst = erdos_renyi_edges(n, p, seed)
    rowptr, col, val = O.csr_build(n, src, dst)
    A = _dense_ahat(n, rowptr, col, val)
    rng = np.random.default_rng(seed)
    F = 5
    H = rng.standard_normal((n, F)).astype(np.float32)
    G = rng.standard_normal((n, F)).astype(np.float32)
    M, T = O.spmm_fwd(n, rowptr, col, val, H, F)
    want = np.zeros((n, F))
    for v in range(n):
        for u in range(n):
            want[v] += A[v, u] * H[u].astype(np.float64)
    assert np.allclose(M, want, rtol=0, atol=1e-13)
    assert np.allclose(T, np.abs(A) @ np.abs(H.astype(np.float64)), atol=1e-13)
    dH, _ = O.spmm_bwd(n, rowptr, col, val, G, F)
    assert np.allclose(dH, A.T @ G.astype(np.float64), atol=1e-13)
    lhs = float(np.sum(M * G))
    rhs = float(np.sum(H.astype(np.float64) * dH))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


# ------------------------------------------------------------------ boundary
def _bruteforce_boundary(n, rowptr, col, P):
    starts = [(p * n) // P for p in range(P + 1)]

    def part(x):
        return max(p for p in range(P) if starts[p] <= x < starts[p + 1])

    pairs = set()
    for v in range(n):
        for k in range(rowptr[v], rowptr[v + 1]):
            u = int(col[k])
            if part(u) != part(v):
                pairs.add((part(v), u))
    return sorted(pairs), part


@pytest.mark.parametrize("n,p,P,seed", [(12, 0.3, 3, 7), (64, 0.1, 4, 8), (50, 0.2, 7, 9), (3, 1.0, 5, 1)])
def test_boundary_bruteforce(n, p, P, seed):
    src, dst = erdos_renyi_edges(n, p, seed)
    rowptr, col, val = O.csr_build(n, src, dst)
    b = O.boundary_index(n, rowptr, col, val, P)
    slots, part = _bruteforce_boundary(n, rowptr, col, P)
    assert b["n_slots"] == len(slots)
    assert [(part(0) * 0 + q, int(u)) for q, u in slots] == \
        [(int(q), int(u)) for q, u in zip(np.repeat(np.arange(P), np.diff(b["send_start"])), b["slot_node"])]
    index = {sl: s for s, sl in enumerate(slots)}
    for v in range(n):
        ks = range(rowptr[v], rowptr[v + 1])
        local = [(int(col[k]), val[k]) for k in ks if part(int(col[k])) == part(v)]
        remote = [(~index[(part(v), int(col[k]))], val[k]) for k in ks if part(int(col[k])) != part(v)]
        want = local + remote
        got = list(zip(b["col_remap"][rowptr[v]:rowptr[v + 1]], b["val_remap"][rowptr[v]:rowptr[v + 1]]))
        assert [(int(c), float(w)) for c, w in got] == [(c, float(w)) for c, w in want]
        assert b["local_cnt"][v] == len(local)
    for s, (q, u) in enumerate(slots):
        ents = [(v, val[k]) for v in range(n) if part(v) == q
                for k in range(rowptr[v], rowptr[v + 1]) if col[k] == u]
        got = list(zip(b["slot_col"][b["slot_rowptr"][s]:b["slot_rowptr"][s + 1]],
                       b["slot_val"][b["slot_rowptr"][s]:b["slot_rowptr"][s + 1]]))
        assert [(int(a), float(c)) for a, c in got] == [(a, float(c)) for a, c in ents]
    for u in range(n):
        owned = [s for s, (q, uu) in enumerate(slots) if uu == u]
        assert list(b["own_slot"][b["own_ptr"][u]:b["own_ptr"][u + 1]]) == owned


def test_partition_of_empty_blocks():
    starts = O.partition_starts(2, 4)
    assert list(starts) == [0, 0, 1, 1, 2]
    assert list(O.part_of([0, 1], starts)) == [1, 3]


# ------------------------------------------------------------------ importance, bits
def test_combine_and_clip_worked_example():
    lines = _golden_lines("combine_and_clip.txt")
    mask = [int(x) for x in lines[0][2:]]
    for row in lines[1:]:
        base = int(row[0])
        want = [int(x) for x in row[2:]]
        assert list(O.combine_and_clip(mask, base)) == want


def test_importance_properties():
    rng = np.random.default_rng(3)
    deg = rng.integers(1, 9, 200)
    pool = rng.random(200) < 0.6
    c, n = O.importance_counts(deg, pool)
    # brute force count
    for u in range(200):
        assert c[u] == sum(1 for w in range(200) if pool[w] and deg[w] <= deg[u])
    # max-degree pool node has importance 1; ties equal
    top = np.argmax(np.where(pool, deg, -1))
    assert c[top] == n
    for a, b in itertools.combinations(np.nonzero(pool)[0][:40], 2):
        if deg[a] == deg[b]:
            assert c[a] == c[b]
    # relabelling invariance
    perm = rng.permutation(200)
    c2, n2 = O.importance_counts(deg[perm], pool[perm])
    assert n2 == n and np.array_equal(c2, c[perm])


def test_mask_bits_top_and_quartiles():
    n = 10
    c = np.arange(1, 11)
    # top 20%: the two highest ranks
    assert list(O.mask_bits(c, n, [80], [4, 8])) == [4] * 8 + [8] * 2
    q = O.mask_bits(np.arange(1, 9), 8, [25, 50, 75], [1, 2, 4, 8])
    assert list(q) == [1, 1, 2, 2, 4, 4, 8, 8]
    # ties at the threshold are all promoted
    assert list(O.mask_bits([3, 3, 3, 1], 4, [50], [2, 8])) == [8, 8, 8, 2]


# ------------------------------------------------------------------ quantiser
@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_quantize_range_and_step_bound(b):
    rng = np.random.default_rng(b)
    X = (rng.standard_normal((64, 37)) * 3).astype(np.float32)
    codes, meta = O.quantize(X, np.full(64, b), np.arange(64), seed=99)
    assert codes.max() <= 2 ** b - 1
    mn, scale = meta[:, 0], meta[:, 1]
    assert np.array_equal(mn, X.min(1))
    assert np.all(scale == ((X.max(1) - X.min(1)) / np.float32(2 ** b - 1)).astype(np.float32))
    # every row reaches near both ends of the grid
    xt = O.dequantize(codes, meta, np.full(64, b))
    ulp = np.spacing(np.maximum(np.abs(X.min(1)), np.abs(X.max(1))).astype(np.float32))
    assert np.all(np.abs(xt - X) <= scale[:, None] + 2 * ulp[:, None])


def test_quantize_constant_row_and_signed_zero():
    X = np.array([[2.5] * 6, [-0.0, 0.0, -0.0, 0.0, 0.0, -0.0]], np.float32)
    codes, meta = O.quantize(X, [4, 2], [0, 1], seed=1)
    assert np.all(codes == 0)
    assert meta[0, 0] == 2.5 and meta[0, 1] == 0
    assert np.signbit(meta[1, 0]) == False and meta[1, 1] == 0  # noqa: E712
    xt = O.dequantize(codes, meta, [4, 2])
    assert np.all(xt[0] == 2.5) and np.all(xt[1] == 0)


def test_quantize_integer_grid_is_exact():
    """x = mn + k*scale exactly representable: t = k, so code = k (only an
    offset u within half an ulp of 1 could round k+u up to k+1)."""
    k = np.arange(256, dtype=np.float32)
    X = np.stack([-64.0 + 0.5 * k, 3.0 + 0.25 * k]).astype(np.float32)
    codes, meta = O.quantize(X, [8, 8], [5, 6], seed=77)
    u = O.sr_uniform(77, np.array([[5], [6]]), np.arange(256)[None, :])
    expect = np.where((k[None, :] + u) >= k[None, :] + 1, k + 1, k)
    assert np.array_equal(codes, np.minimum(expect, 255).astype(np.uint32))
    assert np.array_equal(O.dequantize(codes, meta, [8, 8]), X)


def test_stochastic_rounding_unbiased_and_variance_law():
    """E[deq(q(x))] = x and the mean squared error over uniform fractional
    parts is D*scale^2/6 (section 6).  10^4 seeds, deterministic."""
    D, b = 1024, 2
    rng = np.random.default_rng(11)
    X = rng.uniform(-1, 1, (1, D)).astype(np.float32)
    X[0, 0], X[0, 1] = -1.0, 1.0
    seeds = 10000
    total = np.zeros(D)
    sq = np.zeros(D)
    for sd in range(seeds):
        c, m = O.quantize(X, [b], [0], seed=sd)
        xt = O.dequantize(c, m, [b])[0].astype(np.float64)
        total += xt
        sq += (xt - X[0]) ** 2
    mean = total / seeds
    scale = float(m[0, 1])
    t = (X[0].astype(np.float64) - float(m[0, 0])) / scale
    f = t - np.floor(t)
    sigma = scale * np.sqrt(f * (1 - f)) / np.sqrt(seeds)
    z = (mean - X[0]) / np.where(sigma > 0, sigma, 1)
    inner = sigma > 0
    assert np.mean(np.abs(z[inner]) > 3) <= 0.005
    assert np.max(np.abs(z[inner])) <= 4.5
    assert np.all(np.abs(mean[~inner] - X[0][~inner]) <= 2 * np.spacing(np.abs(X[0][~inner]) + 1e-30) + 1e-12)
    mse_sum = sq.sum() / seeds
    law = D * scale ** 2 / 6
    assert abs(mse_sum - law) / law < 0.05


@pytest.mark.parametrize("F", [1, 5, 16, 37, 100, 129])
def test_pack_layout_and_roundtrip(F):
    rng = np.random.default_rng(F)
    bits = np.array([1, 2, 4, 8, 32, 8, 1, 4])
    codes = np.zeros((bits.size, F), np.uint32)
    for r, b in enumerate(bits):
        codes[r] = rng.integers(0, 2 ** min(int(b), 31), F) if b < 32 else \
            rng.standard_normal(F).astype(np.float32).view(np.uint32)
    off = O.slot_offsets(bits, F)
    assert np.all(off % 16 == 0)
    buf = O.pack(codes, bits, F, off[:-1], int(off[-1]))
    assert buf.size == off[-1]
    assert np.array_equal(O.unpack(buf, bits, F, off[:-1]), codes)
    # bit-level layout by brute force: code j of row r at bit b*(j%(32/b)) of word j*b//32
    for r, b in enumerate(bits):
        b = int(b)
        rb = int(O.rowbytes(b, F))
        assert rb == (16 * math.ceil(F * b / 128) if b < 32 else 16 * math.ceil(4 * F / 16))
        row = buf[off[r]:off[r] + rb]
        allbits = np.unpackbits(row, bitorder="little")
        for j in range(F):
            v = int(codes[r, j])
            start = j * b
            got = sum(int(allbits[start + i]) << i for i in range(b))
            assert got == v
        assert not allbits[F * b:].any()


# ------------------------------------------------------------------ partitioned paths
def _tiny_graph(n=96, P=4, seed=3):
    src, dst = planted_partition_edges(n, 300, 4, 0.85, seed)
    rowptr, col, val = O.csr_build(n, src, dst)
    b = O.boundary_index(n, rowptr, col, val, P)
    return rowptr, col, val, b


def test_fwd_passthrough_partition_equals_plain():
    """Width 32 sends exact fp32 rows, so partitioning changes nothing
    (switching quantisation off recovers the unapproximated run, section 16)."""
    n = 96
    rowptr, col, val, b = _tiny_graph(n)
    H = np.random.default_rng(1).standard_normal((n, 9)).astype(np.float32)
    bits = np.full(b["n_slots"], 32)
    M0, T0 = O.spmm_fwd(n, rowptr, col, val, H, 9)
    M1, T1 = O.spmm_fwd(n, rowptr, col, val, H, 9, b, bits, seed=3)
    assert np.allclose(M0, M1, rtol=0, atol=1e-14)
    G = np.random.default_rng(2).standard_normal((n, 9)).astype(np.float32)
    d0, t0 = O.spmm_bwd(n, rowptr, col, val, G, 9)
    d1, t1 = O.spmm_bwd(n, rowptr, col, val, G, 9, b, bits, seed=4)
    # halo partials are fp32 sums: within fp32 rounding of the terms
    assert np.all(np.abs(d0 - d1) <= 1e-6 * t0 + 1e-12)


def test_fwd_quantised_rows_use_their_slot_message():
    """Each remote edge sees the message of its own (receiving partition,
    node) slot: check one row against a hand-built sum."""
    n = 96
    rowptr, col, val, b = _tiny_graph(n)
    H = np.random.default_rng(5).standard_normal((n, 7)).astype(np.float32)
    bits = np.where(np.arange(b["n_slots"]) % 2 == 0, 2, 8)
    M, _ = O.spmm_fwd(n, rowptr, col, val, H, 7, b, bits, seed=8)
    starts = O.partition_starts(n, 4)
    for v in [0, 30, 50, 95]:
        acc = np.zeros(7)
        for k in range(rowptr[v], rowptr[v + 1]):
            u = int(col[k])
            if O.part_of(u, starts) == O.part_of(v, starts):
                x = H[u].astype(np.float64)
            else:
                s = int(np.searchsorted(b["slot_node"][b["send_start"][O.part_of(v, starts)]:], u)
                        + b["send_start"][O.part_of(v, starts)])
                assert b["slot_node"][s] == u
                c, m = O.quantize(H[u:u + 1], [bits[s]], [s], seed=8)
                x = O.dequantize(c, m, [bits[s]])[0].astype(np.float64)
            acc += float(val[k]) * x
        assert np.allclose(M[v], acc, rtol=0, atol=1e-12)


def test_slot_partials_fixed_order():
    n = 96
    rowptr, col, val, b = _tiny_graph(n)
    G = np.random.default_rng(6).standard_normal((n, 3)).astype(np.float32)
    P = O.slot_partials(b, G, 3)
    for s in range(0, b["n_slots"], 7):
        acc = np.zeros(3, np.float32)
        for k in range(b["slot_rowptr"][s], b["slot_rowptr"][s + 1]):
            prod = np.float32(b["slot_val"][k]) * G[b["slot_col"][k]]
            acc = (acc + prod.astype(np.float32)).astype(np.float32)
        assert np.array_equal(P[s], acc)
        # and the entries are the A_vu of the slot's node
        u = b["slot_node"][s]
        for k in range(b["slot_rowptr"][s], b["slot_rowptr"][s + 1]):
            v = b["slot_col"][k]
            kk = rowptr[v] + np.searchsorted(col[rowptr[v]:rowptr[v + 1]], u)
            assert col[kk] == u and val[kk] == b["slot_val"][k]


def test_bwd_quantised_is_sum_of_local_and_owned_messages():
    n = 96
    rowptr, col, val, b = _tiny_graph(n)
    G = np.random.default_rng(7).standard_normal((n, 4)).astype(np.float32)
    bits = np.full(b["n_slots"], 4)
    dH, _ = O.spmm_bwd(n, rowptr, col, val, G, 4, b, bits, seed=5)
    part = O.slot_partials(b, G, 4)
    c, m = O.quantize(part, bits, np.arange(b["n_slots"]), seed=5)
    deq = O.dequantize(c, m, bits)
    starts = O.partition_starts(n, 4)
    for u in [1, 40, 77]:
        acc = np.zeros(4)
        for k in range(rowptr[u], rowptr[u + 1]):
            v = int(col[k])
            if O.part_of(u, starts) == O.part_of(v, starts):
                acc += float(val[k]) * G[v].astype(np.float64)
        for s in range(b["n_slots"]):
            if b["slot_node"][s] == u:
                acc += deq[s].astype(np.float64)
        assert np.allclose(dH[u], acc, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ dense
def test_bf16_round_ties_to_even():
    one = 1.0
    vals = np.array([one, one + 2 ** -8, one + 3 * 2 ** -8, one + 2 ** -7 + 2 ** -9, -2.5,
                     3.0e38, 1e-40], np.float32)
    want = np.array([one, one, one + 2 ** -6, one + 2 ** -7, -2.5], np.float32)
    got = O.bf16_round(vals)
    assert np.array_equal(got[:5], want)
    # every result is a bf16 value and the nearest one
    assert np.all(got.view(np.uint32) & 0xFFFF == 0)
    for x, g in zip(vals, got):
        up = (np.float32(g).view(np.uint32) + np.uint32(0x10000)).view(np.float32)
        dn = (np.float32(g).view(np.uint32) - np.uint32(0x10000)).view(np.float32)
        assert abs(float(g) - float(x)) <= min(abs(float(up) - float(x)), abs(float(dn) - float(x)))


def test_weight_gradient_matches_finite_differences():
    """Layer backward against finite differences of L = <H', G> with the
    section 7 weight-gradient formula: dW = sum_v (dL/dh'_v * sigma'(z_v)) m_v^T."""
    rng = np.random.default_rng(9)
    N, Fi, Fo = 12, 5, 4
    Mb = rng.standard_normal((N, Fi))
    W = rng.standard_normal((Fi, Fo))
    G = rng.standard_normal((N, Fo)).astype(np.float32)
    Z, Hn = O.dense_fwd(Mb, W, relu=True)
    dM, dW, dZb = O.dense_bwd(Mb, W, G, Hn, relu=True)
    # dZ is bf16-rounded inside dense_bwd; compare with the unrounded formula
    eps = 1e-6
    num = np.zeros_like(W)
    for i in range(Fi):
        for j in range(Fo):
            Wp = W.copy(); Wp[i, j] += eps
            Wm = W.copy(); Wm[i, j] -= eps
            num[i, j] = (np.sum(O.dense_fwd(Mb, Wp, True)[1] * G) -
                         np.sum(O.dense_fwd(Mb, Wm, True)[1] * G)) / (2 * eps)
    assert np.allclose(dW, num, rtol=1e-2, atol=1e-2)  # bf16 rounding of dZ
    numM = np.zeros_like(Mb)
    for i in range(N):
        for j in range(Fi):
            Mp = Mb.copy(); Mp[i, j] += eps
            Mm = Mb.copy(); Mm[i, j] -= eps
            numM[i, j] = (np.sum(O.dense_fwd(Mp, W, True)[1] * G) -
                          np.sum(O.dense_fwd(Mm, W, True)[1] * G)) / (2 * eps)
    assert np.allclose(dM, numM, rtol=1e-2, atol=1e-2)


def test_quantize_divides_rather_than_multiplies_by_reciprocal():
    """On rows x = k*s (k = 0..255, mn = 0, max = 255*s exact) with s not a
    power of two, t = (x - mn)/s is exactly k, so the code is k unless
    k + u rounds up to k + 1.  A reciprocal multiply lands a hair below k for
    some k and yields k - 1 whenever u is tiny; 4096 row keys make sure such
    u values occur."""
    k = np.arange(256, dtype=np.float32)
    rows = []
    for i in range(4096):
        s = np.float32((3 + 2 * (i % 61)) * 2.0 ** (-(i % 7) - 3))
        rows.append(k * s)
    X = np.stack(rows).astype(np.float32)
    R = X.shape[0]
    codes, meta = O.quantize(X, np.full(R, 8), np.arange(R), seed=2024)
    for r in range(R):
        assert meta[r, 1] == X[r, 1]  # scale recovered exactly
    u = O.sr_uniform(2024, np.arange(R)[:, None], np.arange(256)[None, :])
    kk = np.broadcast_to(k, (R, 256))
    expect = np.where((kk + u).astype(np.float32) >= kk + 1, kk + 1, kk)
    assert np.array_equal(codes, np.minimum(expect, 255).astype(np.uint32))


# ------------------------------------------------------------------ mean aggregation (GraphSAGE)
@pytest.mark.parametrize("n,p,seed", [(7, 0.5, 11), (40, 0.2, 12), (64, 0.08, 13)])
def test_mean_csr_and_transpose_bruteforce(n, p, seed):
    """Mean weights are 1/d_v on row v (d with the self-loop); the A^T
    weights on the same pattern are 1/d_u; for GCN weights A^T = A."""
    src, dst = erdos_renyi_edges(n, p, seed)
    rowptr, col, val = O.csr_build(n, src, dst, O.FLAGS_GCN | O.FLAG_MEAN)
    A = _dense_adj(n, src, dst)
    deg = A.sum(1)
    Am = A / deg[:, None].astype(np.float64)
    for v in range(n):
        assert list(col[rowptr[v]:rowptr[v + 1]]) == [u for u in range(n) if A[v, u]]
        for k in range(rowptr[v], rowptr[v + 1]):
            assert val[k] == np.float32(1.0 / float(deg[v]))
    vt = O.transpose_values(n, rowptr, col, val)
    D = _dense_ahat(n, rowptr, col, val)
    Dt = _dense_ahat(n, rowptr, col, vt)
    assert np.array_equal(Dt, D.T)
    assert np.allclose(D, Am, rtol=1e-7, atol=0)
    r2, c2, v2 = O.csr_build(n, src, dst)
    assert np.array_equal(O.transpose_values(n, r2, c2, v2), v2)


def test_transpose_values_rejects_unsymmetric_pattern():
    rowptr, col, val = O.csr_build(3, [0, 1], [1, 2], flags=O.FLAG_SELF_LOOPS | O.FLAG_MEAN)
    with pytest.raises(AssertionError):
        O.transpose_values(3, rowptr, col, val)


@pytest.mark.parametrize("seed", [0, 1])
def test_mean_reproduces_constant_rows_on_irregular_graphs(seed):
    """The mean of a constant column is that constant whatever the degrees;
    GCN weights do not have this property on an irregular graph."""
    n = 300
    src, dst = planted_partition_edges(n, 900, 3, 0.8, seed)
    H = np.full((n, 3), 1.5, np.float32)
    H[:, 2] = -0.25
    rowptr, col, val = O.csr_build(n, src, dst, O.FLAGS_GCN | O.FLAG_MEAN)
    M, _ = O.spmm_fwd(n, rowptr, col, val, H, 3)
    assert np.allclose(M, H, rtol=2e-7, atol=0)
    r2, c2, v2 = O.csr_build(n, src, dst)
    M2, _ = O.spmm_fwd(n, r2, c2, v2, H, 3)
    assert not np.allclose(M2, H, rtol=1e-3)


@pytest.mark.parametrize("P", [2, 5])
def test_mean_partitioned_backward_is_the_transpose(P):
    """With raw (32-bit) messages the partitioned backward equals the dense
    A^T G up to fp32 rounding of the halo partials: the local entries of row
    u must carry A[v][u] = 1/d_v, not row u's own weight 1/d_u."""
    n, F = 64, 6
    src, dst = planted_partition_edges(n, 300, 4, 0.7, 3)
    rowptr, col, val = O.csr_build(n, src, dst, O.FLAGS_GCN | O.FLAG_MEAN)
    vt = O.transpose_values(n, rowptr, col, val)
    b = O.boundary_index(n, rowptr, col, val, P, vt)
    sb = np.full(b["n_slots"], 32, np.uint8)
    rng = np.random.default_rng(P)
    G = rng.standard_normal((n, F)).astype(np.float32)
    dH, T = O.spmm_bwd(n, rowptr, col, val, G, F, b, sb, seed=1)
    Dt = _dense_ahat(n, rowptr, col, val).T
    want = Dt @ G.astype(np.float64)
    assert np.all(np.abs(dH - want) <= 1e-6 * (np.abs(Dt) @ np.abs(G)) + 1e-9)
    dH0, _ = O.spmm_bwd(n, rowptr, col, val, G, F)
    assert np.allclose(dH0, want, atol=1e-12)
    b_wrong = O.boundary_index(n, rowptr, col, val, P)     # A^T weights missing
    dHw, _ = O.spmm_bwd(n, rowptr, col, val, G, F, b_wrong, sb, seed=1)
    assert not np.allclose(dHw, want, atol=1e-4)
