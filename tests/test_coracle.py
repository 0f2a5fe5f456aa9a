"""Pins for the oracle's C routines (oracle/coracle.c): the published
MurmurHash3 vectors, exact integer grids, the d-regular fixed point, thread
count invariance, and bit-for-bit agreement with oracle.py (itself pinned in
test_oracle_pins.py) on messy inputs -- every width, ragged F, constant rows,
signed zeros, split and long slots.  CPU only."""
import os

import numpy as np
import pytest

import oracle as O
from oracle import coracle as C
from synth import circulant_edges, planted_partition_edges, star_edges

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_fmix32_published_vectors():
    for key, seed, want in _golden("murmur3_x86_32.txt"):
        seed, want = int(seed, 16), int(want, 16)
        if key == "-":
            got = C.fmix32(seed)
        else:
            h = ((seed << 13) | (seed >> 19)) & 0xFFFFFFFF
            h = (h * 5 + 0xE6546B64) & 0xFFFFFFFF
            got = C.fmix32(h ^ 4)
        assert got == want


def test_hash32_matches_oracle():
    rng = np.random.default_rng(1)
    for seed, s, j in rng.integers(0, 2 ** 32, (200, 3)):
        assert C.hash32(int(seed), int(s), int(j)) == int(O.hash32(int(seed), int(s), int(j)))


def _messy_rows(rng, R, F):
    X = rng.standard_normal((R, F)).astype(np.float32) * rng.choice([1e-3, 1.0, 50.0], (R, 1)).astype(np.float32)
    X[0] = 3.25                      # constant row
    X[1] = 0.0
    X[1, ::2] = -0.0                 # signed zeros only
    if R > 2:
        X[2] = np.maximum(X[2], 0)   # ReLU row: min +0
    if R > 3:
        X[3] = -np.abs(X[3])         # max <= 0
    if R > 4:
        X[4, :] = np.float32(1e30)
        X[4, 0] = np.float32(-1e30)  # huge range
    if R > 5:
        X[5] = np.float32(1e-38) * (np.arange(F) % 3)  # subnormal range
    return X


@pytest.mark.parametrize("F", [1, 3, 5, 16, 31, 100, 129, 256, 300])
def test_quant_pack_matches_oracle(F):
    rng = np.random.default_rng(F)
    R = 64
    X = _messy_rows(rng, R, F)
    bits = rng.choice([1, 2, 4, 8, 32], R).astype(np.uint8)
    off = O.slot_offsets(bits, F)
    ld = (F + 3) // 4 * 4 + 4
    Xp = np.zeros((R, ld), np.float32)
    Xp[:, :F] = X
    got_p, got_m = C.quant_pack(Xp, F, None, bits, off, 77)
    want_p, want_m, _ = O.quant_pack(X, F, np.arange(R), bits, off, 77)
    assert np.array_equal(got_m.view(np.uint32), want_m.view(np.uint32))
    assert np.array_equal(got_p, want_p)
    # a row index permutation reads the same rows (row key = position r)
    perm = rng.permutation(R).astype(np.int32)
    got_p2, got_m2 = C.quant_pack(Xp, F, perm, bits, off, 77)
    want_p2, want_m2, _ = O.quant_pack(X, F, perm, bits, off, 77)
    assert np.array_equal(got_p2, want_p2) and np.array_equal(got_m2.view(np.uint32), want_m2.view(np.uint32))


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_quant_integer_grid_is_exact(b):
    """x = min + k*scale with exactly representable values: t = k, so the
    code is k except where fp32 rounding of k + u reaches k + 1 (u within
    half an ulp of 1); the codes unpack to k."""
    F = 96
    top = 2 ** b - 1
    rng = np.random.default_rng(b)
    k = rng.integers(0, top + 1, (32, F))
    k[:, 0], k[:, 1] = 0, top
    X = (np.float32(-2.0) + k.astype(np.float32) * np.float32(0.25)).astype(np.float32)
    bits = np.full(32, b, np.uint8)
    off = O.slot_offsets(bits, F)
    packed, meta = C.quant_pack(X, F, None, bits, off, 5)
    assert np.all(meta[:, 0] == -2.0) and np.all(meta[:, 1] == np.float32(top * 0.25) / np.float32(top))
    codes = O.unpack(packed, bits, F, off)
    u = O.sr_uniform(5, np.arange(32)[:, None], np.arange(F)[None, :])
    bump = (k.astype(np.float32) + u) >= (k + 1)
    assert np.array_equal(codes, np.minimum(k + bump, top))


def _graph(name):
    if name == "planted":
        n = 512
        s, d = planted_partition_edges(n, 3000, 4, 0.8, 9)
    elif name == "star":
        n = 300
        s, d = star_edges(n)
    else:
        n = 240
        s, d = circulant_edges(n, 6)
    return n, s, d


@pytest.mark.parametrize("name,P,F", [("planted", 4, 37), ("planted", 8, 256), ("star", 3, 64),
                                      ("circ", 5, 16)])
def test_halo_and_aggregations_match_oracle(name, P, F):
    n, s, d = _graph(name)
    rp, col, val = O.csr_build(n, s, d)
    b = O.boundary_index(n, rp, col, val, P)
    nb = O.node_bits(n, rp, b, [50], [2, 8], 1)
    sb = nb[b["slot_node"]].astype(np.uint8)
    sb[::7] = 32
    off = O.slot_offsets(sb, F)
    rng = np.random.default_rng(n + F)
    Hm = rng.standard_normal((n, F)).astype(np.float32)
    Gm = rng.standard_normal((n, F)).astype(np.float32)
    # forward messages and aggregation
    fp, fm = C.quant_pack(Hm, F, b["slot_node"], sb, off, 3)
    wp, wm, _ = O.quant_pack(Hm, F, b["slot_node"], sb, off, 3)
    assert np.array_equal(fp, wp) and np.array_equal(fm.view(np.uint32), wm.view(np.uint32))
    rows = np.arange(n)
    M, T = C.spmm_fwd_rows(rp, b, Hm, F, fp, fm, sb, off, rows)
    Mr, Tr = O.spmm_fwd(n, rp, col, val, Hm, F, b, sb, 3)
    assert np.all(np.abs(M - Mr) <= 1e-12 * Tr + 1e-300)
    assert np.allclose(T, Tr, rtol=1e-12, atol=0)
    # backward messages (fixed fp32 order: bit-exact) and aggregation
    hp, hm = C.halo_quant_pack(b, Gm, F, sb, off, 4)
    op, om, _ = O.halo_quant_pack(b, Gm, F, sb, off, 4)
    assert np.array_equal(hp, op) and np.array_equal(hm.view(np.uint32), om.view(np.uint32))
    dH, T2 = C.spmm_bwd_rows(rp, b, Gm, F, hp, hm, sb, off, rows)
    dr, T2r = O.spmm_bwd(n, rp, col, val, Gm, F, b, sb, 4)
    assert np.all(np.abs(dH - dr) <= 1e-12 * T2r + 1e-300)


def test_regular_graph_fixed_point():
    """On a d-regular graph every weight is 1/(d+1), so a constant feature
    row is reproduced; remote sources carry constant rows (scale 0), whose
    dequantised value is the constant itself: M = H exactly when d+1 is a
    power of two."""
    n, F, P = 256, 8, 4
    s, d = circulant_edges(n, 15)
    rp, col, val = O.csr_build(n, s, d)
    b = O.boundary_index(n, rp, col, val, P)
    sb = np.full(b["n_slots"], 2, np.uint8)
    off = O.slot_offsets(sb, F)
    H = np.repeat(np.linspace(-3, 3, n, dtype=np.float32)[:, None] * 0 + 1.5, F, 1).astype(np.float32)
    p, m = C.quant_pack(H, F, b["slot_node"], sb, off, 9)
    M, _ = C.spmm_fwd_rows(rp, b, H, F, p, m, sb, off, np.arange(n))
    assert np.array_equal(M, H.astype(np.float64))


def test_thread_count_does_not_change_results():
    n, s, d = _graph("planted")
    F, P = 64, 4
    rp, col, val = O.csr_build(n, s, d)
    b = O.boundary_index(n, rp, col, val, P)
    sb = np.full(b["n_slots"], 4, np.uint8)
    off = O.slot_offsets(sb, F)
    G = np.random.default_rng(0).standard_normal((n, F)).astype(np.float32)
    t0 = C.max_threads()
    try:
        C.set_threads(1)
        a = C.halo_quant_pack(b, G, F, sb, off, 1)
        C.set_threads(max(2, t0))
        z = C.halo_quant_pack(b, G, F, sb, off, 1)
    finally:
        C.set_threads(t0)
    assert np.array_equal(a[0], z[0]) and np.array_equal(a[1], z[1])


def test_quant_pack_in_pieces_equals_whole():
    """Rows processed in pieces with key0 = first row give the same buffer."""
    rng = np.random.default_rng(3)
    R, F = 100, 40
    X = rng.standard_normal((R, F)).astype(np.float32)
    bits = rng.choice([1, 2, 4, 8], R).astype(np.uint8)
    off = O.slot_offsets(bits, F)
    whole_p, whole_m = C.quant_pack(X, F, None, bits, off, 11)
    for a, b in [(0, 37), (37, 64), (64, 100)]:
        p, m = C.quant_pack(X[a:b], F, None, bits[a:b], off[a:b + 1] - off[a], 11, key0=a)
        assert np.array_equal(p, whole_p[off[a]:off[b]])
        assert np.array_equal(m, whole_m[a:b])


def test_halo_in_pieces_equals_whole():
    n, s, d = _graph("planted")
    F, P = 24, 4
    rp, col, val = O.csr_build(n, s, d)
    b = O.boundary_index(n, rp, col, val, P)
    sb = np.random.default_rng(5).choice([1, 2, 4, 8], b["n_slots"]).astype(np.uint8)
    off = O.slot_offsets(sb, F)
    G = np.random.default_rng(6).standard_normal((n, F)).astype(np.float32)
    wp, wm = C.halo_quant_pack(b, G, F, sb, off, 2)
    S = b["n_slots"]
    cut = [0, S // 3, S // 2, S]
    for a, z in zip(cut[:-1], cut[1:]):
        p, m = C.halo_quant_pack(b, G, F, sb, off, 2, a, z)
        assert np.array_equal(p, wp[off[a]:off[z]]) and np.array_equal(m, wm[a:z])
