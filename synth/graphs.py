"""Seeded graph, feature and weight generators.

Graphs come back as an undirected edge list with each unordered pair once
(``src[i] < dst[i]`` is not promised), no self-loops and no duplicates; the
library's CSR builder symmetrises, deduplicates and adds self-loops itself.

Workload shapes follow the five synthetic stand-ins for the datasets the
SYLVIE guide (section 12, "implementation, datasets, models") trains on:
a 4-community planted-partition toy graph, three degree-corrected stochastic
block models shaped like Yelp, Reddit and ogbn-products, and an R-MAT scale
test.  Nodes are numbered community by community, the layout the TorchGT
guide's community reordering produces, so that contiguous node blocks act as
partitions.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

BASE_SEED = 0x5EED0000

# Bit rules: a node of the boundary pool gets level k = #{i : 100*c > pct[i]*n}
# (c = its max-rank count by global degree within the pool, n = pool size) and
# mask bits ``bits[k]``; the per-epoch base width multiplies that, clipped at 8.
CONFIGS = {
    "tiny": dict(
        index=0, kind="planted", n=4096, n_undirected=16384, communities=4,
        intra=0.9, F=16, hidden=16, layers=2, P=4,
        rule=dict(pct=[90], bits=[2, 8]), base_bits=[1],
    ),
    "yelp": dict(
        index=1, kind="dcsbm", n=716847, n_undirected=6975000, communities=64,
        intra=0.9, gamma=2.2, max_deg=None, F=300, hidden=256, layers=3, P=8,
        rule=dict(pct=[80], bits=[4, 8]), base_bits=[1],
    ),
    "reddit": dict(
        index=2, kind="dcsbm", n=232965, n_undirected=57300000, communities=50,
        intra=0.9, gamma=2.2, max_deg=20000, F=602, hidden=128, layers=2, P=8,
        rule=dict(pct=[90], bits=[2, 8]), base_bits=[1],
    ),
    "products": dict(
        index=3, kind="dcsbm", n=2449029, n_undirected=30929570, communities=128,
        intra=0.9, gamma=2.2, max_deg=None, F=100, hidden=256, layers=4, P=8,
        rule=dict(pct=[25, 50, 75], bits=[1, 2, 4, 8]), base_bits=[1],
    ),
    "scale": dict(
        index=4, kind="rmat", scale=24, draws=128 << 20,
        abcd=(0.57, 0.19, 0.19, 0.05), communities=16, F=256, hidden=256,
        layers=3, P=16, rule=dict(pct=[95], bits=[1, 8]), base_bits=[1, 2, 4, 8],
    ),
    # the scale workload's generator at 1/16 of its size (same edge factor),
    # small enough for hardware-counter captures
    "rmat20": dict(
        index=5, kind="rmat", scale=20, draws=8 << 20,
        abcd=(0.57, 0.19, 0.19, 0.05), communities=16, F=256, hidden=256,
        layers=3, P=16, rule=dict(pct=[95], bits=[1, 8]), base_bits=[1, 2, 4, 8],
    ),
}


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng([int(k) & 0xFFFFFFFF for k in key])


def _keys(u: np.ndarray, v: np.ndarray, n: int) -> np.ndarray:
    lo = np.minimum(u, v).astype(np.int64)
    hi = np.maximum(u, v).astype(np.int64)
    return lo * n + hi


def _split_keys(keys: np.ndarray, n: int):
    return (keys // n).astype(np.int32), (keys % n).astype(np.int32)


def _sorted_distinct(a: np.ndarray) -> np.ndarray:
    a.sort()
    if a.size < 2:
        return a
    keep = np.empty(a.size, bool)
    keep[0] = True
    np.not_equal(a[1:], a[:-1], out=keep[1:])
    return a[keep]


def _draw_until(n: int, m_target: int, draw, rng) -> tuple[np.ndarray, np.ndarray]:
    """Call ``draw(rng, k) -> (u, v)`` until at least ``m_target`` distinct
    non-loop unordered pairs have been drawn, then keep a seeded uniform
    subset of exactly ``m_target`` of them."""
    have = np.empty(0, np.int64)
    factor = 1.08
    while have.size < m_target:
        k = int((m_target - have.size) * factor) + 1024
        u, v = draw(rng, k)
        keep = u != v
        have = _sorted_distinct(np.concatenate([have, _keys(u[keep], v[keep], n)]))
        factor = min(4.0, factor * 1.5)
    if have.size > m_target:
        pick = np.sort(rng.choice(have.size, m_target, replace=False))
        have = have[pick]
    return _split_keys(have, n)


def community_starts(n: int, c: int) -> np.ndarray:
    return (np.arange(c + 1, dtype=np.int64) * n) // c


def planted_partition_edges(n: int, m: int, communities: int, intra: float, seed: int):
    """Undirected planted-partition graph: endpoint u uniform; with probability
    ``intra`` the other endpoint is uniform inside u's community, otherwise
    uniform over the nodes of the other communities."""
    cs = community_starts(n, communities)
    comm_of = np.repeat(np.arange(communities), np.diff(cs))

    def draw(rng, k):
        u = rng.integers(0, n, k, dtype=np.int64)
        cu = comm_of[u]
        lo, hi = cs[cu], cs[cu + 1]
        inside = rng.random(k) < intra
        v_in = lo + (rng.random(k) * (hi - lo)).astype(np.int64)
        # outside: uniform over the n - size(cu) nodes not in cu
        r = (rng.random(k) * (n - (hi - lo))).astype(np.int64)
        v_out = np.where(r < lo, r, r + (hi - lo))
        v = np.where(inside, v_in, v_out)
        return u, v

    return _draw_until(n, m, draw, _rng(seed, 0))


def dcsbm_edges(n: int, m: int, communities: int, intra: float, gamma: float,
                max_deg: Optional[float], seed: int):
    """Degree-corrected SBM (Karrer and Newman, 2011): node weights theta drawn
    from a Pareto law with density ~ theta^-gamma, scaled so the expected
    degree is 2m/n and capped at ``max_deg``.  Each edge picks u with
    probability ~ theta; with probability ``intra`` v ~ theta inside u's
    community, else v ~ theta over the whole graph.  Draws are made as
    multinomial counts per node, expanded and shuffled, which has the same law
    as independent draws."""
    rng = _rng(seed, 0)
    theta = (1.0 - rng.random(n)) ** (-1.0 / (gamma - 1.0))
    mean_deg = 2.0 * m / n
    w = theta * (mean_deg / theta.mean())
    if max_deg is not None:
        for _ in range(8):
            w = np.minimum(w, max_deg)
            w *= mean_deg / w.mean()
        w = np.minimum(w, max_deg)
    p = w / w.sum()
    cs = community_starts(n, communities)
    comm_of = np.repeat(np.arange(communities), np.diff(cs))

    def pick(rng, k, lo, hi):
        # k i.i.d. draws from nodes lo..hi-1 with probability ~ w: multinomial
        # counts, expanded and shuffled (same law as k independent draws)
        q = p[lo:hi] / p[lo:hi].sum()
        cnt = rng.multinomial(k, q)
        out = np.repeat(np.arange(lo, hi, dtype=np.int64), cnt)
        rng.shuffle(out)
        return out

    def draw(rng, k):
        u = pick(rng, k, 0, n)
        inside = rng.random(k) < intra
        v = np.empty(k, np.int64)
        ins = np.nonzero(inside)[0]
        cu = comm_of[u[ins]]
        order = np.argsort(cu, kind="stable")
        ins = ins[order]
        m_c = np.bincount(cu, minlength=communities)
        off = 0
        for c in range(communities):
            mc = int(m_c[c])
            if mc:
                v[ins[off:off + mc]] = pick(rng, mc, int(cs[c]), int(cs[c + 1]))
            off += mc
        out = np.nonzero(~inside)[0]
        v[out] = pick(rng, out.size, 0, n)
        return u, v

    return _draw_until(n, m, draw, _rng(seed, 1))


def rmat_edges(scale: int, draws: int, abcd, seed: int, blocks: int = 16):
    """R-MAT (Chakrabarti, Zhan, Faloutsos 2004) with quadrant probabilities
    ``abcd`` quantised to 1/65536, ``draws`` edge draws over 2^scale nodes;
    symmetrised, self-loops dropped, deduplicated.  Node IDs are then randomly
    permuted and finally renumbered in breadth-first order from a seeded root
    (unreached nodes appended in ID order), the stand-in for a community order
    when no graph partitioner is present."""
    n = 1 << scale
    a, b, c, _ = abcd
    ta = np.uint16(round(a * 65536))
    tab = np.uint16(round((a + b) * 65536))
    tabc = np.uint16(round((a + b + c) * 65536))
    rng = _rng(seed, 0)
    chunk = 1 << 23
    keys = []
    done = 0
    while done < draws:
        k = min(chunk, draws - done)
        s = np.zeros(k, np.uint32)
        d = np.zeros(k, np.uint32)
        for _ in range(scale):
            # quadrant 0..3 = a, b, c, d: source bit q >> 1, destination bit q & 1
            r = np.frombuffer(rng.bytes(2 * k), dtype=np.uint16)
            q = (r >= ta).view(np.uint8) + (r >= tab).view(np.uint8) + (r >= tabc).view(np.uint8)
            s <<= 1
            d <<= 1
            s |= q >> 1
            d |= q & 1
        keep = s != d
        keys.append(_sorted_distinct(_keys(s[keep].astype(np.int64), d[keep].astype(np.int64), n)))
        done += k
    keys = _sorted_distinct(np.concatenate(keys))
    u, v = _split_keys(keys, n)
    perm = rng.permutation(n).astype(np.int32)
    u, v = perm[u], perm[v]
    # breadth-first renumbering
    import scipy.sparse as sp
    from scipy.sparse.csgraph import breadth_first_order

    g = sp.csr_matrix((np.ones(u.size, np.int8), (u, v)), shape=(n, n))
    root = int(rng.integers(0, n))
    order = breadth_first_order(g, root, directed=False, return_predecessors=False)
    seen = np.zeros(n, bool)
    seen[order] = True
    order = np.concatenate([order, np.nonzero(~seen)[0]]).astype(np.int64)
    new_id = np.empty(n, np.int32)
    new_id[order] = np.arange(n, dtype=np.int32)
    return new_id[u], new_id[v]


def circulant_edges(n: int, d: int):
    """d-regular circulant graph: i ~ i+k (mod n) for k = 1..d//2, plus the
    antipode i ~ i+n/2 when d is odd (n must then be even)."""
    us, vs = [], []
    i = np.arange(n, dtype=np.int64)
    for k in range(1, d // 2 + 1):
        us.append(i)
        vs.append((i + k) % n)
    if d % 2:
        assert n % 2 == 0
        h = i[: n // 2]
        us.append(h)
        vs.append(h + n // 2)
    u = np.concatenate(us)
    v = np.concatenate(vs)
    keys = _sorted_distinct(_keys(u, v, n))
    return _split_keys(keys, n)


def erdos_renyi_edges(n: int, p: float, seed: int):
    rng = _rng(seed, 7)
    iu, ju = np.triu_indices(n, 1)
    keep = rng.random(iu.size) < p
    return iu[keep].astype(np.int32), ju[keep].astype(np.int32)


def star_edges(n: int, hub: int = 0):
    others = np.array([i for i in range(n) if i != hub], np.int32)
    return np.full(others.size, hub, np.int32), others


def make_features(n: int, F: int, ld: int, seed: int, device: str = "cpu"):
    """fp32 N(0,1) rows of width F in an [n, ld] array, columns F..ld zero.
    ``device='cuda...'`` draws on the GPU with torch (same recipe, different
    stream of numbers); the result is then a torch tensor."""
    if device == "cpu":
        rng = _rng(seed, 1)
        out = np.zeros((n, ld), np.float32)
        step = 1 << 20
        for r0 in range(0, n, step):
            r1 = min(n, r0 + step)
            out[r0:r1, :F] = rng.standard_normal((r1 - r0, F), dtype=np.float32)
        return out
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    out = torch.zeros((n, ld), dtype=torch.float32, device=device)
    out[:, :F] = torch.randn((n, F), generator=g, device=device, dtype=torch.float32)
    return out


def make_weight_bf16(F_in: int, F_out: int, seed: int, layer: int) -> np.ndarray:
    """Glorot-uniform weights in [-sqrt(6/(F_in+F_out)), +...], returned as
    bf16 bit patterns (uint16, [F_in, F_out] row-major): the upper half of each
    fp32 draw, so every weight is a bf16 value inside the Glorot interval."""
    rng = _rng(seed, 2, layer)
    lim = np.sqrt(6.0 / (F_in + F_out))
    w = rng.uniform(-lim, lim, (F_in, F_out)).astype(np.float32)
    return (w.view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def ld_for(F: int) -> int:
    """Row stride (elements) for an fp32 feature matrix: F rounded up to 4."""
    return (F + 3) // 4 * 4


@dataclasses.dataclass
class Workload:
    name: str
    n: int
    src: np.ndarray
    dst: np.ndarray
    P: int
    dims: list  # [F_in of layer 1, hidden, ..., hidden]
    rule_pct: list
    rule_bits: list
    base_bits: list
    seed: int

    @property
    def layers(self) -> int:
        return len(self.dims) - 1


def make_workload(name: str) -> Workload:
    cfg = CONFIGS[name]
    seed = BASE_SEED + cfg["index"]
    kind = cfg["kind"]
    if kind == "planted":
        n = cfg["n"]
        src, dst = planted_partition_edges(n, cfg["n_undirected"], cfg["communities"],
                                           cfg["intra"], seed)
    elif kind == "dcsbm":
        n = cfg["n"]
        src, dst = dcsbm_edges(n, cfg["n_undirected"], cfg["communities"], cfg["intra"],
                               cfg["gamma"], cfg["max_deg"], seed)
    elif kind == "rmat":
        n = 1 << cfg["scale"]
        src, dst = rmat_edges(cfg["scale"], cfg["draws"], cfg["abcd"], seed)
    else:
        raise ValueError(kind)
    dims = [cfg["F"]] + [cfg["hidden"]] * cfg["layers"]
    return Workload(name=name, n=n, src=src, dst=dst, P=cfg["P"], dims=dims,
                    rule_pct=list(cfg["rule"]["pct"]), rule_bits=list(cfg["rule"]["bits"]),
                    base_bits=list(cfg["base_bits"]), seed=seed)
