"""Epoch controller (SYLVIE guide sections 8, 10, 11): the oracle pinned to
hand-worked sequences and closed forms, then the library's gnn_ldr_update
(host code, no GPU) compared with the oracle bit for bit."""
import math

import numpy as np
import pytest

from oracle.controller import LdrController, run


def _decisions(c):
    return [(h[3], h[4]) for h in c.history]


# ------------------------------------------------------------------ oracle pins
def test_mean_over_partitions_and_first_epoch():
    c = LdrController(lam=0.9, delta=3)
    assert c.report([1.0, 2.0, 6.0], 2.0) == (1, False)
    L, F, ldr, b, a = c.history[0]
    assert L == 3.0 and F == 3.0 and ldr == 0.0     # F_0 = L_0, LDR_0 = 0


def test_ema_closed_form():
    """F_t = lam^t L_0 + (1 - lam) sum_{k=1..t} lam^(t-k) L_k."""
    rng = np.random.default_rng(1)
    L = rng.uniform(0.5, 3.0, 40)
    lam = 0.9
    c = run([[x] for x in L], [1.0] * L.size, lam=lam, delta=5)
    for t in range(L.size):
        want = lam ** t * L[0] + (1 - lam) * sum(lam ** (t - k) * L[k] for k in range(1, t + 1))
        assert math.isclose(c.history[t][1], want, rel_tol=1e-12)


def test_ldr_is_descent_per_second():
    """A falling loss gives a positive rate; the same drop over a longer epoch
    a smaller one (lam = 0: F_t = L_t)."""
    c = run([[10.0], [8.0], [7.0]], [1.0, 2.0, 4.0], lam=0.0, delta=1)
    assert [h[2] for h in c.history] == [0.0, 1.0, 0.25]


def test_worked_sequence_delta_1():
    """lam = 0, delta = 1, et = 1: LDR = 0, 1, 2, 0.5, 0.1, 1.4, 0.01 (exact
    in binary up to the subtraction).  t = 1 is inside the look-back and keeps
    (1, sync); t = 2: 2 >= 1 halves (clipped at 1), async; t = 3: 0.5 < 2
    doubles, sync; t = 4: 0.1 < 0.5 doubles; t = 5: 1.4 >= 0.1 halves,
    async; t = 6: 0.01 < 1.4 doubles, sync."""
    L = [10.0, 9.0, 7.0, 6.5, 6.4, 5.0, 4.99]
    c = run([[x] for x in L], [1.0] * len(L), lam=0.0, delta=1)
    assert _decisions(c) == [(1, False), (1, False), (1, True), (2, False), (4, False),
                             (2, True), (4, False)]


def test_worked_sequence_delta_2_compares_two_back():
    """delta = 2: LDR_t is compared with LDR_{t-2}.  LDR = 0, 3, 1, 2, 0.5:
    t = 3 compares 2 with 3 (worse: double, sync); t = 4 compares 0.5 with 1
    (worse: double).  Comparing one epoch back instead would give t = 3:
    2 >= 1, halve."""
    L = [10.0, 7.0, 6.0, 4.0, 3.5]
    c = run([[x] for x in L], [1.0] * len(L), lam=0.0, delta=2)
    assert _decisions(c) == [(1, False), (1, False), (1, False), (2, False), (4, False)]


def test_bounds_saturate():
    # steadily slowing descent: 1 -> 2 -> 4 -> 8 and stays at b_max
    L = [100.0 - sum(1.0 / 2 ** k for k in range(t)) for t in range(12)]
    c = run([[x] for x in L], [1.0] * len(L), lam=0.0, delta=1)
    bits = [d[0] for d in _decisions(c)]
    assert bits[2:] == [2, 4, 8, 8, 8, 8, 8, 8, 8, 8]
    assert all(not d[1] for d in _decisions(c))
    # steadily accelerating descent: stays at b_min, async from t = delta + 1 on
    L = [100.0 - t * t for t in range(10)]
    c = run([[x] for x in L], [1.0] * len(L), lam=0.0, delta=1)
    assert [d[0] for d in _decisions(c)] == [1] * 10
    assert [d[1] for d in _decisions(c)] == [False, False] + [True] * 8


def test_width_range_and_other_limits():
    L = [100.0 - sum(1.0 / 2 ** k for k in range(t)) for t in range(10)]
    c = run([[x] for x in L], [1.0] * len(L), lam=0.0, delta=1, b_min=2, b_max=4)
    assert [d[0] for d in _decisions(c)] == [2, 2, 4, 4, 4, 4, 4, 4, 4, 4]


def test_nothing_changes_inside_the_look_back():
    rng = np.random.default_rng(3)
    c = run([[x] for x in rng.uniform(0, 5, 6)], [1.0] * 6, lam=0.9, delta=5)
    assert _decisions(c) == [(1, False)] * 6


def test_constant_loss_is_not_worse():
    """LDR = 0 every epoch: LDR_t >= LDR_{t-delta} always, so halving (at
    b_min) and asynchronous after the look-back."""
    c = run([[2.0, 2.0]] * 9, [1.0] * 9, lam=0.9, delta=3)
    assert _decisions(c) == [(1, False)] * 4 + [(1, True)] * 5


# ------------------------------------------------------------------ library against the oracle
def _lib():
    G = pytest.importorskip("sparse_aggregation_message_gb300")
    try:
        G.load()
    except Exception as e:  # pragma: no cover
        pytest.skip(f"library not built: {e}")
    return G


@pytest.mark.parametrize("lam,delta,b_min,b_max", [(0.9, 5, 1, 8), (0.9, 1, 1, 8), (0.0, 2, 1, 8),
                                                   (0.5, 10, 2, 8), (0.99, 20, 1, 4)])
def test_library_controller_matches_oracle(lam, delta, b_min, b_max):
    G = _lib()
    rng = np.random.default_rng(delta * 7 + b_min)
    T, N = 120, 4
    # a noisy, decaying loss with plateaus, and varying epoch times
    base = 3.0 * np.exp(-np.arange(T) / 30.0) + 0.2 * (np.arange(T) > 60)
    losses = base[:, None] + rng.normal(0, 0.05, (T, N))
    times = rng.uniform(0.5, 2.0, T)
    ref = LdrController(lam, delta, b_min, b_max)
    st = G.gnn_ldr_init(lam, delta, b_min, b_max)
    for t in range(T):
        want = ref.report(list(losses[t]), float(times[t]))
        got = G.gnn_ldr_update(st, list(losses[t]), float(times[t]))
        assert got == want, t
        assert st.F == ref.history[t][1], t                        # bitwise (==)
        assert st.ldr[t % (delta + 1)] == ref.history[t][2], t
        assert st.t == t + 1
    # the sequence exercised both directions
    assert len({h[3] for h in ref.history}) > 1
    assert {h[4] for h in ref.history} == {False, True}


def test_library_controller_rejects_bad_arguments():
    G = _lib()
    for args in [(1.0, 5, 1, 8), (-0.1, 5, 1, 8), (0.9, 0, 1, 8), (0.9, 65, 1, 8), (0.9, 5, 3, 8),
                 (0.9, 5, 8, 4)]:
        with pytest.raises(G.GnnError):
            G.gnn_ldr_init(*args)
    st = G.gnn_ldr_init()
    with pytest.raises(G.GnnError):
        G.gnn_ldr_update(st, [1.0], 0.0)
    with pytest.raises(G.GnnError):
        G.gnn_ldr_update(st, [], 1.0)
    assert st.t == 0
