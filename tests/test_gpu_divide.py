"""The quantiser's division (x - min) / scale, tested directly through
gnn_quant_divide against IEEE fp32 division: bit-exact wherever the codes
can depend on its last bits (quotients from 2^-26 up), below 2^-25 under
that, on random operands over the whole exponent range, on every step of the
quantiser's own range for a set of scales, and on quotients constructed to lie
within about 2^-25 ulp of a rounding midpoint (the cases a division that is
not correctly rounded gets wrong), whose exact rounding is computed with
integers."""
from fractions import Fraction

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

G = pytest.importorskip("sparse_aggregation_message_gb300")

LO, HI = 2.0 ** -76, 2.0 ** 100


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    G.load()
    return t


def _run(torch, a, b):
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    ad, bd = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    q = torch.empty_like(ad)
    G.gnn_quant_divide(ad, bd, q)
    G.gnn_sync_check()
    return q.cpu().numpy()


def _check(a, b, got):
    with np.errstate(all="ignore"):
        ref = (a / b).astype(np.float32)
    inside = (b >= LO) & (b <= HI)
    big = inside & (np.abs(ref) >= 2.0 ** -26) & (np.abs(ref) <= 2.0 ** 100)
    small = inside & (np.abs(ref) < 2.0 ** -26)
    outside = ~inside
    assert np.array_equal(got[big].view(np.uint32), ref[big].view(np.uint32)), \
        f"{int(np.sum(got[big].view(np.uint32) != ref[big].view(np.uint32)))} quotients differ"
    assert np.all(np.abs(got[small]) < 2.0 ** -25)
    eq = (got[outside].view(np.uint32) == ref[outside].view(np.uint32)) | \
        (np.isnan(got[outside]) & np.isnan(ref[outside]))
    assert np.all(eq)
    return int(big.sum())


def _floats(rng, n, e_lo, e_hi):
    m = rng.integers(1 << 23, 1 << 24, n).astype(np.float64)
    e = rng.integers(e_lo, e_hi + 1, n)
    return (m * np.exp2(e - 23)).astype(np.float32)


def test_random_operands(torch):
    rng = np.random.default_rng(5)
    n = 1 << 24
    a = _floats(rng, n, -140, 60)
    a[::97] = 0.0
    a[1::101] *= -1
    b = _floats(rng, n, -100, 120)
    assert _check(a, b, _run(torch, a, b)) > n // 8


def test_quantiser_range(torch):
    """a on a dense grid of [0, range] for scales of many magnitudes; the
    quotient runs over [0, 2^bits - 1] as in the quantiser."""
    rng = np.random.default_rng(6)
    a_all, b_all = [], []
    for top in (1.0, 3.0, 15.0, 255.0):
        for e in (-70, -30, -8, -1, 0, 3, 20, 90):
            scale = np.float32(rng.uniform(1, 2) * 2.0 ** e)
            rng_ = np.float32(scale * np.float32(top))
            k = np.arange(1 << 18, dtype=np.float64)
            a = (k / k[-1] * np.float64(rng_)).astype(np.float32)
            a_all.append(a)
            b_all.append(np.full(a.size, scale, np.float32))
    a, b = np.concatenate(a_all), np.concatenate(b_all)
    _check(a, b, _run(torch, a, b))


def _rn32(x: Fraction) -> float:
    """Round a positive rational to the nearest fp32 (ties to even), exactly."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    k = x / ulp
    f = k.numerator // k.denominator
    rem = k - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return float(f * ulp)


def test_near_midpoint_quotients(torch):
    """For significands B, the A whose quotient A/B lies nearest an fp32
    rounding midpoint: |A 2^24 mod 2B - B| smallest (quotient in [1, 2)) and
    |A 2^25 mod 2B - B| smallest (quotient in [1/2, 1)); then scaled by powers
    of two into the quantiser's range and beyond."""
    rng = np.random.default_rng(7)
    Bs = [0xFFFFFF, 0x800000, 0x800001, 0xAAAAAB, 0xC00001, 0xFFFFFD] + \
        [int(x) for x in rng.integers(1 << 23, 1 << 24, 10)]
    pairs = []
    for B in Bs:
        A = np.arange(1 << 23, 1 << 24, dtype=np.int64)
        for shift, sel in ((24, A >= B), (25, A < B)):
            As = A[sel]
            d = np.abs(((As << shift) % (2 * B)) - B)
            best = As[np.argsort(d, kind="stable")[:48]]
            pairs += [(int(x), B) for x in best]
    a, b, want = [], [], []
    for A, B in pairs:
        for ea, eb in ((0, 0), (-3, -9), (7, 5), (-60, -70), (40, 39), (-20, 30)):
            av = A * 2.0 ** (ea - 23)
            bv = B * 2.0 ** (eb - 23)
            a.append(av)
            b.append(bv)
            want.append(_rn32(Fraction(A, B) * Fraction(2) ** (ea - eb)))
    a = np.array(a, np.float32)
    b = np.array(b, np.float32)
    want = np.array(want, np.float32)
    got = _run(torch, a, b)
    with np.errstate(all="ignore"):
        assert np.array_equal((a / b).astype(np.float32).view(np.uint32), want.view(np.uint32))
    keep = (np.abs(want) >= 2.0 ** -26) & (b >= LO) & (b <= HI)
    assert keep.sum() > 1000
    assert np.array_equal(got[keep].view(np.uint32), want[keep].view(np.uint32))
