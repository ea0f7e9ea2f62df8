"""The error-free digit splitting behind the tensor-core block scores, checked
on the CPU with exact rational arithmetic (Ozaki, Ogita, Oishi and Rump,
Numer. Algorithms 2012: a product split into digit products that the
hardware sums without rounding).

Each row of double-float means v = hi + lo (fp32 pairs) is scaled by 2^-e
(max|hi| < 2^e) and written as seven 7-bit digits, each step taking
d = rint(128 x) and carrying the remainder as a TwoSum-normalised fp32 pair.
The claims the kernel rests on, checked here for random and adversarial rows:
  * |d_0| <= 128 and |d_s| <= 64 for s >= 1 (integers bf16 holds exactly);
  * the digits and the final remainder reproduce v 2^-e exactly, with the
    remainder below 2^-50 (1 + 2^-20);
  * every digit-level sum P_u = sum_{s+t=u} sum_c d_s d_t (u <= 6, d = 128
    channels) is an integer below 2^23, so fp32 accumulation is exact;
  * the score from levels u <= 6, summed in double-float, is within
    2^(eq+ek) d 1.3 2^-49 of the exact dot of the means.
This pins the method; tests/test_score_tc.py holds the kernel to the same
bound on the GPU."""
from fractions import Fraction

import numpy as np

F = np.float32
SLICES = 7


def _two_sum(a, b):
    s = F(a + b)
    bb = F(s - a)
    return s, F(F(a - F(s - bb)) + F(b - bb))


def _exponent(hi):
    m = float(np.max(np.abs(hi)))
    if m == 0.0:
        return 0
    _, e = np.frexp(m)          # m = f 2^e, 0.5 <= f < 1
    return min(int(e), 127)


def _digits(hi, lo):
    e = _exponent(hi)
    D = np.zeros((SLICES, hi.size), np.int64)
    rem = []
    for c in range(hi.size):
        x = F(hi[c] * F(2.0 ** -e))
        y = F(lo[c] * F(2.0 ** -e))
        for s in range(SLICES):
            z = F(x * F(128.0))
            dg = F(np.rint(z))
            x, y = _two_sum(F(z - dg), F(y * F(128.0)))
            D[s, c] = int(dg)
        rem.append(Fraction(float(x)) + Fraction(float(y)))
    return D, e, rem


def _score(Dq, eq, Dk, ek):
    P = [0] * SLICES
    for s in range(SLICES):
        for t in range(SLICES - s):
            P[s + t] += int(Dq[s] @ Dk[t])
    terms = [F(F(P[u]) * F(2.0 ** (-7 * (u + 2)))) for u in range(SLICES)]
    acc, cc = terms[-1], F(0.0)
    for u in range(SLICES - 2, -1, -1):
        acc, t = _two_sum(acc, terms[u])
        cc = F(cc + t)
    hi = F(acc + cc)
    lo = F(cc - F(hi - acc))
    scale = Fraction(2) ** (eq + ek)
    return (Fraction(float(hi)) + Fraction(float(lo))) * scale, P, terms


def _df(v):
    hi = v.astype(np.float32)
    lo = (v - hi.astype(np.float64)).astype(np.float32)
    return hi, lo


def _check_pair(vq, vk):
    d = vq.size
    qh, ql = _df(vq)
    kh, kl = _df(vk)
    Dq, eq, rq = _digits(qh, ql)
    Dk, ek, rk = _digits(kh, kl)
    for D, rem, h, l, e in ((Dq, rq, qh, ql, eq), (Dk, rk, kh, kl, ek)):
        assert np.abs(D[0]).max() <= 128 and np.abs(D[1:]).max() <= 64
        for c in range(d):
            rebuilt = sum(Fraction(int(D[s, c])) * Fraction(2) ** (-7 * (s + 1))
                          for s in range(SLICES)) + rem[c] * Fraction(2) ** (-7 * SLICES)
            assert rebuilt == (Fraction(float(h[c])) + Fraction(float(l[c]))) * Fraction(2) ** -e
            # remainder in units of 2^-49: |rem 2^-49| <= 2^-50 (1 + 2^-20)
            assert abs(rem[c]) <= Fraction(1, 2) * (1 + Fraction(1, 2 ** 20))
    got, P, terms = _score(Dq, eq, Dk, ek)
    assert max(abs(p) for p in P) < 2 ** 23
    for u in range(SLICES):  # each level's term is exact in fp32
        assert Fraction(float(terms[u])) == Fraction(P[u]) * Fraction(2) ** (-7 * (u + 2))
    exact = sum((Fraction(float(qh[c])) + Fraction(float(ql[c]))) *
                (Fraction(float(kh[c])) + Fraction(float(kl[c]))) for c in range(d))
    bound = Fraction(2) ** (eq + ek) * d * Fraction(13, 10) * Fraction(2) ** -49
    assert abs(got - exact) <= bound, float(abs(got - exact) / bound)
    return float(abs(got - exact) / bound)


def test_random_rows_of_many_magnitudes():
    rng = np.random.default_rng(5)
    worst = 0.0
    for _ in range(24):
        scale = 10.0 ** rng.uniform(-4, 4, size=2)
        spread = rng.uniform(size=(2, 128)) ** rng.integers(0, 8, size=(2, 1))
        v = rng.standard_normal((2, 128)) * scale[:, None] * spread
        worst = max(worst, _check_pair(v[0], v[1]))
    assert worst < 1.0


def test_adversarial_rows():
    # digits at their extremes: values just below the scale, alternating
    # signs, a row with one large and many tiny channels, and a zero row
    d = 128
    # the largest fp32 below 1 (minus a lo part): x -> 1, first digit 128
    near_one = np.full(d, 1.0 - 2.0 ** -24 - 2.0 ** -40) * np.where(np.arange(d) % 2, -1.0, 1.0)
    half_ulp = np.full(d, 0.5 + 2.0 ** -40)
    one_big = np.full(d, 1e-9)
    one_big[17] = 3.0e3
    _check_pair(near_one, near_one)
    _check_pair(near_one, half_ulp)
    _check_pair(one_big, near_one)
    _check_pair(one_big, one_big)
    _check_pair(np.zeros(d), near_one)
    Dq, _, _ = _digits(*_df(near_one))
    assert np.abs(Dq[0]).max() == 128
