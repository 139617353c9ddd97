"""CPU checks of the two arguments the GPU quantizers rely on to avoid per-element
fp32 work, by brute force over fp16 inputs (numpy float16/float32 arithmetic is
IEEE round-to-nearest-even, like the kernels').

KIVI page "Makale Bulteni -- KIVI", section "Iddia ve Gerceklik", paragraphs 2-3
fixes the quantizer: per group, min and max, the scale s and codes by
round-to-nearest of (x - min) / s, clamped.  The 2-bit codes are the comparison form
[d > s/2] + [d >= 3s/2] + [d > 5s/2] of d = fl32(x - min) (pinned against the
literal rounding in test_oracle_quantizer.py); the 4-bit codes are
clamp(rint(fl32(d / s)), 0, 15).

1. fp16 thresholds (2-bit): each comparison term is [x > X] for the fp16 threshold
   X proven from the round-down estimate of fl32(min + t) and its neighbour.  Here,
   for many (min, s), every proven X is checked against the term itself on every
   finite fp16 x >= min.
2. Reciprocal product (4-bit): when q = fl32(d * fl32(1/s)) lies below 64 and more
   than 2^-15 from every half-integer, rint(q) equals rint(fl32(d / s)).
"""
import numpy as np

F16_ALL = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16).view(np.float16)
F16_FINITE = F16_ALL[np.isfinite(F16_ALL.astype(np.float32))]


def _rd16(y: np.float32) -> np.float16:
    """fp16 rounding of an fp32 value toward -inf."""
    with np.errstate(over="ignore"):
        h = np.float16(y)
    if not np.isfinite(np.float32(h)) or np.float32(h) > y:
        h = np.nextafter(h, np.float16(-np.inf))
        if not np.isfinite(np.float32(h)):  # y above the fp16 range: the largest finite
            h = np.float16(65504.0)
    return h


def _term(x32: np.ndarray, mn: np.float32, t: np.float32, strict: bool) -> np.ndarray:
    d = (x32 - mn).astype(np.float32)
    return d >= t if strict else d > t


def _threshold(mn: np.float32, t: np.float32, strict: bool):
    """The kernels' threshold: (X, proven)."""
    c = _rd16(np.float32(mn + t))
    at_c = bool(_term(np.array([np.float32(c)]), mn, t, strict)[0])
    nb = np.nextafter(c, np.float16(-np.inf)) if at_c else np.nextafter(c, np.float16(np.inf))
    with np.errstate(invalid="ignore"):
        at_n = bool(_term(np.array([np.float32(nb)]), mn, t, strict)[0])
    # the term is 0 at c and 1 above: X = c; 1 at c and 0 below: X = the fp16 below
    if not at_c and at_n:
        return c, True
    if at_c and not at_n:
        return nb, True
    return c, False


def _params(mn16: np.float16, mx16: np.float16):
    mn, mx = np.float32(mn16), np.float32(mx16)
    s = np.float32(np.float16(np.float32(np.float32(mx - mn) / np.float32(3))))
    return mn, s


def test_fp16_thresholds_equal_the_comparison_terms_on_every_fp16_input():
    rng = np.random.default_rng(7)
    pairs = []
    for _ in range(150):  # ordinary ranges
        e = rng.uniform(-14, 14)
        a = np.float16(rng.uniform(-1, 1) * 2.0 ** e)
        b = np.float16(float(a) + 2.0 ** rng.uniform(-20, 8))
        pairs.append((a, b))
    for _ in range(60):  # minima far below zero: thresholds next to zero
        a = np.float16(-rng.uniform(100, 30000))
        b = np.float16(min(65504.0, -float(a) * rng.choice([1.0, 5.0, 0.2]) + rng.uniform(0, 1)))
        pairs.append((a, b))
    pairs += [(np.float16(-65504.0), np.float16(65504.0)), (np.float16(0.0), np.float16(2.0 ** -24)),
              (np.float16(-0.0), np.float16(1.0)), (np.float16(-1.0), np.float16(2.0))]
    proven = unproven = 0
    for mn16, mx16 in pairs:
        if not float(mx16) > float(mn16):
            continue
        mn, s = _params(mn16, mx16)
        if s == 0:
            continue
        xs = F16_FINITE[F16_FINITE.astype(np.float32) >= mn].astype(np.float32)
        for f, strict in ((0.5, False), (1.5, True), (2.5, False)):
            t = np.float32(np.float32(f) * s)
            X, ok = _threshold(mn, t, strict)
            if not ok:
                unproven += 1
                continue
            proven += 1
            got = xs > np.float32(X)
            want = _term(xs, mn, t, strict)
            assert np.array_equal(got, want), (float(mn16), float(mx16), f, float(X))
    assert proven > 400
    # the minima far below zero do produce thresholds the estimate misses
    assert unproven >= 1


def test_reciprocal_product_rounds_like_the_division_outside_the_margin():
    rng = np.random.default_rng(11)
    n = 1_500_000
    # scales: any positive finite fp16, subnormals included
    s = rng.integers(1, 0x7C00, size=n).astype(np.uint16).view(np.float16).astype(np.float32)
    # quotients spread over [0, 20), a third of them within a few ulps of a half-integer
    Q = rng.uniform(0, 20, size=n)
    near = rng.random(n) < 0.35
    Q[near] = np.floor(Q[near]) + 0.5 + rng.integers(-40, 41, size=int(near.sum())) * 2.0 ** -21
    with np.errstate(over="ignore"):
        d = (Q * s.astype(np.float64)).astype(np.float32)
    keep = np.isfinite(d)
    d, s = d[keep], s[keep]
    rs = (np.float32(1.0) / s).astype(np.float32)
    q = (d * rs).astype(np.float32)
    div = (d / s).astype(np.float32)
    fast = (q < 64) & (np.abs(q - np.rint(q)) <= np.float32(0.5) - np.float32(2.0 ** -15))
    assert fast.sum() > 0.5 * d.size
    assert (~fast).sum() > 1000  # the margin is exercised
    assert np.array_equal(np.rint(q[fast]), np.rint(div[fast]))
    # near half-integers the product alone would be wrong somewhere: the margin matters
    assert not np.array_equal(np.rint(q), np.rint(div))
    # from 64 up the code clamps to 15 either way
    big = q >= 64
    assert np.all(np.rint(div[big]) >= 15)


def _code4x2_emulated(d: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The paired 4-bit coder's steps in numpy float32: q = fl(d * rs) (rs = fl(1/s),
    0 where s = 0), rint(q) as fl(fl(q + 1.5 * 2^23) - 1.5 * 2^23) and its integer from
    the sum's bit pattern, the division within 2^-15 of a half-integer, a clamp to 15."""
    M = np.float32(12582912.0)
    with np.errstate(divide="ignore"):
        rs = np.where(s == 0, np.float32(0), (np.float32(1.0) / s).astype(np.float32)).astype(np.float32)
    q = (d * rs).astype(np.float32)
    t = (q + M).astype(np.float32)
    r = (t - M).astype(np.float32)
    e = (q - r).astype(np.float32)
    c = t.view(np.int32) - np.array([M], np.float32).view(np.int32)[0]
    near = np.abs(e) > np.float32(0.5) - np.float32(2.0 ** -15)
    with np.errstate(divide="ignore", invalid="ignore"):
        div = np.rint((d / s).astype(np.float32))
    c = np.where(near, div, c)
    return np.minimum(c, 15)


def test_magic_constant_rounding_is_round_half_even():
    """fl(fl(q + 1.5 * 2^23) - 1.5 * 2^23) == rint(q) (half to even), and the sum's
    bit pattern minus the constant's is that integer, for every q the 4-bit
    quantizer can produce (0 <= q < 32): all float32 values near each half-integer
    and a million random ones."""
    M = np.float32(12582912.0)
    halves = np.arange(0, 32, dtype=np.float64) + 0.5
    near = np.concatenate([np.atleast_1d(np.nextafter(np.float32(h), np.float32(np.inf))) for h in halves] +
                          [np.atleast_1d(np.nextafter(np.float32(h), np.float32(-np.inf))) for h in halves] +
                          [np.float32(h) + np.arange(-600, 601, dtype=np.float32) * np.float32(2.0 ** -18) for h in halves])
    rng = np.random.default_rng(5)
    q = np.concatenate([near.astype(np.float32), halves.astype(np.float32), np.arange(32, dtype=np.float32),
                        rng.uniform(0, 32, 1_000_000).astype(np.float32)])
    q = q[(q >= 0) & (q < 32)]
    t = (q + M).astype(np.float32)
    r = (t - M).astype(np.float32)
    assert np.array_equal(r, np.rint(q))
    assert np.array_equal(t.view(np.int32) - np.array([M], np.float32).view(np.int32)[0], np.rint(q).astype(np.int32))
    assert np.array_equal((q - r).astype(np.float64), q.astype(np.float64) - r.astype(np.float64))  # exact


def test_paired_4bit_coder_equals_the_division():
    """The paired coder's codes equal clamp(rint(fl(d / s)), 0, 15) on the quotients of
    the reciprocal test (a third within a few ulps of a half-integer) and on s = 0."""
    rng = np.random.default_rng(12)
    n = 1_000_000
    s = rng.integers(1, 0x7C00, size=n).astype(np.uint16).view(np.float16).astype(np.float32)
    Q = rng.uniform(0, 20, size=n)
    near = rng.random(n) < 0.35
    Q[near] = np.floor(Q[near]) + 0.5 + rng.integers(-40, 41, size=int(near.sum())) * 2.0 ** -21
    with np.errstate(over="ignore"):
        d = (Q * s.astype(np.float64)).astype(np.float32)
    keep = np.isfinite(d) & (d >= 0)
    d, s = d[keep], s[keep]
    ref = np.clip(np.rint((d / s).astype(np.float32)), 0, 15)
    assert np.array_equal(_code4x2_emulated(d, s), ref)
    z = np.zeros(1000, np.float32)
    assert np.array_equal(_code4x2_emulated(rng.uniform(0, 5, 1000).astype(np.float32) * 0, z), np.zeros(1000))
