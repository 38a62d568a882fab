"""Division by a launch-invariant divisor (Granlund and Montgomery, "Division
by invariant integers using multiplication", 1994), as used by the
rank-local kernels to split a flattened (row, vector) index: with
l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, the quotient of any
n < 2^31 is (umulhi(n, m) + n) >> l.  Checked here against exact integer
division for every divisor up to 4096 (each row width in 16-byte vectors of
a row up to 64 KB) and large odd divisors, on edge and random dividends.
The GPU parity tests of the rank-local kernels cover the device side."""
import random


def magic(d):
    l = 0
    while (1 << l) < d:
        l += 1
    m = ((1 << 32) * ((1 << l) - d)) // d + 1
    assert 0 < m < (1 << 32)
    return m, l


def div(n, m, l):
    t = (n * m) >> 32          # umulhi
    assert t + n < (1 << 32)   # no 32-bit overflow for n < 2^31
    return (t + n) >> l


def test_fast_div_matches_integer_division():
    rng = random.Random(5)
    divisors = list(range(1, 4097)) + [rng.randrange(4097, 1 << 31) for _ in range(300)] + [(1 << 31) - 1]
    top = (1 << 31) - 1
    for d in divisors:
        m, l = magic(d)
        ns = {0, 1, d - 1, d, d + 1, top, top - 1, (top // d) * d, (top // d) * d - 1}
        ns |= {k * d + r for k in (1, 2, 3, 1000) for r in (0, d - 1) if k * d + r <= top}
        ns |= {rng.randrange(0, top + 1) for _ in range(40)}
        for n in ns:
            if 0 <= n <= top:
                assert div(n, m, l) == n // d, (n, d)
