"""The prefill kernel's item arithmetic divides by launch constants with one
multiplication (Granlund and Montgomery, "Division by Invariant Integers using
Multiplication", 1994): l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
n // d = (umulhi(m, n) + n) >> l for 0 <= n < 2^31.  This pins the formula the
kernel and its host set-up follow against exact integer division."""
import random


def _magic(d):
    l = (d - 1).bit_length()
    m = (1 << 32) * ((1 << l) - d) // d + 1
    return m, l


def _div(n, m, l):
    t = (m * n) >> 32
    return ((t + n) & 0xFFFFFFFF) >> l


def test_multiplier_fits_32_bits_and_add_never_wraps():
    rng = random.Random(3)
    for d in list(range(1, 4097)) + [rng.randrange(1, 1 << 31) for _ in range(500)] + [(1 << 31) - 1]:
        m, l = _magic(d)
        assert 0 < m < (1 << 32) and l <= 31
        for n in (0, 1, d - 1, d, (1 << 31) - 1):
            assert ((m * n) >> 32) + n < (1 << 32)


def test_exact_for_launch_sized_divisors():
    rng = random.Random(7)
    divisors = list(range(1, 600)) + [1024, 4096, 65535, 65536, 123457] + [rng.randrange(1, 1 << 31) for _ in range(200)]
    for d in divisors:
        m, l = _magic(d)
        ns = list(range(0, 2048)) + [k * d + r for k in (1, 3, 1000) for r in (0, d - 1) if k * d + r < (1 << 31)]
        ns += [rng.randrange(0, 1 << 31) for _ in range(200)] + [(1 << 31) - 1]
        for n in ns:
            assert _div(n, m, l) == n // d, (n, d)
