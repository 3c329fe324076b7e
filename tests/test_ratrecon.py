"""The solve's host rational reconstruction (rg_rational_reconstruct), on the
CPU: planted fractions N/D must come back in lowest terms from
X = N D^-1 mod M whenever 2 |N| D < M, with moduli from one limb to
thousands of bits (the long-division paths of the big-integer code)."""
import math
import random

import pytest



@pytest.fixture(scope="module")
def lib():
    import exact_modular_int8_gb300 as rg  # the CPU path needs no GPU
    rg.library()
    return rg


def planted(rng, nbits, dbits, mbits):
    while True:
        m = rng.getrandbits(mbits) | (1 << (mbits - 1)) | 1
        d = rng.randrange(1, 1 << dbits)
        n = rng.randrange(-(1 << nbits) + 1, 1 << nbits)
        if math.gcd(d, m) == 1:
            g = math.gcd(abs(n), d)
            return n // g, d // g, m, (n * pow(d, -1, m)) % m


@pytest.mark.parametrize("nbits,dbits,mbits", [(3, 3, 10), (30, 30, 64), (60, 60, 130), (500, 400, 1000),
                                               (2000, 1500, 3600), (9000, 3000, 12100),
                                               (27200, 27100, 54400)])  # the n = 1024 solve's sizes
def test_planted_fractions(lib, nbits, dbits, mbits):
    rng = random.Random(nbits * 7 + dbits)
    for _ in range(6):
        n, d, m, x = planted(rng, nbits, dbits, mbits)
        assert lib.rational_reconstruct(x, m, nbits, dbits) == (n, d)


def test_integers_and_zero(lib):
    m = (1 << 200) + 235
    assert lib.rational_reconstruct(0, m, 50, 50) == (0, 1)
    assert lib.rational_reconstruct(12345, m, 50, 50) == (12345, 1)
    assert lib.rational_reconstruct(m - 12345, m, 50, 50) == (-12345, 1)


def test_no_fraction_within_the_bounds(lib):
    """A residue whose smallest fraction needs more bits than allowed."""
    m = (1 << 127) - 1
    rng = random.Random(5)
    n, d, m, x = planted(rng, 60, 60, 127)
    assert lib.rational_reconstruct(x, m, 10, 10) is None


def test_many_sizes_around_the_lehmer_boundary(lib):
    """Moduli from 65 to 5000 bits, bounds from 0 to half the modulus: the leading-digit
    batches and the single-step tail must together stop at the first small remainder."""
    rng = random.Random(11)
    for _ in range(300):
        mbits = rng.randrange(65, 5000)
        nbits = rng.randrange(0, mbits // 2)
        dbits = rng.randrange(0, mbits - nbits - 2)
        n, d, m, x = planted(rng, max(nbits, 1), max(dbits, 1), mbits)
        r = lib.rational_reconstruct(x, m, nbits, dbits)
        if abs(n) <= 2**nbits and d <= 2**dbits:
            assert r == (n, d)
        else:
            assert r is None or (abs(r[0]) <= 2**nbits and 0 < r[1] <= 2**dbits and (r[1] * x - r[0]) % m == 0)


@pytest.mark.parametrize("bits", [1, 63, 64, 65, 128, 129, 200, 1000, 5000, 15000, 30000])
def test_gcd_against_python(lib, bits):
    """The host gcd (Lehmer batches over two limbs, Euclid below) against math.gcd, with planted
    common factors of every size and operands of unequal length."""
    rng = random.Random(bits)
    for _ in range(8):
        g = rng.getrandbits(rng.randrange(1, bits + 1)) | 1
        a = g * rng.getrandbits(bits)
        b = g * rng.getrandbits(max(1, bits - rng.randrange(0, bits // 2 + 1)))
        assert lib.big_gcd(a, b) == math.gcd(a, b)
        assert lib.big_gcd(b, a) == math.gcd(a, b)


def test_gcd_special_cases(lib):
    fib = [0, 1]
    while fib[-1].bit_length() < 4000:  # consecutive Fibonacci numbers: every quotient is 1
        fib.append(fib[-1] + fib[-2])
    cases = [(0, 0), (0, 7), (7, 0), (1, 1), (2**4000, 2**1234), (2**4000 + 1, 2**4000 + 1),
             (fib[-1], fib[-2]), (fib[-1] * 3, fib[-2] * 3), (12345 * (2**3000 + 7), 2**3000 + 7),
             (2**3000 + 7, 5), (3**2000, 3**1500 * 2**100), ((1 << 5000) - 1, (1 << 3000) - 1)]
    for a, b in cases:
        assert lib.big_gcd(a, b) == math.gcd(a, b), (a.bit_length(), b.bit_length())


@pytest.mark.parametrize("mbits", [2, 63, 64, 65, 2000, 2048, 64 * 31 + 5, 64 * 33, 64 * 97, 64 * 300 + 17, 56000])
def test_mulmod_karatsuba_and_barrett(lib, mbits):
    """(a b) mod m by the Karatsuba product and Barrett's reduction the solve's numerators use, against
    Python integers: one to 880 limbs (the size at n = 1024), unbalanced factors, and operands at the
    edges (0, 1, m - 1, dense all-ones limbs)."""
    rng = random.Random(mbits)
    m = rng.getrandbits(mbits) | (1 << (mbits - 1)) | 1
    cases = [(0, 0), (1, m - 1), (m - 1, m - 1), ((1 << (mbits - 1)) - 1, m - 1)]
    cases += [(rng.randrange(m), rng.randrange(m)) for _ in range(4)]
    cases += [(rng.randrange(m), rng.randrange(min(m, 1 << 64 * 40))) for _ in range(2)]  # unbalanced
    for a, b in cases:
        assert lib.big_mulmod(a, b, m) == a * b % m
