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
                                               (2000, 1500, 3600), (9000, 3000, 12100)])
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
