"""The integer identity the hash kernel uses for `h mod rows`: with
m = floor((2^64 - 1) / d), q = floor(h * m / 2^64) is floor(h / d) or one less,
so h - q*d lies in [0, 2d) and one conditional subtraction gives h mod d.
Checked here in exact Python integers on edge and random cases; the GPU tests
check the kernel's row ids against the oracle's plain `%` bit for bit."""
import random

M64 = (1 << 64) - 1


def mod_by_reciprocal(x, d):
    m = M64 // d
    q = (x * m) >> 64
    r = x - q * d
    assert 0 <= r < 2 * d
    return r - d if r >= d else r


def test_reciprocal_mod_equals_mod():
    rnd = random.Random(1)
    ds = [1, 2, 3, 7, 4096, 1_000_003, 5_040_000, 2**31 - 1, 2**31 - 19]
    ds += [rnd.randrange(1, 2**31) for _ in range(100)]
    xs = [0, 1, 2, M64, M64 - 1, 2**63, 2**63 - 1, 2**32, 2**32 - 1]
    xs += [rnd.getrandbits(64) for _ in range(500)]
    for d in ds:
        m = M64 // d
        for x in xs + [d - 1, d, d + 1, m * d, m * d - 1, M64 - M64 % d]:
            assert mod_by_reciprocal(x & M64, d) == (x & M64) % d
