"""The RoPE angle routine every kernel uses (sine and cosine of m * theta_i,
"Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践" §3), pinned to the mathematics on the host:
the 96-bit fractions theta_i / 2pi against a 200-bit evaluation, and cos / sin as float32 hi + lo
pairs against 200-bit cos / sin of the exact product m * theta_i (theta_i the float64 value)."""

import math
import random

import pytest

from rope_gqa_paged_gb300 import _build

mpmath = pytest.importorskip("mpmath")

RRA_OK, RRA_EINVAL = 0, -1
# Bound on |hi + lo - exact| of the float-float evaluation: its largest rounding terms (the
# float32 tails of the two series, ~2^-23 of terms below 5e-7) stay near 2^-45.
BOUND = 2.0 ** -44
CASES = [(128, 10000.0), (64, 500000.0), (128, 1.0e6), (512, 10000.0), (2, 10000.0)]
EXTREME = [(512, 1.0e9), (64, 1.0001)]  # theta_i down to ~1e-9 (tiny fractions); every theta_i near 1


@pytest.fixture(scope="module")
def rra():
    _build.build()
    from rope_gqa_paged_gb300 import rra as binding
    return binding


def _theta(D, base, i):
    return base ** (-2.0 * i / D)  # float64, as the host forms it


def _positions(seed):
    rnd = random.Random(seed)
    edge = [0, 1, 2, 3, 7, 8, 4095, 4096, 8191, 131071, 131072, 2 ** 20 + 3, 2 ** 30 - 1, 2 ** 31 - 1]
    return edge + [rnd.randrange(0, 2 ** 31) for _ in range(30)] + [rnd.randrange(0, 1 << 17) for _ in range(30)]


@pytest.mark.parametrize("D,base", CASES + EXTREME)
def test_phi_is_theta_over_two_pi(rra, D, base):
    mpmath.mp.prec = 200
    phi = rra.rra_rope_phi(D, base)
    assert len(phi) == D // 2
    for i, w in enumerate(phi):
        got = mpmath.mpf(w[0] + (w[1] << 32) + (w[2] << 64)) / mpmath.mpf(2) ** 96
        exact = mpmath.mpf(_theta(D, base, i)) / (2 * mpmath.pi)
        assert 0 <= exact - got < mpmath.mpf(2) ** -95, (D, base, i)  # truncated, not rounded


@pytest.mark.parametrize("D,base", CASES + EXTREME)
def test_cos_sin_within_bound(rra, D, base):
    mpmath.mp.prec = 200
    phi = rra.rra_rope_phi(D, base)
    worst = 0.0
    for pos in _positions(D):
        for i in range(0, D // 2, max(1, D // 40)):
            ang = mpmath.mpf(pos) * mpmath.mpf(_theta(D, base, i))
            ch, cl, sh, sl = rra.rra_rope_cos_sin_host(pos, phi[i])
            for hi, lo, ref in ((ch, cl, mpmath.cos(ang)), (sh, sl, mpmath.sin(ang))):
                assert abs(lo) <= abs(hi) * 2.0 ** -24 or (hi == 0.0 and lo == 0.0)  # normalised pair
                worst = max(worst, float(abs(mpmath.mpf(hi) + mpmath.mpf(lo) - ref)))
    assert worst < BOUND, math.log2(worst)


def test_special_angles(rra):
    """Position 0 is exactly (1, 0); a quarter turn lands on the axis in every quadrant."""
    phi = rra.rra_rope_phi(128, 10000.0)
    assert rra.rra_rope_cos_sin_host(0, phi[5]) == (1.0, 0.0, 0.0, 0.0)
    quarter = [0, 0, 1 << 30]  # phi = 1/4 turn
    for m, (c, s) in enumerate([(1, 0), (0, 1), (-1, 0), (0, -1)] * 2):
        ch, cl, sh, sl = rra.rra_rope_cos_sin_host(m, quarter)
        assert (ch + cl, sh + sl) == (c, s), m
    eighth = [0, 0, 1 << 29]  # 1/8 turn: both at sqrt(1/2), the remainder at its largest
    ch, cl, sh, sl = rra.rra_rope_cos_sin_host(1, eighth)
    assert abs((ch + cl) - math.sqrt(0.5)) < BOUND and abs((sh + sl) - math.sqrt(0.5)) < BOUND


def test_bad_arguments(rra):
    import ctypes
    lib = ctypes.CDLL(_build.LIB_PATH)
    buf = (ctypes.c_uint32 * 3 * 512)()
    lib.rra_rope_phi.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
    assert lib.rra_rope_phi(128, 10000.0, ctypes.cast(buf, ctypes.c_void_p)) == RRA_OK
    for D, base in ((127, 1e4), (0, 1e4), (1024, 1e4), (128, 0.0), (128, -1.0), (128, float("inf")),
                    (128, float("nan"))):
        assert lib.rra_rope_phi(D, base, ctypes.cast(buf, ctypes.c_void_p)) == RRA_EINVAL, (D, base)
    assert lib.rra_rope_phi(128, 1e4, None) == RRA_EINVAL
    out = (ctypes.c_float * 4)()
    lib.rra_rope_cos_sin_host.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.rra_rope_cos_sin_host(-1, ctypes.cast(buf, ctypes.c_void_p), ctypes.cast(out, ctypes.c_void_p)) == RRA_EINVAL
    assert lib.rra_rope_cos_sin_host(1, None, ctypes.cast(out, ctypes.c_void_p)) == RRA_EINVAL
