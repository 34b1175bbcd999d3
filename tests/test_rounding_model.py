"""The finalize's bf16 rounding method, modelled on the CPU.

The exact tier's finalize rounds an integer sum V (in units of 2^s) to bf16
without a 64-bit integer rounding routine: V is first rounded to 53
significant bits when wider (the float64 rounding of the literal algorithm)
and its zero low bits moved into s, then truncated to float32 with the lowest bit set when a set bit was dropped
(rounding to odd at 24 bits; the dropped bits, at most 29, are tested in the
low 32-bit word of |V|), scaled by 2^s in the exponent field and rounded
to nearest even at bf16's 8 bits.  Rounding to odd at p + 2 or more bits and
then to nearest at p bits equals one rounding to nearest at p bits (Boldo and
Melquiond, "Emulation of FMA and correctly rounded sums: proved algorithms
using rounding to odd", IEEE Trans. Computers 57(4), 2008).  This test models
those integer and bit steps in Python and compares them with the direct
definition, RN_bf16(RN_float64(V * 2^s)), computed on exact integers, on
random and midpoint-heavy V at every scale; the kernel itself is compared
with the oracle by the GPU tests.
"""
import random

M32 = (1 << 32) - 1


def rn_bits(mag, p):
    """mag rounded to p significant bits, nearest even: (m, shift)."""
    nb = mag.bit_length()
    if nb <= p:
        return mag, 0
    sh = nb - p
    m, rem, half = mag >> sh, mag & ((1 << sh) - 1), 1 << (sh - 1)
    if rem > half or (rem == half and m & 1):
        m += 1
    return m, sh


def direct(V, s):
    """bf16 bits of RN_bf16(RN_float64(V * 2^s)); None outside the normal range."""
    if V == 0:
        return 0
    m, sh = rn_bits(abs(V), 53)
    m8, sh8 = rn_bits(m << sh, 8)
    val = m8 << sh8
    nb = val.bit_length()
    E = nb - 1 + s
    if E < -126 or E > 127:
        return None
    frac = ((val >> (nb - 8)) if nb >= 8 else (val << (8 - nb))) & 0x7F
    return (0x8000 if V < 0 else 0) | ((E + 127) << 7) | frac


def f32_truncated_bits(V):
    """float32 bits of V truncated toward zero (cvt.rz.f32.s64)."""
    mag, nb = abs(V), abs(V).bit_length()
    m24 = mag >> (nb - 24) if nb > 24 else mag << (24 - nb)
    return (0x80000000 if V < 0 else 0) | ((nb - 1 + 127) << 23) | (m24 & 0x7FFFFF)


def bf16_nearest_even(fb):
    """bf16 bits of a finite float32 rounded to nearest even (cvt.rn.bf16.f32)."""
    return ((fb + 0x7FFF + ((fb >> 16) & 1)) >> 16) & 0xFFFF


def below_pow2(v, k):
    return -(1 << k) <= v < (1 << k)


def via_round_to_odd(V, s):
    """The kernel's steps; None where it takes the float64 route."""
    if not below_pow2(V, 53):                       # the float64 rounding, zero bits to s
        m, sh = rn_bits(abs(V), 53)
        V, s = m * (1 if V > 0 else -1), s + sh
    if V == 0:
        return 0
    fb = f32_truncated_bits(V)
    e = (fb >> 23) & 0xFF
    if not 1 <= e + s <= 254:
        return None
    drop = e - 150                                    # bits the truncation dropped (<= 29)
    lo = V & M32                                      # the low word of V; of |V|, minus it
    if drop > 0 and ((((-lo) & M32) if V < 0 else lo) & ((1 << drop) - 1)) != 0:
        fb |= 1
    fb = (fb + ((s << 23) & 0xFFFFFFFF)) & 0xFFFFFFFF
    h = bf16_nearest_even(fb)
    return None if (h & 0x7FFF) >= 0x7F80 else h


def cases(rng, n):
    for _ in range(n):
        nb = rng.randint(1, 63)
        V = rng.getrandbits(nb) | (1 << (nb - 1))
        r = rng.random()
        if r < 0.3 and nb > 9:
            V = (V >> (nb - 9)) << (nb - 9)                       # 9 bits: midpoint or exact
        elif r < 0.5 and nb > 54:
            V = ((V >> (nb - 54)) << (nb - 54)) | rng.choice([0, 1, 1 << rng.randint(0, nb - 55)])
        V = min(V, (1 << 63) - 1)
        yield (-V if rng.random() < 0.5 else V), rng.randint(-200, 140)
    for _ in range(n // 4):
        # wide sums whose float64 rounding leaves a bf16 midpoint, or one just
        # off it by a bit far below the kept 24 (past the low 32-bit word)
        nb = rng.randint(40, 63)
        top = (rng.getrandbits(7) | 0x80) << 1 | 1            # 8 bits and the midpoint bit
        V = top << (nb - 9)
        if rng.random() < 0.7:
            V |= 1 << rng.randint(max(0, nb - 53), nb - 10)    # a bit the float64 rounding may keep
        V = min(V, (1 << 63) - 1)
        yield (-V if rng.random() < 0.5 else V), rng.randint(-200, 140)
    for s in range(-200, 141, 7):
        for V in (1, 255, 256, 257, 0x180, 0x181, 0x1FF, (1 << 24) + 1, (1 << 53) - 1, 1 << 53,
                  (1 << 53) + 1, (1 << 62) + (1 << 9)):
            yield V, s
            yield -V, s


def test_round_to_odd_equals_one_rounding_to_nearest():
    rng = random.Random(2008)
    n = 0
    for V, s in cases(rng, 40000):
        want, got = direct(V, s), via_round_to_odd(V, s)
        # the kernel may leave an in-range result to the float64 route (a
        # rounding that carries into the smallest normal binade), never the
        # other way round, and never with other bits
        assert got == want or (got is None and want is not None), (V, s, want, got)
        n += got is not None
    assert n > 30000


def test_midpoints_round_to_even():
    # 1 + 2^-8 is the midpoint between bf16 1.0 and 1 + 2^-7: even wins
    assert via_round_to_odd((1 << 8) + 1, -8) == 0x3F80
    # 1 + 3 * 2^-8 lies between 1 + 2^-7 and 1 + 2^-6: even (1 + 2^-6) wins
    assert via_round_to_odd((1 << 8) + 3, -8) == 0x3F82
    # just above the midpoint: rounds up, the sticky bit decides it
    assert via_round_to_odd((1 << 40) + (1 << 32) + 1, -40) == 0x3F81
    # above 2^53 the float64 rounding comes first: 2^61 + 2^53 + 1 loses the 1
    # there and is then a bf16 midpoint rounding to even (down)
    assert via_round_to_odd((1 << 61) + (1 << 53) + 1, -61) == 0x3F80
    assert direct((1 << 61) + (1 << 53) + 1, -61) == 0x3F80
