"""The seeded input generator that the oracle and the GPU path share.

It holds none of the method's arithmetic, but every parity test depends on
it drawing what it says: SplitMix64 (Steele, Lea and Flood, 2014; the
finaliser constants of Vigna's public-domain reference code), a
counter-based stream per (seed, tensor id), Box-Muller normals and uniform
small integers.  Pinned here against the generator's published first
outputs, a pure-Python reimplementation of its stated definition, and the
distributions' moments.
"""
import math

import numpy as np
import pytest

import fc_inputs

MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def _mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def _draw(seed, tid, k):
    x0 = ((seed << 32) + (tid << 16)) & MASK
    return _mix((x0 + (k + 1) * GAMMA) & MASK)


def test_splitmix64_published_outputs():
    """The first outputs of SplitMix64 from state 0, as printed by the
    reference implementation."""
    got = [int(v) for v in fc_inputs.splitmix64(0, 4)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                   0xF88BB8A8724C81EC]


@pytest.mark.parametrize("x0", [1, 1234567, 2**63 + 5, MASK])
def test_splitmix64_matches_its_definition(x0):
    x, want = x0, []
    for _ in range(7):
        x = (x + GAMMA) & MASK
        want.append(_mix(x))
    assert [int(v) for v in fc_inputs.splitmix64(x0, 7)] == want


def _bf16_of(v):
    """float64 -> float32 (nearest) -> bf16 bits (nearest even), finite v."""
    f = np.float32(v)
    u = int(np.array([f], dtype=np.float32).view(np.uint32)[0])
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFFFFFF
    return u >> 16


@pytest.mark.parametrize("seed,tid,sigma", [(1002, 17, 1.0), (7, 2, 0.02), (0, 0, 3.5)])
def test_normal_elements_follow_the_stated_mapping(seed, tid, sigma):
    """Element n: u1 from draw 2n, u2 from draw 2n+1, one Box-Muller value
    in double, rounded to float32 and then to bf16.  Compared element by
    element where the double value is not within a rounding step of a
    float32 or bf16 tie (libm's log/cos may differ in the last bit)."""
    n = 64
    bits = fc_inputs.normal_bf16((n,), seed, tid, sigma=sigma)
    checked = 0
    for k in range(n):
        u1 = ((_draw(seed, tid, 2 * k) >> 11) + 0.5) * 2.0 ** -53
        u2 = (_draw(seed, tid, 2 * k + 1) >> 11) * 2.0 ** -53
        v = sigma * math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
        lo, hi = _bf16_of(v * (1 - 1e-12)), _bf16_of(v * (1 + 1e-12))
        if lo != hi:
            continue                       # too close to a rounding boundary
        assert int(bits[k]) == lo, k
        checked += 1
    assert checked >= n - 2


def test_sub_ranges_regenerate_the_same_elements():
    full = fc_inputs.normal_bf16((1000,), 5, 3)
    part = fc_inputs.normal_bf16((100,), 5, 3, start=450)
    assert np.array_equal(full[450:550], part)
    assert not np.array_equal(fc_inputs.normal_bf16((1000,), 5, 4), full)   # other tensor


def test_normal_moments():
    x = fc_inputs.bf16_bits_to_f32(fc_inputs.normal_bf16((1 << 20,), 11, 1, sigma=0.02))
    x = x.astype(np.float64)
    n = x.size
    assert abs(x.mean()) < 5 * 0.02 / math.sqrt(n)
    assert abs(x.std() / 0.02 - 1) < 0.005
    # Gaussian tail: about 4.55 % beyond two standard deviations
    assert abs(np.mean(np.abs(x) > 0.04) - 0.0455) < 0.002


@pytest.mark.parametrize("h", [1, 2, 7])
def test_small_integers_uniform_in_range(h):
    x = fc_inputs.bf16_bits_to_f32(fc_inputs.small_int_bf16((300000,), 9, 2, h=h))
    vals, counts = np.unique(x, return_counts=True)
    assert list(vals) == list(range(-h, h + 1))
    expect = x.size / (2 * h + 1)
    assert np.all(np.abs(counts - expect) < 6 * math.sqrt(expect))
    k = np.arange(16)
    want = [(_draw(9, 2, int(i)) % (2 * h + 1)) - h for i in k]
    assert list(x[:16].astype(int)) == want
