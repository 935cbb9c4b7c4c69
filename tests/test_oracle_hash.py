"""Pins for the oracle's hash (CPU only).

The noise family is the counter-based murmur3 fmix32 hash of "RandOpt
Speedrun", section "What was slow, and the fix". fmix32 is pinned to the
published MurmurHash3_x86_32 test vectors (tests/golden), its bijectivity to
an independently built inverse, and the counter folding to distinctness.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "murmur3_x86_32_vectors.txt")
M32 = 0xFFFFFFFF


def _rotl(x, r):
    return ((x << r) | (x >> (32 - r))) & M32


def _murmur3_x86_32(data: bytes, seed: int, fmix) -> int:
    """MurmurHash3_x86_32 body and tail, finalised with the oracle's fmix32."""
    c1, c2 = 0xCC9E2D51, 0x1B873593
    h = seed & M32
    nblocks = len(data) // 4
    for b in range(nblocks):
        k = int.from_bytes(data[4 * b:4 * b + 4], "little")
        k = (k * c1) & M32
        k = _rotl(k, 15)
        k = (k * c2) & M32
        h ^= k
        h = _rotl(h, 13)
        h = (h * 5 + 0xE6546B64) & M32
    tail = data[4 * nblocks:]
    k = 0
    if len(tail) >= 3:
        k ^= tail[2] << 16
    if len(tail) >= 2:
        k ^= tail[1] << 8
    if len(tail) >= 1:
        k ^= tail[0]
        k = (k * c1) & M32
        k = _rotl(k, 15)
        k = (k * c2) & M32
        h ^= k
    h ^= len(data)
    return fmix(h)


def _vectors():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, seed, want = line.split()
            data = b"" if key == "-" else bytes.fromhex(key)
            rows.append((data, int(seed, 16), int(want, 16)))
    return rows


@pytest.mark.parametrize("data,seed,want", _vectors())
def test_fmix32_murmur3_vectors(orc, data, seed, want):
    assert _murmur3_x86_32(data, seed, orc.fmix32) == want


def test_fmix32_zero_fixed_point(orc):
    assert orc.fmix32(0) == 0


def _inv_xorshift(y, s):
    x = y
    for _ in range(32 // s + 1):
        x = y ^ (x >> s)
    return x & M32


def test_fmix32_is_bijective_by_inverse(orc):
    """Each step of fmix32 is invertible (xor-shift, odd multiplier), so the
    whole map is a bijection on 32-bit words; check the inverse round-trips."""
    inv1 = pow(0x85EBCA6B, -1, 1 << 32)
    inv2 = pow(0xC2B2AE35, -1, 1 << 32)
    rng = np.random.default_rng(7)
    xs = list(rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).tolist())
    xs += [0, 1, 2, M32, 0x80000000, 0x7FFFFFFF]
    for x in xs:
        y = orc.fmix32(x)
        y = _inv_xorshift(y, 16)
        y = (y * inv2) & M32
        y = _inv_xorshift(y, 13)
        y = (y * inv1) & M32
        y = _inv_xorshift(y, 16)
        assert y == x


def test_words_distinct_over_token_channel(orc):
    """Within one (seed, draw, stream) the counter t*d_out + c is distinct for
    every (t, c), and fmix32 is a bijection, so the words are distinct."""
    w = orc.words(seed=123, draw_begin=5, n_draws=1, T=512, d_out=1000, stream=0)
    assert np.unique(w).size == w.size
    w1 = orc.words(seed=123, draw_begin=5, n_draws=1, T=512, d_out=1000, stream=1)
    assert np.unique(w1).size == w1.size
    assert np.mean(w == w1) < 1e-4


def test_keys_depend_on_both_seed_halves_and_stream(orc):
    ks = {orc.seed_key(s) for s in (0, 1, 1 << 32, (1 << 32) + 1, (1 << 63), M32)}
    assert len(ks) == 6
    dk = {orc.draw_key(9, i, s) for i in range(64) for s in (0, 1)}
    assert len(dk) == 128


def test_words_match_definition_composition(orc):
    """word(i,t,c,s) = fmix32(draw_key(i,s) ^ (t*d_out + c)) with draw_key =
    fmix32(seed_key ^ (2i+s)*0x9E3779B9) and seed_key folding both halves."""
    seed, d_out = 0x1234_5678_9ABC_DEF0, 37
    sk = orc.fmix32((seed & M32) ^ orc.fmix32(((seed >> 32) + 0x9E3779B9) & M32))
    assert sk == orc.seed_key(seed)
    w = orc.words(seed, 3, 2, 5, d_out, stream=1)
    for k in range(2):
        i = 3 + k
        dk = orc.fmix32(sk ^ (((2 * i + 1) * 0x9E3779B9) & M32))
        assert dk == orc.draw_key(seed, i, 1)
        for t in range(5):
            for c in range(d_out):
                assert w[k, t, c] == orc.fmix32(dk ^ ((t * d_out + c) & M32))
