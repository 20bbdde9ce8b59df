"""Pins of the oracle's consistency checksum: closed forms, exactness, and
that it sees a flipped bit and a swap (the point of the guard)."""
import numpy as np

import oracle

MOD = 1 << 64


def test_closed_forms():
    for U in [0, 1, 2, 7, 1000, 123_457]:
        ones = np.ones(U, np.uint16)
        assert oracle.checksum16(ones) == (U % MOD, (U * (U + 1) // 2) % MOD)
        top = np.full(U, 0xFFFF, np.uint16)
        assert oracle.checksum16(top) == ((U * 0xFFFF) % MOD, (0xFFFF * U * (U + 1) // 2) % MOD)


def test_exact_against_python_integers_and_wraps_mod_2_64():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 1 << 16, 5001).astype(np.uint16)
    s1 = sum(int(x) for x in u) % MOD
    s2 = sum((i + 1) * int(x) for i, x in enumerate(u)) % MOD
    assert oracle.checksum16(u) == (s1, s2)
    # fp32 buffers are read as their 16-bit halves, low half first
    f = rng.standard_normal(100).astype(np.float32)
    assert oracle.checksum16(f) == oracle.checksum16(f.view(np.uint16))
    assert oracle.checksum16(f.view(np.uint16)[::1].copy()) == oracle.checksum16(f)


def test_sees_a_flipped_bit_and_a_swap():
    rng = np.random.default_rng(2)
    u = rng.integers(0, 1 << 16, 4096).astype(np.uint16)
    base = oracle.checksum16(u)
    for i, bit in [(0, 0), (17, 15), (4095, 7)]:
        v = u.copy()
        v[i] ^= np.uint16(1 << bit)
        assert oracle.checksum16(v)[0] != base[0]
    v = u.copy()
    i, j = 10, 3000
    while v[i] == v[j]:
        j += 1
    v[[i, j]] = v[[j, i]]
    c = oracle.checksum16(v)
    assert c[0] == base[0] and c[1] != base[1]
