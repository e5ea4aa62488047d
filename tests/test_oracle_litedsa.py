"""Pins for the LiteDSA packing oracle: a hand-derived case, brute force from
the definition on random small inputs, and the round-trip property."""
import numpy as np
import pytest

import oracle.litedsa as ld


def test_hand_example():
    # group of 2: query 0 picked {7, 3, 9}, query 1 picked {3, 12, -1}
    idx = np.array([[7, 3, 9], [3, 12, -1]])
    union, lens, masks = ld.pack(idx, 2)
    assert lens.tolist() == [4]
    assert union[0, :4].tolist() == [3, 7, 9, 12] and (union[0, 4:] == -1).all()
    assert masks.shape == (2, 1)
    assert masks[0, 0] == 0b0111            # 3, 7, 9
    assert masks[1, 0] == 0b1001            # 3, 12


def test_bruteforce_small():
    rng = np.random.default_rng(1)
    for _ in range(50):
        T = int(rng.integers(1, 7))
        k = int(rng.integers(1, 6))
        G = int(rng.integers(1, 4))
        idx = rng.integers(-1, 12, size=(T, k))
        # selections hold distinct keys (a top-k never repeats a key)
        for t in range(T):
            seen = set()
            for c in range(k):
                if idx[t, c] in seen:
                    idx[t, c] = -1
                seen.add(int(idx[t, c]))
        union, lens, masks = ld.pack(idx, G)
        for g in range((T + G - 1) // G):
            members = [int(i) for t in range(g * G, min(T, g * G + G)) for i in idx[t] if i >= 0]
            expect = sorted(set(members))
            assert union[g, : lens[g]].tolist() == expect
            for t in range(g * G, min(T, g * G + G)):
                for j, key in enumerate(expect):
                    bit = (int(masks[t, j // 32]) >> (j % 32)) & 1
                    assert bit == (key in set(int(i) for i in idx[t] if i >= 0))


def test_round_trip_and_sharing():
    rng = np.random.default_rng(2)
    T, k, G = 24, 50, 8
    base = rng.choice(400, size=200, replace=False)
    idx = np.stack([rng.choice(base, size=k, replace=False) for _ in range(T)])
    union, lens, masks = ld.pack(idx, G)
    for t in range(T):
        g = t // G
        np.testing.assert_array_equal(ld.unpack_row(union[g], lens[g], masks[t]), np.sort(idx[t]))
    assert lens.sum() < T * k       # overlapping selections share list entries
