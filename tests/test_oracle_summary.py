"""Pins of the min/max summary oracle."""
import numpy as np
import pytest

from conftest import from_f32
from oracle import bf16
from oracle.summary import block_summary, valid_blocks


def _brute(keys_bits, L):
    """Pure-Python IEEE minimum / maximum with -0 < +0, token by token."""
    def lt(a, b):  # total order on non-NaN bf16 bit patterns
        fa, fb = float(bf16.to_f64(a)), float(bf16.to_f64(b))
        if fa != fb:
            return fa < fb
        return (a & 0x8000) and not (b & 0x8000)
    nb, _, D = keys_bits.shape
    mins, maxs = [], []
    for b in range(nb):
        n = min(16, L - 16 * b)
        if n <= 0:
            break
        lo = [int(keys_bits[b, 0, d]) for d in range(D)]
        hi = list(lo)
        for t in range(1, n):
            for d in range(D):
                x = int(keys_bits[b, t, d])
                if lt(x, lo[d]):
                    lo[d] = x
                if lt(hi[d], x):
                    hi[d] = x
        mins.append(lo)
        maxs.append(hi)
    return np.array(mins, dtype=np.uint16), np.array(maxs, dtype=np.uint16)


def _random_keys(rng, nb, D, zeros=False):
    vals = rng.standard_normal((nb, 16, D)).astype(np.float32)
    u = (vals.view(np.uint32) >> 16).astype(np.uint16)
    if zeros:
        m = rng.random((nb, 16, D))
        u[m < 0.2] = 0x0000
        u[(m >= 0.2) & (m < 0.4)] = 0x8000
    return u


@pytest.mark.parametrize("L", [16 * 5, 16 * 5 - 3, 1, 17, 33])
def test_matches_brute_force(rng, L):
    keys = _random_keys(rng, 5, 8, zeros=True)
    mn, mx, ids = block_summary(keys, L)
    bmn, bmx = _brute(keys, L)
    assert ids == list(range(valid_blocks(L)))
    assert np.array_equal(mn, bmn) and np.array_equal(mx, bmx)


def test_bounds_every_valid_key(rng):
    keys = _random_keys(rng, 7, 32)
    L = 7 * 16 - 5
    mn, mx, _ = block_summary(keys, L)
    k = bf16.to_f64(keys)
    for b in range(7):
        n = min(16, L - 16 * b)
        assert np.all(bf16.to_f64(mn[b]) <= k[b, :n].min(axis=0))
        assert np.all(bf16.to_f64(mn[b]) == k[b, :n].min(axis=0))
        assert np.all(bf16.to_f64(mx[b]) == k[b, :n].max(axis=0))


def test_one_token_block_is_the_key(rng):
    keys = _random_keys(rng, 3, 16, zeros=True)
    mn, mx, _ = block_summary(keys, 2 * 16 + 1)
    assert np.array_equal(mn[2], keys[2, 0]) and np.array_equal(mx[2], keys[2, 0])


def test_signed_zero_rule():
    D = 4
    keys = np.zeros((1, 16, D), dtype=np.uint16)
    keys[0, :, 0] = 0x0000                      # all +0
    keys[0, :, 1] = 0x8000                      # all -0
    keys[0, :, 2] = 0x0000
    keys[0, 5, 2] = 0x8000                      # +0 and -0 mixed
    keys[0, :, 3] = from_f32([1.0])[0]
    keys[0, 3, 3] = 0x8000                      # -0 and +1
    mn, mx, _ = block_summary(keys, 16)
    assert mn[0].tolist() == [0x0000, 0x8000, 0x8000, 0x8000]
    assert mx[0].tolist() == [0x0000, 0x8000, 0x0000, int(from_f32([1.0])[0])]


def test_invalid_tokens_are_ignored():
    D = 2
    keys = np.tile(from_f32([1.0, -1.0]), (2, 16, 1)).astype(np.uint16)
    keys[1, 3:, :] = from_f32([2.0**100, -2.0**100]).astype(np.uint16)   # beyond L
    mn, mx, ids = block_summary(keys, 16 + 3)
    assert ids == [0, 1]
    assert bf16.to_f64(mx[1]).tolist() == [1.0, -1.0]
    assert bf16.to_f64(mn[1]).tolist() == [1.0, -1.0]


def test_block_subset_and_empty_blocks(rng):
    keys = _random_keys(rng, 6, 8)
    full_mn, full_mx, _ = block_summary(keys, 40)      # 3 valid blocks
    mn, mx, ids = block_summary(keys, 40, blocks=[2, 4, 0])
    assert ids == [2, 0]                                # block 4 holds no valid token
    assert np.array_equal(mn, full_mn[[2, 0]]) and np.array_equal(mx, full_mx[[2, 0]])
    assert block_summary(keys, 0)[2] == []
