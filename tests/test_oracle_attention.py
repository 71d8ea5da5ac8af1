"""Pins of the sparse-attention oracle."""
import math

import numpy as np
import torch

from oracle import bf16
from oracle.attention import sparse_decode_attention


def _bits(rng, shape):
    v = rng.standard_normal(shape).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def test_all_blocks_resident_equals_dense_sdpa():
    rng = np.random.default_rng(11)
    G, D, nb = 4, 64, 6
    L = nb * 16 - 5
    q = _bits(rng, (G, D))
    tiles = _bits(rng, (nb, 2, 16, D))
    perm = rng.permutation(nb)
    pool = tiles[perm]
    scale = np.float32(1.0 / math.sqrt(D))
    out, lse = sparse_decode_attention(q, pool, perm.tolist(), L, scale)
    k = torch.from_numpy(bf16.to_f64(tiles[:, 0].reshape(-1, D)[:L]))
    v = torch.from_numpy(bf16.to_f64(tiles[:, 1].reshape(-1, D)[:L]))
    qt = torch.from_numpy(bf16.to_f64(q))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt[None, :, None, :], k[None, None].expand(1, G, L, D), v[None, None].expand(1, G, L, D),
        scale=float(scale))[0, :, 0, :].numpy()
    assert np.abs(out - ref).max() < 1e-12
    logits = float(scale) * (qt @ k.T).numpy()
    assert np.abs(lse - np.log(np.exp(logits).sum(axis=1))).max() < 1e-12


def test_slot_permutation_invariance_and_empty_slots():
    rng = np.random.default_rng(12)
    G, D = 2, 32
    tiles = _bits(rng, (5, 2, 16, D))
    q = _bits(rng, (G, D))
    table = [3, -1, 0, 4, -1]
    pool = np.stack([tiles[b] if b >= 0 else np.full_like(tiles[0], 0x7F80) for b in table])
    o1, l1 = sparse_decode_attention(q, pool, table, 5 * 16, 0.25)
    idx = [2, 0, 4, 1, 3]
    o2, l2 = sparse_decode_attention(q, pool[idx], [table[i] for i in idx], 5 * 16, 0.25)
    assert np.abs(o1 - o2).max() < 1e-13 and np.abs(l1 - l2).max() < 1e-13


def test_single_valid_token_gives_its_value():
    rng = np.random.default_rng(13)
    D = 16
    tiles = _bits(rng, (3, 2, 16, D))
    q = _bits(rng, (3, D))
    out, lse = sparse_decode_attention(q, tiles[[2]], [2], 2 * 16 + 1, 0.5)
    assert np.array_equal(out, np.tile(bf16.to_f64(tiles[2, 1, 0]), (3, 1)))
    assert np.allclose(lse, 0.5 * bf16.to_f64(q) @ bf16.to_f64(tiles[2, 0, 0]), rtol=0, atol=1e-12)


def test_equal_logits_give_the_mean():
    rng = np.random.default_rng(14)
    D = 16
    tiles = _bits(rng, (4, 2, 16, D))
    q = np.zeros((2, D), dtype=np.uint16)
    L = 4 * 16 - 9
    out, lse = sparse_decode_attention(q, tiles, [0, 1, 2, 3], L, 1.0)
    v = bf16.to_f64(tiles[:, 1].reshape(-1, D)[:L])
    assert np.abs(out - v.mean(axis=0)).max() < 1e-14
    assert np.allclose(lse, math.log(L))


def test_nothing_valid():
    out, lse = sparse_decode_attention(np.zeros((2, 8), np.uint16), np.zeros((2, 2, 16, 8), np.uint16), [-1, 5], 16 * 5, 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
