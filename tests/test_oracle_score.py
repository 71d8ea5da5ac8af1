"""Pins of the block-scoring oracle."""
import json
import os

import numpy as np

from conftest import GOLDEN, from_f32
from oracle import bf16
from oracle.score import score_blocks, segment_queries
from oracle.summary import block_summary


def _toy():
    with open(os.path.join(GOLDEN, "score_toy.json")) as f:
        return json.load(f)


def test_hand_computed_toy():
    g = _toy()
    s = score_blocks(from_f32(g["kmin"]), from_f32(g["kmax"]), from_f32(g["queries"]))
    assert s.dtype == np.float32
    assert s.tolist() == g["expected_scores"]


def test_summation_order_is_ascending_d_in_fp32():
    c = _toy()["order_case"]
    k = from_f32([c["k"]])
    s = score_blocks(k, k, from_f32([c["query"]]))
    assert s.tolist() == [c["expected_score"]]


def _dot_fp32_seq(q, k):
    """fp32 dot product, terms added in ascending d from +0."""
    acc = np.float32(0.0)
    for d in range(len(q)):
        acc = np.float32(acc + np.float32(q[d]) * np.float32(k[d]))
    return acc


def _rand_bits(rng, shape, scale=1.0):
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def test_quest_bound_holds_for_every_key(rng):
    nb, D, nq = 6, 32, 5
    keys = _rand_bits(rng, (nb, 16, D))
    queries = _rand_bits(rng, (nq, D))
    L = nb * 16 - 7
    mn, mx, ids = block_summary(keys, L)
    s = score_blocks(mn, mx, queries)
    q = bf16.to_f32(queries)
    k = bf16.to_f32(keys)
    for b in ids:
        best = max(_dot_fp32_seq(q[j], k[b, t]) for j in range(nq) for t in range(min(16, L - 16 * b)))
        assert s[b] >= best


def test_one_token_block_score_equals_best_dot(rng):
    D, nq = 16, 4
    keys = _rand_bits(rng, (3, 16, D))
    queries = _rand_bits(rng, (nq, D))
    L = 2 * 16 + 1
    mn, mx, _ = block_summary(keys, L)
    s = score_blocks(mn[2:3], mx[2:3], queries)
    q, k = bf16.to_f32(queries), bf16.to_f32(keys[2, 0])
    assert s[0] == max(_dot_fp32_seq(q[j], k) for j in range(nq))


def test_group_and_draft_layout():
    B, Nd, Hkv, G, D = 2, 3, 2, 2, 4
    d = np.arange(B * Nd * Hkv * G * D, dtype=np.uint16).reshape(B, Nd, Hkv * G, D)
    q = segment_queries(d, 1, 1, G)
    assert q.shape == (Nd * G, D)
    assert np.array_equal(q[0], d[1, 0, 2]) and np.array_equal(q[1], d[1, 0, 3])
    assert np.array_equal(q[-1], d[1, Nd - 1, 3])
