"""Pins of the selection / capped-eviction oracle."""
import itertools
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle.select import STATUS_NAN_SCORE, ranking_key, select_topk_capped, top_k


def _cases():
    with open(os.path.join(GOLDEN, "select_toy.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    scores = np.array(case["scores"], dtype=np.float32)
    table, plan, status = select_topk_capped(scores, case["table_in"], case["K"], case["W"], case["C"])
    assert table == case["table_out"]
    assert [list(p) for p in plan] == case["plan"]
    assert status == case["status"]


def _brute_new_set(scores, resident, K, C):
    """Best admissible resident set by exhaustive search.

    Admissible: a subset of the residents and the top-K set T with at most C
    blocks that are not resident, of the largest size such sets reach (K, or
    fewer when residents plus admissible newcomers are fewer than K).  Best:
    its members' ranking keys, sorted, form the lexicographically smallest
    list.
    """
    nc = len(scores)
    T = sorted(range(nc), key=lambda b: ranking_key(scores, b))[:K]
    universe = sorted(set(resident) | set(T))
    size = min(K, len(resident) + min(C, len(set(T) - set(resident))))
    best = None
    for sub in itertools.combinations(universe, size):
        if len(set(sub) - set(resident)) > C:
            continue
        keyv = sorted(ranking_key(scores, b) for b in sub)
        if best is None or keyv < best[0]:
            best = (keyv, set(sub))
    return best[1]


def test_exhaustive_search_on_small_inputs():
    rng = np.random.default_rng(7)
    for _ in range(400):
        nc = int(rng.integers(1, 11))
        K = int(rng.integers(1, 5))
        C = int(rng.integers(0, K + 2))
        scores = rng.integers(0, 5, nc).astype(np.float32)      # many ties
        n_res = min(K, nc)
        res = [int(x) for x in rng.choice(nc, size=int(rng.integers(0, n_res + 1)), replace=False)]
        table_in = res + [-1] * (K - len(res))
        rng.shuffle(table_in)
        table, plan, status = select_topk_capped(scores, table_in, K, 0, C)
        assert status == 0
        new = {b for b in table if b >= 0}
        assert new == _brute_new_set(scores, res, K, C)
        # invariants
        R = set(res)
        T = set(top_k(scores, K))
        assert len(new - R) <= C
        assert (R & T) <= new
        assert len(plan) == len(new - R)
        assert len(new) == min(K, len(R) + len(plan))
        if len(T - R) <= C:
            assert T <= new
        for slot, (a, b) in enumerate(zip(table_in, table)):
            if a != b:
                assert (b, slot) in plan
        assert [p[1] for p in plan] == sorted(p[1] for p in plan)


def test_top_k_matches_full_sort():
    rng = np.random.default_rng(3)
    scores = rng.integers(-3, 3, 300).astype(np.float32)
    order = np.lexsort((np.arange(300), -scores))
    assert top_k(scores, 50) == order[:50].tolist()


def test_nan_score_is_flagged_and_ranked_last():
    scores = np.array([1.0, np.nan, 0.5], dtype=np.float32)
    assert top_k(scores, 3) == [0, 2, 1]
    _, _, status = select_topk_capped(scores, [-1, -1], 2, 0, 2)
    assert status == STATUS_NAN_SCORE
