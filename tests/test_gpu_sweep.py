"""The fetch-ratio / top-K / admission-set study (sparse_kv_cache_quest_gb300.sweep)
against the same counts computed by the oracle: per decode step and segment,
the blocks the capped selection admits, whether the draft top-K held more
non-resident blocks than the cap, the overlap of the draft top-K with the next
step's true top-K, the next step's true top-K blocks resident after the step;
per sequence, the union over its KV heads of the first step's true top-K.  All
counts are integers and compared exactly, over several steps of a drifting
workload, at two fetch ratios."""
import numpy as np
import pytest
import torch

from conftest import bits
from oracle.score import score_blocks, segment_queries
from oracle.select import select_topk_capped, top_k
from oracle.summary import block_summary
import sparse_kv_cache_quest_gb300 as okv
from sparse_kv_cache_quest_gb300 import sweep
from synth import workload as wl

pytestmark = pytest.mark.gpu


def _oracle_counts(w):
    S, nc, K = w.S, w.nc, w.K
    T = w.steps
    qt = [bits(wl.q_true(w, 0, t)) for t in range(T)]
    qd = [bits(wl.drafts(w, 0, t)) for t in range(T)]
    out = {k: np.zeros((T, S), dtype=np.int64) for k in ("fetched", "binds", "overlap", "recall")}
    heads0 = [[] for _ in range(w.B)]
    for s in range(S):
        b, h = divmod(s, w.Hkv)
        keys = bits(wl.kv_tiles(w, 0, [s])[0])[:, 0]
        kmin, kmax, _ = block_summary(keys, w.L)
        kmin, kmax = kmin[:nc], kmax[:nc]
        true_sets = [set(top_k(score_blocks(kmin, kmax, qt[t][b, h * w.G:(h + 1) * w.G]), K)) for t in range(T)]
        heads0[b].append(true_sets[0])
        table = sorted(true_sets[0]) + [-1] * (K - len(true_sets[0])) + wl.window_blocks(w)
        for t in range(T):
            r_in = {x for x in table[:K] if x >= 0}
            sc = score_blocks(kmin, kmax, segment_queries(qd[t], b, h, w.G))
            t_draft = set(top_k(sc, K))
            table_out, plan, st = select_topk_capped(sc, table, K, w.W, w.cap)
            assert st == 0
            t_next = true_sets[(t + 1) % T]
            out["fetched"][t, s] = len(plan)
            out["binds"][t, s] = int(len(t_draft - r_in) > w.cap)
            out["overlap"][t, s] = len(t_draft & t_next)
            out["recall"][t, s] = len({x for x in table_out[:K] if x >= 0} & t_next)
            table = table_out
    out["admission"] = np.array([len(set().union(*hs)) for hs in heads0], dtype=np.int64)
    return out


@pytest.mark.parametrize("ratio", ["0.1", "0.03"])
def test_sweep_counts_equal_the_oracle(ratio):
    okv.load()
    base = wl.WORKLOADS[2].with_(B=2, L=16 * 256, plants=16)
    w = sweep.sweep_workload(ratio, 32, 4, base=base)
    got = sweep.run_counts(w, torch.device("cuda"))
    ref = _oracle_counts(w)
    for k in ("fetched", "binds", "overlap", "recall", "admission"):
        assert np.array_equal(got[k].numpy().astype(np.int64), ref[k]), k
    # the study's own claims on this input: the cap binds and admits `cap` blocks
    assert (ref["fetched"][1:] == w.cap).mean() > 0.5
    s = sweep.summarize(w, got)
    assert 0.0 < s["draft_true_topk_overlap"] <= 1.0 and 0.0 < s["admission_set_fraction"] <= 1.0
