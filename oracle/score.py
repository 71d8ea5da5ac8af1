"""Look-ahead block scoring: draft queries against the min/max key summaries.

What the pages fix:
  * [XR] §2 solution overview and §3 decode flow ("background, layer l"): the
    draft queries scan the compressed key summaries to predict the top-K
    blocks of the next step; the true query is not part of this scan.
  * [XR] §4 Fig. 7: look-ahead attention = compressed key cache (min/max
    summaries) + selection of the sparse working set.
  * The score of a block for one query vector is the Quest upper bound
    sum_d max(q_d * min_d, q_d * max_d); a KV head's block score is the
    maximum of that bound over the head's GQA group and over the draft
    queries.

Readings where the pages are silent (each listed in the design notes):
  * Arithmetic and order: the summaries and queries are bf16; they are widened
    to fp32 (exact), and each query's sum runs over d = 0, 1, ..., D-1 in that
    order, starting from +0, with one fp32 round-to-nearest addition per term.
    A product of two bf16 values has at most 16 significant bits, so every
    term q_d * sel_d is exact in fp32 and "max(q*min, q*max)" equals
    "q * (max if q >= 0 else min)" bit for bit.
  * No 1/sqrt(D) factor: a positive scale does not change the ranking but can
    round distinct scores into ties.
  * Window blocks (the last W blocks) are always resident and not scored:
    only the nc = ceil(L / 16) - W candidate blocks are.

Pins (tests/test_oracle_score.py): hand-computed scores of a 2-query, 4-dim
toy (tests/golden/score_toy.json); a cancellation example whose fp32 result
differs under every other summation order; the Quest bound - the score is at
least the fp32 dot product of every query with every key of the block; and
equality with that dot product for one-token blocks.
"""
import numpy as np

from . import bf16


def score_blocks(kmin_bits, kmax_bits, queries_bits) -> np.ndarray:
    """Scores of a segment's candidate blocks.

    kmin_bits, kmax_bits: uint16 [n][D] summaries of the n candidate blocks.
    queries_bits:         uint16 [Nq][D], the Nd draft queries of each of the
                          G query heads that share this KV head.
    Returns float32 [n]: for every block, the max over the Nq queries of the
    ordered fp32 sum over d of q_d * (kmax_d if q_d >= 0 else kmin_d).
    """
    kmin = bf16.to_f32(kmin_bits)
    kmax = bf16.to_f32(kmax_bits)
    q = bf16.to_f32(queries_bits)
    n, D = kmin.shape
    best = np.full(n, -np.inf, dtype=np.float32)
    for j in range(q.shape[0]):
        acc = np.zeros(n, dtype=np.float32)
        for d in range(D):
            qd = q[j, d]
            sel = kmax[:, d] if qd >= 0 else kmin[:, d]
            acc = acc + qd * sel          # exact product, one fp32 rounding
        best = np.maximum(best, acc)
    return best


def segment_queries(drafts_bits, b: int, h: int, G: int) -> np.ndarray:
    """The Nd * G query vectors of KV head h of sequence b.

    drafts_bits: uint16 [B][Nd][Hq][D]; query heads h*G .. h*G + G - 1 share
    KV head h (grouped-query attention).  Returns uint16 [Nd * G][D].
    """
    d = np.asarray(drafts_bits, dtype=np.uint16)
    return d[b, :, h * G:(h + 1) * G, :].reshape(-1, d.shape[-1])
