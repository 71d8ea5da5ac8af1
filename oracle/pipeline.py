"""One decode step of one layer for one segment, chaining the oracle steps.

Order, from [XR] §3 decode flow and Fig. 8 (asynchronous prefetch pipeline):
the foreground attends the true query over the blocks resident now; the
background scans the summaries with the draft queries, selects the next
resident set under the cap and transfers the admitted blocks for the next
step.  A summary update of the newest block ([XR] §5, compressed-key update)
runs first.
"""
import numpy as np

from .attention import sparse_decode_attention
from .score import score_blocks
from .select import select_topk_capped
from .stage import stage_blocks
from .summary import block_summary

BLOCK = 16


def run_segment(tiles, L, queries_draft, q_true, table_in, K, W, C, scale,
                kmin=None, kmax=None, update_blocks=None):
    """One step for one segment.

    tiles:         uint16 [Nb][2][16][D], the segment's full KV cache (host tier).
    queries_draft: uint16 [Nd*G][D];  q_true: uint16 [G][D].
    table_in:      int [K+W], the resident set before the step.
    kmin, kmax:    uint16 [Nb][D] summaries to update in place (built from the
                   keys when None); update_blocks: ids to rebuild (default: all).
    Returns a dict with kmin, kmax, scores, table_out, plan, status, out, lse,
    pool_before and pool_after.
    """
    tiles = np.asarray(tiles, dtype=np.uint16)
    Nb, _, _, D = tiles.shape
    nbv = min(-(-L // BLOCK), Nb)
    if kmin is None:
        kmin = np.zeros((Nb, D), dtype=np.uint16)
        kmax = np.zeros((Nb, D), dtype=np.uint16)
        update_blocks = None
    mn, mx, ids = block_summary(tiles[:, 0], L, update_blocks)
    for i, b in enumerate(ids):
        kmin[b], kmax[b] = mn[i], mx[i]
    nc = nbv - W
    scores = score_blocks(kmin[:max(nc, 0)], kmax[:max(nc, 0)], queries_draft)
    table_out, plan, status = select_topk_capped(scores, table_in, K, W, C)
    pool = np.stack([tiles[b] if b >= 0 else np.zeros_like(tiles[0]) for b in table_in])
    out, lse = sparse_decode_attention(q_true, pool, table_in, L, scale)
    pool_after, st2 = stage_blocks(tiles, plan, pool)
    return dict(kmin=kmin, kmax=kmax, scores=scores, table_out=table_out, plan=plan,
                status=status | st2, out=out, lse=lse, pool_before=pool, pool_after=pool_after)
