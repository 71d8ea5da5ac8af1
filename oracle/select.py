"""Per-KV-head top-K selection with capped eviction, transfer plan and table.

What the pages fix:
  * [XR] §3 decode flow ("background, layer l"): predict the top-K blocks,
    compare them with the resident set, build a transfer plan, transfer
    asynchronously.
  * [XR] §3 component table: top-K = 128 blocks per head (2,048 tokens at
    16-token blocks); "Capped Eviction Policy" limits how many new blocks each
    head admits per step, fetch ratio 0.05 by default; "Head-wise Mapping" is a
    logical-to-logical table per KV head on top of the paged cache.
  * [XR] §4 innovations table: at most C new blocks per head per step; only the
    head-wise mapping entries change, the page table does not.
  * [LP] Key Takeaways and FAQ Q7: the cap bounds newly admitted blocks at the
    KV-selection stage so transfers stay within the link budget.
  * [XR] §3 decode flow, sparsification: a local window of recent blocks stays
    on the GPU.

Readings where the pages are silent (each listed in the design notes):
  * C = ceil(fetch_ratio * K) new blocks per head per step (the caller passes
    C as an integer).
  * Ranking key: higher fp32 score first, ties to the lower block id.  -0 and
    +0 compare equal.  A NaN score ranks below every number (and is flagged).
  * Admission: A = the first C blocks, in ranking order, of the top-K set T
    that are not resident.
  * Eviction: the new resident set is the first K, in ranking order, of the
    residents together with A; an empty slot (-1) counts as a resident below
    every block, so empty slots are filled before any block is evicted, lowest
    slot first.
  * Slot assignment: the admitted blocks in ascending block id take the freed
    slots in ascending slot order; every other slot keeps its block.  Plan
    entries are listed in ascending destination slot.
  * Window slots K .. K+W-1 pass through unchanged.  Candidates are blocks
    0 .. nc-1 with nc = ceil(L / 16) - W.
  * A resident entry outside [0, nc) or a block resident in two slots is an
    invalid table: the status word records it, the table passes through
    unchanged and the plan is empty (the table is not repaired).
  * No corrective fetch on a miss ([XR] §6 comparison with FreeKV).

Pins (tests/test_oracle_select.py): exhaustive search over every admissible
K-subset on small inputs (the greedy rule is optimal for this budget, a
partition matroid); T against a full sort; hand-worked tables and plans in
tests/golden/select_toy.json; the invariants |R'| = K, |R' \\ R| <= C,
R n T in R', count = |R' \\ R|, stable slots, R' = T when |T \\ R| <= C.
"""
import math

import numpy as np

# status bits of the device status word (the values are part of the C ABI)
STATUS_TABLE_RANGE = 1
STATUS_TABLE_DUP = 2
STATUS_NAN_SCORE = 4
STATUS_PLAN_RANGE = 8


def ranking_key(scores, b: int):
    """Sort key of block b: ascending key = better block."""
    x = float(scores[b])
    if math.isnan(x):
        return (1, 0.0, b)
    return (0, -x, b)


def top_k(scores, K: int) -> list:
    """The first min(K, nc) candidate blocks in ranking order."""
    nc = len(scores)
    return sorted(range(nc), key=lambda b: ranking_key(scores, b))[:K]


def select_topk_capped(scores, table_in, K: int, W: int, C: int):
    """One head's selection step.

    scores:   float32 [nc], the candidate blocks' scores.
    table_in: int [K + W], slot -> block id, -1 = empty.
    Returns (table_out list[int], plan list[(src_block, dst_slot)], status int).
    """
    scores = np.asarray(scores, dtype=np.float32)
    nc = len(scores)
    table_in = [int(x) for x in table_in]
    status = STATUS_NAN_SCORE if np.isnan(scores).any() else 0

    resident = {}                      # block -> slot
    empty_slots = []
    for slot in range(K):
        blk = table_in[slot]
        if blk == -1:
            empty_slots.append(slot)
        elif not 0 <= blk < nc:
            status |= STATUS_TABLE_RANGE
        elif blk in resident:
            status |= STATUS_TABLE_DUP
        else:
            resident[blk] = slot
    if status & (STATUS_TABLE_RANGE | STATUS_TABLE_DUP):
        return list(table_in), [], status

    key = lambda b: ranking_key(scores, b)   # noqa: E731
    T = top_k(scores, K)
    new = [b for b in T if b not in resident]
    A = new[:C]
    pool = sorted(list(resident) + A, key=key)
    kept = set(pool[:K])
    evicted = [b for b in resident if b not in kept]
    n_fill_empty = len(A) - len(evicted)
    freed = sorted([resident[b] for b in evicted] + empty_slots[:n_fill_empty])

    table_out = list(table_in)
    plan = []
    for blk, slot in zip(sorted(A), freed):
        table_out[slot] = blk
        plan.append((blk, slot))
    return table_out, plan, status
