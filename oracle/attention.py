"""Sparse paged decode attention over the head-wise logical-to-logical table.

What the pages fix:
  * [XR] §3 Fig. 5 and decode flow: the foreground forward pass runs sparse
    attention of the true query over the working set resident in HBM.
  * [LX] "The Insight" point 1: only the KV entries of the most relevant
    tokens are kept in HBM and attended to.
  * [XR] §3 component table, "Head-wise Mapping": each KV head has its own set
    of resident blocks, addressed through a logical-to-logical table.

Readings where the pages are silent (each listed in the design notes):
  * Standard scaled dot-product attention: logits = scale * q . k with
    scale = 1/sqrt(D) passed by the caller, softmax over every valid token of
    every non-empty slot, output = sum p * v.  Token t of the block in a slot
    is valid when 16 * block + t < L.
  * The G query heads of a KV head share its resident set (grouped-query
    attention).
  * Output in float64 here; the device writes fp32, and lse = log sum exp of
    the scaled logits.  No valid token gives out = 0 and lse = -inf.

Pins (tests/test_oracle_attention.py): when the table holds every block, the
result equals torch.nn.functional.scaled_dot_product_attention in float64;
permuting the slots changes nothing; one valid token gives out = v; equal
logits give the mean of v.
"""
import numpy as np

from . import bf16

BLOCK = 16


def sparse_decode_attention(q_bits, pool_bits, table, L: int, scale: float):
    """Attention of one KV head's G queries over its resident slots.

    q_bits:    uint16 [G][D], the true queries of the group.
    pool_bits: uint16 [slots][2][16][D], slot i holds the K tile then the V
               tile of block table[i].
    table:     int [slots], slot -> block id, negative = empty.
    Returns (out float64 [G][D], lse float64 [G]).
    """
    pool = np.asarray(pool_bits, dtype=np.uint16)
    q = bf16.to_f64(q_bits)
    keys, vals = [], []
    for i, blk in enumerate(table):
        blk = int(blk)
        if blk < 0:
            continue
        for t in range(BLOCK):
            if BLOCK * blk + t < L:
                keys.append(pool[i, 0, t])
                vals.append(pool[i, 1, t])
    G, D = q.shape
    if not keys:
        return np.zeros((G, D)), np.full(G, -np.inf)
    k = bf16.to_f64(np.stack(keys))            # [n][D]
    v = bf16.to_f64(np.stack(vals))            # [n][D]
    logits = float(scale) * (q @ k.T)          # [G][n]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ v) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse
