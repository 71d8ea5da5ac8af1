"""Quest-style compressed key cache: per-block, per-dimension min and max.

What the pages fix:
  * [XR] §3 component table, row "Compressed Key Cache": every logical block
    stores a per-dimension min/max summary, and the summaries occupy 1/16 of
    the full KV cache.
  * [XR] §2 solution overview: the draft query scans a compressed key summary
    built by Quest-style min/max pooling.
  * [XR] §6 default parameters: block size 16 tokens.
  * [XR] §5: the implementation updates compressed keys during decode.

Readings where the pages are silent (each listed in the design notes):
  * Only keys are summarised, in the KV dtype (bf16): 2 values x D dims x 2 B
    per block against 2 x 16 x D x 2 B of K and V per block is exactly the
    stated 1/16; fp32 summaries (1/8) or value summaries would not be.
  * A partial last block (L not a multiple of 16) is summarised over its valid
    tokens only; a block with no valid token has no summary.
  * Signed zeros follow the IEEE 754-2019 minimum / maximum operations: -0 is
    below +0, so a block holding both has min -0 and max +0.  NaN and infinite
    keys are outside the contract.

Pins (tests/test_oracle_summary.py): a pure-Python brute force on small
blocks, the bound kmin <= k <= kmax, a one-token block giving kmin = kmax = k,
the signed-zero cases, partial blocks whose invalid tokens hold extreme values,
and the 1/16 byte ratio in closed form.
"""
import numpy as np

from . import bf16

BLOCK = 16


def _minimum(bits: np.ndarray) -> np.ndarray:
    """IEEE minimum over axis 0 of bf16 bit patterns [n][D] (n >= 1)."""
    vals = bf16.to_f64(bits)
    out = bits[np.argmin(vals, axis=0), np.arange(bits.shape[1])].copy()
    zero = vals.min(axis=0) == 0.0
    has_neg_zero = (bits == bf16.NEG_ZERO).any(axis=0)
    out[zero & has_neg_zero] = bf16.NEG_ZERO
    out[zero & ~has_neg_zero] = bf16.POS_ZERO
    return out


def _maximum(bits: np.ndarray) -> np.ndarray:
    """IEEE maximum over axis 0 of bf16 bit patterns [n][D] (n >= 1)."""
    vals = bf16.to_f64(bits)
    out = bits[np.argmax(vals, axis=0), np.arange(bits.shape[1])].copy()
    zero = vals.max(axis=0) == 0.0
    has_pos_zero = (bits == bf16.POS_ZERO).any(axis=0)
    out[zero & has_pos_zero] = bf16.POS_ZERO
    out[zero & ~has_pos_zero] = bf16.NEG_ZERO
    return out


def valid_blocks(L: int) -> int:
    """Number of blocks holding at least one of the L valid tokens."""
    return max(0, -(-L // BLOCK))


def block_summary(keys_bits, L: int, blocks=None):
    """Min/max key summary of one segment (one sequence, one KV head).

    keys_bits: uint16 [Nb][16][D], bf16 keys of the segment's blocks in order.
    L:         the sequence's valid token count; token t of block b is valid
               when 16 * b + t < L.
    blocks:    block ids to summarise (default: every block with a valid token).
    Returns (kmin, kmax, ids): uint16 [len(ids)][D] each, and the summarised
    block ids (blocks without a valid token are dropped from ``ids``).
    """
    keys_bits = np.asarray(keys_bits, dtype=np.uint16)
    nbv = min(valid_blocks(L), keys_bits.shape[0])
    ids = list(range(nbv)) if blocks is None else [b for b in blocks if 0 <= b < nbv]
    D = keys_bits.shape[2]
    kmin = np.zeros((len(ids), D), dtype=np.uint16)
    kmax = np.zeros((len(ids), D), dtype=np.uint16)
    for i, b in enumerate(ids):
        n_valid = min(BLOCK, L - BLOCK * b)
        tokens = keys_bits[b, :n_valid, :]
        kmin[i] = _minimum(tokens)
        kmax[i] = _maximum(tokens)
    return kmin, kmax, ids
