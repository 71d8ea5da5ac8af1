"""Closed forms of the pages: KV footprint, HBM batch limit, link budget, and
the byte counts of the summary and the KV.

  eq. (1) [XR] §3 "core formulas": M_KV(B, L) = B * L * N_layer * 2 N_kv d_h * s
  eq. (2) [XR] §3: B_max = floor(M_HBM / (L * N_layer * 2 N_kv d_h * s))
  eq. (3) [XR] §3: C_token = B_link * T_decode (hideable transfer per step)
  1/16    [XR] §3 component table: summaries take 1/16 of the full KV cache.
Eq. (4) (the slowest background stage within T_step / N_layer) compares measured
stage times; it has no closed form to restate here.

Pins (tests/test_oracle_sizing.py): the worked example of [XR] §2 problem
definition (about 8.6 GB of KV per 32K-token request; at most 9 requests in
80 GB; tests/golden/sizing_worked_example.json); eq. (3) against the rows of
[XR] §6 Table 2 (tests/golden/fetch_cap_table2.json: the per-step fetch of each
fetch ratio from its link bandwidth and step time); and the 1/16 ratio.
"""

BLOCK = 16


def m_kv(B: int, L: int, n_layer: int, n_kv: int, d_h: int, s: int) -> int:
    """Eq. (1): bytes of K and V for B requests of L tokens."""
    return B * L * n_layer * 2 * n_kv * d_h * s


def b_max(m_hbm: int, L: int, n_layer: int, n_kv: int, d_h: int, s: int) -> int:
    """Eq. (2): requests of L tokens whose full KV fits in m_hbm bytes."""
    return m_hbm // (L * n_layer * 2 * n_kv * d_h * s)


def c_token(b_link: float, t_decode: float) -> float:
    """Eq. (3): bytes that one decode step of t_decode seconds can hide."""
    return b_link * t_decode


def summary_bytes(D: int, n_blocks: int, s: int = 2) -> int:
    """min and max, D dims each, per block, in the KV dtype (s bytes)."""
    return 2 * D * n_blocks * s


def full_kv_bytes(D: int, n_blocks: int, s: int = 2) -> int:
    """K and V of 16 tokens of D dims per block."""
    return 2 * BLOCK * D * n_blocks * s


def selected_kv_bytes(D: int, K: int, W: int, s: int = 2) -> int:
    """K and V of the K selected blocks plus the W window blocks."""
    return full_kv_bytes(D, K + W, s)
