"""Pins of the closed forms: eqs. (1)/(2) against the page's worked example,
eq. (3) against the rows of the fetch-cap ablation (Table 2)."""
import json
import os

from conftest import GOLDEN
from oracle import sizing


def _load():
    with open(os.path.join(GOLDEN, "sizing_worked_example.json")) as f:
        return json.load(f)


def test_eq1_worked_example_per_request():
    g = _load()
    a = g["assumed_shape"]
    m = sizing.m_kv(1, g["L"], a["n_layer"], a["n_kv"], a["d_h"], a["s"])
    assert m == 8_589_934_592
    assert round(m / 1e9, 1) == g["kv_gb_per_request_printed"]


def test_eq2_worked_example_batch_limit():
    g = _load()
    a = g["assumed_shape"]
    assert sizing.b_max(g["m_hbm_bytes"], g["L"], a["n_layer"], a["n_kv"], a["d_h"], a["s"]) == g["b_max_printed"]
    # the example uses decimal gigabytes: 80 GiB would admit 10
    assert sizing.b_max(80 * 2**30, g["L"], a["n_layer"], a["n_kv"], a["d_h"], a["s"]) == 10


def test_eq1_is_linear_and_eq2_is_its_floor_inverse():
    for B in (1, 3, 17):
        assert sizing.m_kv(B, 4096, 36, 8, 128, 2) == B * sizing.m_kv(1, 4096, 36, 8, 128, 2)
    per = sizing.m_kv(1, 4096, 36, 8, 128, 2)
    for budget in (per - 1, per, 5 * per + per // 2):
        n = sizing.b_max(budget, 4096, 36, 8, 128, 2)
        assert n * per <= budget < (n + 1) * per


def test_summary_is_one_sixteenth_of_full_kv():
    for D in (64, 128):
        for nb in (1, 64, 2048):
            assert 16 * sizing.summary_bytes(D, nb) == sizing.full_kv_bytes(D, nb)
    # the selected working set of the default budget: K = 128 blocks = 2,048 tokens
    assert sizing.selected_kv_bytes(128, 128, 0) == 2048 * 2 * 128 * 2


def _table2():
    with open(os.path.join(GOLDEN, "fetch_cap_table2.json")) as f:
        return json.load(f)["rows"]


def test_eq3_reproduces_table2_per_step_fetch():
    """A step of a batch of about 128 sequences lasts 128 / TPS seconds; the link
    moving BW for that long moves the printed GB/step (eq. 3), every row within
    the 5 % that the printed digits and the unprinted batch leave."""
    for ratio, gb_step, bw, tps in _table2():
        got = sizing.c_token(bw * 1e9, 128 / tps) / 1e9
        assert abs(got - gb_step) <= 0.05 * gb_step, (ratio, got, gb_step)


def test_eq3_row_ratios_need_no_batch():
    """Between two rows the batch cancels: eq. (3) predicts GB/step_i / GB/step_j
    = (BW_i / TPS_i) / (BW_j / TPS_j); within 9 % for every pair (two rows'
    rounding)."""
    rows = _table2()
    for ri, gi, bi, ti in rows:
        for rj, gj, bj, tj in rows:
            pred = sizing.c_token(bi, 1.0 / ti) / sizing.c_token(bj, 1.0 / tj)
            assert abs(pred / (gi / gj) - 1.0) <= 0.09, (ri, rj)
