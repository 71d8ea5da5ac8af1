"""Pins of the closed forms: eqs. (1)/(2) against the page's worked example."""
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


def test_eq3_eq4():
    assert sizing.c_token(64e9, 0.02) == 64e9 * 0.02
    assert sizing.pipeline_fits(1.0, 2.0, 3.0, 36 * 3.0, 36)
    assert not sizing.pipeline_fits(1.0, 2.0, 3.5, 36 * 3.0, 36)
