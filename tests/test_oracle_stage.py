"""Pin of the staging oracle: exactly the planned slots change, byte for byte."""
import numpy as np

from oracle.stage import STATUS_PLAN_RANGE, stage_blocks


def test_planned_slots_replaced_others_untouched():
    rng = np.random.default_rng(5)
    host = rng.integers(0, 65536, (10, 2, 16, 8), dtype=np.uint16)
    pool = rng.integers(0, 65536, (4, 2, 16, 8), dtype=np.uint16)
    out, st = stage_blocks(host, [(7, 1), (2, 3)], pool)
    assert st == 0
    assert np.array_equal(out[1], host[7]) and np.array_equal(out[3], host[2])
    assert np.array_equal(out[[0, 2]], pool[[0, 2]])
    out2, st2 = stage_blocks(host, [(10, 0), (1, 4)], pool)
    assert st2 == STATUS_PLAN_RANGE and np.array_equal(out2, pool)
