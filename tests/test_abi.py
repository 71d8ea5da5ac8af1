"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before any launch (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import sparse_kv_cache_quest_gb300 as okv
from sparse_kv_cache_quest_gb300 import binding as ob


def _declared():
    with open(os.path.join(ROOT, "include", "oasis.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(oasis_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_cache_quest_gb300 import build
    build.build()
    return ob.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(ob.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    assert okv.abi_version() == 3


def test_strerror(lib):
    assert "invalid" in okv.strerror(-1)
    assert "NaN" in okv.strerror(ob.STATUS_NAN_SCORE)


def _einval(fn, *args):
    with pytest.raises(ob.OasisError) as e:
        fn(*args)
    assert e.value.code == ob.EINVAL


# A 16-byte aligned fake address.  Every call below is rejected by a check that
# looks only at the arguments themselves (null, alignment, ranges, sizes from the
# same device-independent formula), before anything reads device state.
P = 1 << 20


def test_build_summary_validation(lib):
    f = okv.oasis_build_summary
    _einval(f, P, 0, 0, 0, 1, 1, 96, P, 0, 1, P, P, 4, None, 0)          # D
    _einval(f, P, 0, 0, 0, 1, 1, 128, P, 3, 2, P, P, 4, None, 0)         # range past Nb_max
    _einval(f, P, 4, 0, 0, 1, 1, 128, P, 0, 1, P, P, 4, None, 0)         # stride not a multiple of 8
    _einval(f, P + 2, 0, 0, 0, 1, 1, 128, P, 0, 1, P, P, 4, None, 0)     # misaligned keys
    _einval(f, None, 0, 0, 0, 1, 1, 128, P, 0, 1, P, P, 4, None, 0)      # NULL
    _einval(f, P, 0, 0, 0, 0, 1, 128, P, 0, 1, P, P, 4, None, 0)         # B
    with pytest.raises(ob.OasisError):                                    # misaligned wrong-side sums
        f(P, 0, 0, 0, 1, 1, 128, P, 0, 1, P, P, 4, None, 0, wsum=P + 2)


def test_score_validation(lib):
    f = okv.oasis_score_blocks
    _einval(f, P, P, 16, P, 1, 1, 17, 1, 128, P, 0, P, None, 0)          # G > 16
    _einval(f, P, P, 16, P, 1, 1, 16, 5, 128, P, 0, P, None, 0)          # G*Nd > 64
    _einval(f, P, P, 16, P, 1, 1, 4, 1, 128, P, -1, P, None, 0)          # W < 0
    _einval(f, P, P, 0, P, 1, 1, 4, 1, 128, P, 0, P, None, 0)            # Nb_max
    _einval(f, P, P, 16, P + 8, 1, 1, 4, 1, 128, P, 0, P, None, 0)       # qdraft not 16-byte aligned


def test_score_tc_validation(lib):
    f = okv.oasis_score_blocks_tc
    _einval(f, P, P, 16, P, 1, 1, 17, 1, 128, P, 0, P, P, None, 0)       # G > 16
    _einval(f, P, P, 16, P, 1, 1, 16, 5, 128, P, 0, P, P, None, 0)       # G*Nd > 64
    _einval(f, P, P, 16, P, 1, 1, 4, 1, 96, P, 0, P, P, None, 0)         # D
    _einval(f, P, P, 16, P, 1, 1, 4, 1, 128, P, 0, P, None, None, 0)     # radius required
    _einval(f, P, P, 16, P, 1, 1, 4, 1, 128, P, 0, P, P + 2, None, 0)    # radius misaligned


def test_select_tc_validation(lib):
    f = okv.oasis_select_topk_capped_tc
    #   scores radius kmin kmax qd  G  Nd  D  Nb_max sl  B  Hkv K  W  cap tin tout plan cnt status
    _einval(f, P, P, P, P, P, 4, 1, 128, 20000, P, 1, 1, 8, 0, 2, P, P, P, P, P, 0)   # Nb_max > 16384
    _einval(f, P, P, P, P, P, 4, 1, 96, 64, P, 1, 1, 8, 0, 2, P, P, P, P, P, 0)       # D
    _einval(f, P, P, P, P, P, 17, 1, 128, 64, P, 1, 1, 8, 0, 2, P, P, P, P, P, 0)     # G
    _einval(f, P, None, P, P, P, 4, 1, 128, 64, P, 1, 1, 8, 0, 2, P, P, P, P, P, 0)   # radius
    _einval(f, P, P, P + 8, P, P, 4, 1, 128, 64, P, 1, 1, 8, 0, 2, P, P, P, P, P, 0)  # kmin alignment
    _einval(f, P, P, P, P, P, 4, 1, 128, 64, P, 1, 1, 8, 0, 9, P, P, P, P, P, 0)      # cap > K


def test_select_validation(lib):
    f = okv.oasis_select_topk_capped
    _einval(f, P, 64, P, 1, 1, 8, 0, 9, P, P, P, P, P, 0)                # cap > K
    _einval(f, P, 64, P, 1, 1, 0, 0, 0, P, P, P, P, P, 0)                # K = 0
    _einval(f, P, 64, P, 1, 1, 8, 0, 2, P, P, P, P, None, 0)             # status required
    _einval(f, P, 40000, P, 1, 1, 8, 0, 2, P, P, P, P, P, 0)             # Nb_max too large


def test_attention_workspace_validation(lib):
    assert okv.oasis_attn_workspace_bytes(2, 4, 4, 128, 128) > 0
    assert okv.oasis_attn_workspace_bytes(2, 4, 4, 96, 128) == 0                    # D
    assert okv.oasis_attn_workspace_bytes(2, 4, 17, 128, 128) == 0                  # G
    f = okv.oasis_sparse_decode_attn_ws
    n = okv.oasis_attn_workspace_bytes(1, 1, 4, 128, 8)
    _einval(f, P, P, P, 8, P, 1, 1, 4, 128, 0.1, P, None, None, n, None, 0)      # NULL workspace
    _einval(f, P, P, P, 8, P, 1, 1, 4, 128, 0.1, P, None, P, n - 1, None, 0)     # workspace too small
    _einval(f, P, P, P, 8, P, 1, 1, 4, 128, 0.1, P, None, P + 8, n, None, 0)     # misaligned workspace


def test_stage_and_attention_validation(lib):
    _einval(okv.oasis_stage_blocks, P, 8, 4, P, P, 2, 1, 1, 128, P, 8, P, 0)        # stride % 16
    _einval(okv.oasis_stage_blocks, P, 16, 0, P, P, 2, 1, 1, 128, P, 8, P, 0)       # host_nb
    _einval(okv.oasis_sparse_decode_attn, P, P, P, 8, P, 1, 1, 0, 128, 0.1, P, None, None, 0)  # G
    _einval(okv.oasis_sparse_decode_attn, P, P, P, 0, P, 1, 1, 4, 128, 0.1, P, None, None, 0)  # slots
    _einval(okv.oasis_sparse_decode_attn, P + 8, P, P, 8, P, 1, 1, 4, 128, 0.1, P, None, None, 0)  # q align
    f = okv.oasis_sparse_decode_attn_tc
    _einval(f, P, P, P, 8, P, 1, 1, 4, 64, 0.1, P, None, None, 0)        # D 64: the tcgen05 kernel takes d_h 128
    _einval(f, P, P, P, 8, P, 1, 1, 17, 128, 0.1, P, None, None, 0)      # G
    _einval(f, P, P + 8, P, 8, P, 1, 1, 4, 128, 0.1, P, None, None, 0)   # pool not 16-byte aligned
    _einval(f, P, P, None, 8, P, 1, 1, 4, 128, 0.1, P, None, None, 0)    # NULL table
