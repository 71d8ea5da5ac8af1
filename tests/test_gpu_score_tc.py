"""The tensor-core scoring path: estimates with certified radii
(oasis_score_blocks_tc) and the certified selection
(oasis_select_topk_capped_tc).

* Every estimate lies within its radius of the fixed-order score of
  oasis_score_blocks (itself bit-exact against the oracle), on the workloads'
  shapes, ragged lengths, d_h 64, and adversarial keys (one-signed channels,
  heavy cancellation), with a margin: the observed error stays below 1/16 of
  the radius - both with the per-block wrong-side sums the summary build keeps
  (wsum) and without them (read from the summaries in the kernel).
* wsum is an upper bound within 2^-13 of the exact sum.
* The certified selection gives exactly the tables, plans and counts of the
  exact path, and the scores it recomputes are bit-identical to the
  fixed-order ones; the same holds with the radii inflated (more
  recomputation) and with infinite radii (everything recomputed), on exact
  ties, and against the oracle on sampled segments.
"""
import numpy as np
import pytest
import torch

from conftest import bits
from helpers import device_tiles, prior_tables, run_oracle_segment, default_scale, sample_segments
import sparse_kv_cache_quest_gb300 as okv
from synth import workload as wl

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": wl.WORKLOADS[1],
    "qwen3-8b-layer": wl.WORKLOADS[2],
    "qwen3-235b-8seq": wl.WORKLOADS[5].with_(B=8),
    "llama-long-2seq": wl.WORKLOADS[4].with_(B=2),
    "d64-64q": wl.WORKLOADS[5].with_(B=2, D=64),
    "nq32": wl.WORKLOADS[5].with_(B=2, Nd=2),
    "nq48": wl.WORKLOADS[5].with_(B=2, Nd=3),
}


def _summaries(w, seq_len=None, tiles=None):
    tiles = device_tiles(w, 0) if tiles is None else tiles
    sl = (wl.seq_lens(w) if seq_len is None else seq_len).cuda()
    kmin = torch.zeros((w.S, w.D // 8, w.Nb, 8), dtype=torch.bfloat16, device="cuda")
    kmax = torch.zeros_like(kmin)
    wsum = torch.full((w.S, w.Nb), -7.0, dtype=torch.float32, device="cuda")
    okv.oasis_build_summary(tiles, tiles.stride(0), tiles.stride(1), tiles.stride(3), w.B, w.Hkv, w.D, sl, 0, w.Nb,
                            kmin, kmax, w.Nb, wsum=wsum)
    return tiles, sl, kmin, kmax, wsum


def _score_both(w, kmin, kmax, qd, sl, wsum=None):
    exact = torch.full((w.S, w.Nb), -7.0, dtype=torch.float32, device="cuda")
    est = torch.full_like(exact, -7.0)
    rad = torch.full_like(exact, -7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    okv.oasis_score_blocks(kmin, kmax, w.Nb, qd, w.B, w.Hkv, w.G, w.Nd, w.D, sl, w.W, exact, status)
    okv.oasis_score_blocks_tc(kmin, kmax, w.Nb, qd, w.B, w.Hkv, w.G, w.Nd, w.D, sl, w.W, est, rad, status, wsum=wsum)
    torch.cuda.synchronize()
    assert status.item() == 0, okv.strerror(status.item())
    return exact, est, rad


def _check_radius(w, sl, exact, est, rad, margin=16.0):
    ncs = [-(-int(L) // 16) - w.W for L in sl.cpu().tolist()]
    e, a, r = exact.cpu().numpy(), est.cpu().numpy(), rad.cpu().numpy()
    worst = 0.0
    for s in range(w.S):
        nc = ncs[s // w.Hkv]
        if nc <= 0:
            assert np.all(a[s] == -7.0) and np.all(r[s] == -7.0)
            continue
        err = np.abs(a[s, :nc].astype(np.float64) - e[s, :nc])
        assert np.all(r[s, :nc] > 0)
        assert np.all(err <= r[s, :nc]), (s, float((err / r[s, :nc]).max()))
        worst = max(worst, float((err / r[s, :nc]).max()))
        # entries past the candidates are not touched
        assert np.all(a[s, nc:] == -7.0) and np.all(r[s, nc:] == -7.0)
    assert worst * margin <= 1.0, f"observed error reaches {worst:.3g} of the radius"
    return worst


def _wrong_side_sums(w, kmin, kmax):
    """float64 [S][Nb]: sum over dims of |kmax| where kmax < 0 plus kmin where kmin > 0."""
    f = lambda t: torch.from_numpy(bits(t.permute(0, 2, 1, 3).reshape(w.S, w.Nb, w.D)).astype(np.uint32) << 16)  # noqa
    mn = f(kmin).numpy().view(np.float32).astype(np.float64)
    mx = f(kmax).numpy().view(np.float32).astype(np.float64)
    return (np.where(mx < 0, -mx, 0.0) + np.where(mn > 0, mn, 0.0)).sum(axis=-1)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("with_wsum", [True, False])
def test_estimates_within_radius(name, with_wsum):
    okv.load()
    w = CASES[name]
    _, sl, kmin, kmax, wsum = _summaries(w)
    qd = wl.drafts(w, 0).cuda()
    exact, est, rad = _score_both(w, kmin, kmax, qd, sl, wsum if with_wsum else None)
    _check_radius(w, sl, exact, est, rad)


@pytest.mark.parametrize("name", ["tiny", "qwen3-235b-8seq", "d64-64q"])
def test_wrong_side_sums_bound(name):
    okv.load()
    w = CASES[name]
    _, sl, kmin, kmax, wsum = _summaries(w)
    ref = _wrong_side_sums(w, kmin, kmax)
    got = wsum.cpu().numpy().astype(np.float64)
    nc = w.nc
    assert np.all(got[:, :nc] >= ref[:, :nc])
    assert np.all(got[:, :nc] <= ref[:, :nc] * (1 + 2.0 ** -13))
    assert np.all(got[:, nc:] == -7.0)


# Summary capacities that are not a multiple of 8 blocks (as also in the
# adversarial cases below, 700 blocks): the kernel then moves the summaries with
# 16-byte bulk copies per chunk instead of tensor copies, in whole-half stages
# (16 query columns, d_h 64) or in half-half pieces (32 and 64 columns at d_h
# 128); lengths end inside a block and inside a tile.
ODD = {
    "odd-nb-16q-ragged": wl.WORKLOADS[2].with_(B=3, L=16 * 203),
    "odd-nb-32q": wl.WORKLOADS[5].with_(B=1, Nd=2, L=16 * 301 - 5),
    "odd-nb-64q": wl.WORKLOADS[5].with_(B=1, L=16 * 389 + 7),
    "odd-nb-d64-64q": wl.WORKLOADS[5].with_(B=1, D=64, L=16 * 133),
}


@pytest.mark.parametrize("name", list(ODD))
@pytest.mark.parametrize("with_wsum", [True, False])
def test_estimates_within_radius_odd_capacity(name, with_wsum):
    okv.load()
    w = ODD[name]
    assert w.Nb % 8 != 0
    sl = wl.ragged_seq_lens(w, 16 * 129 + 3) if name.endswith("ragged") else None
    _, sld, kmin, kmax, wsum = _summaries(w, sl)
    qd = wl.drafts(w, 0).cuda()
    exact, est, rad = _score_both(w, kmin, kmax, qd, sld, wsum if with_wsum else None)
    _check_radius(w, sld, exact, est, rad)


def test_estimates_within_radius_ragged_and_empty():
    okv.load()
    w = wl.WORKLOADS[2].with_(B=6)
    sl = wl.ragged_seq_lens(w, 1)
    sl[1] = 0                                    # an empty sequence
    sl[2] = 16 * 128                             # exactly one full tile
    sl[3] = 16 * 129 + 3                         # a tile and a ragged tail
    _, sld, kmin, kmax, wsum = _summaries(w, sl)
    qd = wl.drafts(w, 0).cuda()
    for ws in (wsum, None):
        exact, est, rad = _score_both(w, kmin, kmax, qd, sld, ws)
        _check_radius(w, sld, exact, est, rad)


def _adversarial(w, seed):
    """Keys with one-signed channels (every token of a block above or below zero
    there) and a few blocks of large keys, and queries that make the terms
    cancel: the radius must cover sum |terms|, far above the score itself."""
    g = torch.Generator().manual_seed(seed)
    S, D, Nb = w.S, w.D, w.Nb
    k = torch.randn((S, Nb, 16, D), generator=g)
    pos = torch.randperm(D, generator=g)[:D // 4]     # channels whose keys are all positive
    neg = torch.randperm(D, generator=g)[:D // 8]     # ... all negative
    k[..., pos] = k[..., pos].abs() + 4.0
    k[..., neg] = -(k[..., neg].abs() + 4.0)
    big = torch.randperm(Nb, generator=g)[:Nb // 16]   # a few blocks with large values
    k[:, big] *= 64.0
    tiles = torch.zeros((S, Nb, 2, 16, D), dtype=torch.bfloat16)
    tiles[:, :, 0] = k.to(torch.bfloat16)
    q = torch.randn((w.B, w.Nd, w.Hq, D), generator=g) * 3.0
    _, sl, kmin, kmax, wsum = _summaries(w, tiles=tiles.cuda())
    return sl, kmin, kmax, wsum, q.to(torch.bfloat16).cuda()


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("with_wsum", [True, False])
def test_radius_covers_one_signed_channels_and_cancellation(seed, with_wsum):
    okv.load()
    w = wl.WORKLOADS[5].with_(B=2, L=16 * 700)
    sl, kmin, kmax, wsum, qd = _adversarial(w, seed)
    exact, est, rad = _score_both(w, kmin, kmax, qd, sl, wsum if with_wsum else None)
    _check_radius(w, sl, exact, est, rad)
    # the wrong-side term is active: radii well above 2^-12 |estimate|
    r, a = rad.cpu().numpy(), est.cpu().numpy()
    assert np.median(r / np.maximum(np.abs(a), 1e-30)) > 2.0 ** -12 * 1.5


def _select(w, sl, scores, table0, tc=None):
    S, slots = w.S, w.slots
    tout = torch.full((S, slots), -9, dtype=torch.int32, device="cuda")
    plan = torch.full((S, max(w.cap, 1), 2), -9, dtype=torch.int32, device="cuda")
    cnt = torch.full((S,), -9, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if tc is None:
        okv.oasis_select_topk_capped(scores, w.Nb, sl, w.B, w.Hkv, w.K, w.W, w.cap, table0, tout, plan, cnt, status)
    else:
        rad, kmin, kmax, qd = tc
        okv.oasis_select_topk_capped_tc(scores, rad, kmin, kmax, qd, w.G, w.Nd, w.D, w.Nb, sl, w.B, w.Hkv, w.K, w.W,
                                        w.cap, table0, tout, plan, cnt, status)
    torch.cuda.synchronize()
    return tout.cpu(), plan.cpu(), cnt.cpu(), int(status.item())


def _compare_selection(w, sl, kmin, kmax, qd, table0, inflate=(1.0, 1e3, float("inf")), wsum=None):
    exact, est, rad = _score_both(w, kmin, kmax, qd, sl, wsum)
    ref = _select(w, sl, exact, table0)
    assert ref[3] == 0
    e_np = exact.cpu().numpy()
    recomputed = []
    for f in inflate:
        sc = est.clone()
        r = rad * f if np.isfinite(f) else torch.full_like(rad, float("inf"))
        got = _select(w, sl, sc, table0, (r, kmin, kmax, qd))
        assert got[3] == 0, okv.strerror(got[3])
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]), f
        # recomputed scores are the fixed-order ones, bit for bit; the rest are the estimates
        changed = (sc != est).cpu().numpy()
        s_np = sc.cpu().numpy()
        assert np.array_equal(s_np[changed].view(np.uint32), e_np[changed].view(np.uint32))
        recomputed.append(int(changed.sum()))
    return recomputed, ref


@pytest.mark.parametrize("name", ["tiny", "qwen3-8b-layer", "qwen3-235b-8seq", "llama-long-2seq", "d64-64q"])
def test_certified_selection_equals_exact(name):
    okv.load()
    w = CASES[name]
    tiles, sl, kmin, kmax, wsum = _summaries(w)
    segs = sample_segments(w)
    tiles_cpu = {s: bits(tiles[s]) for s in segs}
    table0 = prior_tables(w, 0, set(segs), lambda s: tiles_cpu[s], wl.seq_lens(w)).cuda()
    qd = wl.drafts(w, 0).cuda()
    recomputed, ref = _compare_selection(w, sl, kmin, kmax, qd, table0, wsum=wsum)
    if w.nc > w.K:
        # with the true radii only a small part of the candidates is recomputed
        assert recomputed[0] < 0.25 * w.S * w.nc, recomputed
    # and the result is the oracle's on the sampled segments
    q = wl.q_true(w, 0)
    for s in segs:
        o = run_oracle_segment(w, 0, s, tiles_cpu[s], w.L, table0[s].tolist(), default_scale(w.D), bits(qd), bits(q))
        assert ref[0][s].tolist() == o["table_out"]
        n = len(o["plan"])
        assert int(ref[2][s]) == n and [tuple(x) for x in ref[1][s, :n].tolist()] == o["plan"]


def test_certified_selection_on_ties_and_ragged_lengths():
    okv.load()
    w = wl.WORKLOADS[5].with_(B=4)
    sl = wl.ragged_seq_lens(w, 16 * 100)
    sl[1] = 16 * 60                                       # fewer candidates than K
    tiles, sld, kmin, kmax, wsum = _summaries(w, sl)
    # exact ties: many blocks share one summary (the rank among them is by block id)
    for s in range(w.S):
        kmin[s, :, 100:160] = kmin[s, :, 99:100]
        kmax[s, :, 100:160] = kmax[s, :, 99:100]
    table0 = torch.stack([wl.prior_random(w, 0, s) for s in range(w.S)])
    for s in range(w.S):                                  # keep the prior within each sequence's candidates
        nc = -(-int(sl[s // w.Hkv]) // 16)
        row = [b if b < nc else -1 for b in table0[s].tolist()]
        table0[s] = torch.tensor(row, dtype=torch.int32)
    qd = wl.drafts(w, 0).cuda()
    _compare_selection(w, sld, kmin, kmax, qd, table0.cuda())   # no wsum: the copied summaries have none


@pytest.mark.parametrize("seed", [4, 5])
def test_certified_selection_on_adversarial_summaries(seed):
    okv.load()
    w = wl.WORKLOADS[5].with_(B=2, L=16 * 700, K=64)
    sl, kmin, kmax, wsum, qd = _adversarial(w, seed)
    table0 = torch.stack([wl.prior_random(w, 0, s) for s in range(w.S)]).cuda()
    _compare_selection(w, sl, kmin, kmax, qd, table0, wsum=wsum)
