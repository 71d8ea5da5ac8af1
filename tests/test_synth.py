"""The seeded input generator: published splitmix64, stable draws, shapes."""
import torch

from synth import rng, workload as wl


def test_splitmix64_matches_integer_reference():
    x = torch.tensor([0, 1, 2**62, -1, -(2**63), 123456789], dtype=torch.int64)
    got = rng.splitmix64(x).tolist()
    ref = [rng._s64(rng.splitmix64_int(v & ((1 << 64) - 1))) for v in x.tolist()]
    assert got == ref


def test_normal_bf16_moments_and_determinism():
    idx = torch.arange(200_000)
    a = rng.normal_bf16(7, 1, idx)
    assert torch.equal(a, rng.normal_bf16(7, 1, idx))
    assert not torch.equal(a, rng.normal_bf16(8, 1, idx))
    f = a.float()
    assert abs(f.mean().item()) < 0.01 and abs(f.std().item() - 1.0) < 0.01
    # the fp32 form rounds to the bf16 form
    assert torch.equal(rng.normal_f32(7, 1, idx).to(torch.bfloat16), a)


def test_subsets_and_orders():
    s = rng.random_subset(3, 5, 100, 50, 10)
    assert s.tolist() == sorted(set(s.tolist())) and len(s) == 10 and s.max() < 50
    p = rng.random_order(3, 5, 100, 50)
    assert sorted(p.tolist()) == list(range(50))


def test_workload_shapes_and_structure():
    w = wl.WORKLOADS[1]
    k = wl.keys(w, 0, [1])
    assert k.shape == (1, w.Nb, 16, w.D) and k.dtype == torch.bfloat16
    v = wl.values(w, 0, [0, 1])
    assert v.shape == (2, w.Nb, 16, w.D)
    t = wl.kv_tiles(w, 0, [1])
    assert torch.equal(t[:, :, 0], k)
    # segment draws do not depend on which other segments are generated
    assert torch.equal(wl.keys(w, 0, [0, 1])[1], k[0])
    assert wl.prior_random(w, 0, 0).shape == (w.K + w.W,)
    d = wl.drafts(w, 0)
    assert d.shape == (w.B, w.Nd, w.Hq, w.D)
    w2 = wl.WORKLOADS[2]
    assert w2.cap == 7 and wl.WORKLOADS[1].cap == 2 and w2.with_(fetch_ratio="0.1", K=30).cap == 3


def test_planted_blocks_drift_stays_distinct_and_in_range():
    w = wl.WORKLOADS[5].with_(L=16 * 200, plants=16)
    prev = wl.planted_blocks(w, 0, 3, 0)
    for st in range(1, 8):
        cur = wl.planted_blocks(w, 0, 3, st)
        assert len(set(cur.tolist())) == len(cur) == 16
        assert cur.min() >= 0 and cur.max() < w.nc
        moved = sorted(set(cur.tolist()) ^ set(prev.tolist()))
        assert len(moved) > 0
        prev = cur


def test_prior_from_topk_overlap():
    w = wl.WORKLOADS[2]
    topk = list(range(0, 256, 2))
    t = wl.prior_from_topk(w, 0, 5, topk)
    blocks = [b for b in t.tolist() if b >= 0]
    assert len(blocks) == 128 and len(set(blocks)) == 128
    assert len(set(blocks) & set(topk)) == 115
    assert blocks == sorted(blocks)
