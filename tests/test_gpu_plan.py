"""The launch plan a step takes (``lf_step_plan``): consistent with the shape,
with the environment switches and with the cluster residency the device
reports. The plans the bench workloads rely on are pinned here."""
import pytest

import decode_kv_cache_step_gb300 as lf

pytestmark = pytest.mark.gpu

TILE = 64
SHAPES = [(1, 32, 8, 128, 2400), (2, 32, 8, 128, 3200), (4, 32, 8, 128, 3200),
          (8, 32, 8, 128, 3200), (128, 32, 8, 128, 3200), (256, 32, 8, 128, 2400),
          (32, 32, 8, 128, 16384), (2, 4, 2, 64, 256), (1, 8, 1, 64, 9000), (3, 2, 2, 128, 1)]


@pytest.mark.parametrize("shape", SHAPES)
def test_plan_covers_the_slots(shape):
    B, Hq, Hkv, d, S = shape
    p = lf.step_plan(B, Hq, Hkv, d, S)
    tiles = -(-S // TILE)
    assert 1 <= p["chunk_tiles"] <= 32
    assert p["nchunk"] == -(-tiles // p["chunk_tiles"])
    assert p["stages"] in (2, 3, 6)
    if p["cluster"]:
        assert p["nchunk"] <= 16 and not p["split"]
        assert p["cluster_fit"] >= 1
    if p["stages"] == 6:
        assert p["cluster"]


@pytest.mark.parametrize("cmax", [None, "8", "4"])
@pytest.mark.parametrize("shape", SHAPES)
def test_clusters_only_when_all_resident(monkeypatch, shape, cmax):
    """Without LF_CLUSTER=1 a cluster plan has every unit's cluster resident
    at once, within the cap."""
    B, Hq, Hkv, d, S = shape
    if cmax:
        monkeypatch.setenv("LF_CLUSTER_MAX", cmax)
    p = lf.step_plan(B, Hq, Hkv, d, S)
    if p["cluster"]:
        assert p["nchunk"] <= int(cmax or 16) and B * Hkv <= p["cluster_fit"]


@pytest.mark.parametrize("B,S", [(8, 3200), (16, 3200), (20, 2400), (4, 16384), (2, 30000)])
def test_longer_chunks_to_fit_clusters(monkeypatch, B, S):
    """A batch too large for clusters of its short-chunk plan takes fewer,
    longer chunks whose clusters all fit; the next larger cluster would not."""
    Hq, Hkv, d = 32, 8, 128
    p = lf.step_plan(B, Hq, Hkv, d, S)
    assert p["cluster"] and B * Hkv <= p["cluster_fit"], p
    tiles = -(-S // TILE)
    ct_next = -(-tiles // (p["nchunk"] + 1))
    if p["nchunk"] < 16 and ct_next < p["chunk_tiles"]:
        # Forced clusters of the next size report how many fit at once.
        monkeypatch.setenv("LF_CHUNK_TILES", str(ct_next))
        monkeypatch.setenv("LF_CLUSTER", "1")
        q = lf.step_plan(B, Hq, Hkv, d, S)
        assert q["cluster"] and q["nchunk"] > p["nchunk"], (p, q)
        assert B * Hkv > q["cluster_fit"], (p, q)


@pytest.mark.parametrize("shape", SHAPES)
def test_switches(monkeypatch, shape):
    B, Hq, Hkv, d, S = shape
    monkeypatch.setenv("LF_CLUSTER", "0")
    p = lf.step_plan(B, Hq, Hkv, d, S)
    assert not p["cluster"] and p["stages"] == 2 and p["cluster_fit"] == -1
    monkeypatch.setenv("LF_SPLIT", "0")
    assert not lf.step_plan(B, Hq, Hkv, d, S)["split"]
    monkeypatch.setenv("LF_CHUNK_TILES", "7")
    assert lf.step_plan(B, Hq, Hkv, d, S)["chunk_tiles"] == min(7, -(-S // TILE))
    monkeypatch.setenv("LF_STAGES", "3")
    assert lf.step_plan(B, Hq, Hkv, d, S)["stages"] == 3


def test_topk_above_one_never_clusters():
    for shape in SHAPES:
        p = lf.step_plan(*shape, topk=4)
        assert not p["cluster"] and not p["split"]


def test_bench_workload_plans():
    # The Fig. 1 shape: 4 chunks of 13 tiles per unit, last-CTA merge.
    p = lf.step_plan(128, 32, 8, 128, 3200)
    assert (p["nchunk"], p["chunk_tiles"], p["cluster"], p["split"]) == (4, 13, False, False)
    # 16K-slot units: the split finish.
    assert lf.step_plan(32, 32, 8, 128, 16384)["split"]
    # One 2400-slot sequence: a cluster merge.
    assert lf.step_plan(1, 32, 8, 128, 2400)["cluster"]


def test_invalid_shapes_are_refused():
    with pytest.raises(lf.LFError):
        lf.step_plan(1, 6, 4, 128, 100)   # Hq not a multiple of Hkv
    with pytest.raises(lf.LFError):
        lf.step_plan(1, 32, 8, 96, 100)   # head dim 96
    with pytest.raises(lf.LFError):
        lf.step_plan(1, 32, 8, 128, 100, topk=0)
