"""CPU checks of the prefill work plan (cf_prefill_plan): the work unit kind,
the key-range cuts per chunk and the queue length, on the layer workloads'
chunks and on random chunk lists (Adaptive Context Parallelism §2.2 Eq. 1:
a query tile's keys are the cached prefix plus the causal part of the
chunk)."""
import random

import pytest

BQ = 128          # query tile rows
BKV = 128         # key tile columns
MAX_SPLITS = 16
PART_TILES = 2048


@pytest.fixture(scope="module")
def cf():
    from co_prefill_decode_gb300 import build
    build.build()
    import co_prefill_decode_gb300 as cf
    cf.load_library()
    return cf


def kv_tiles(prefix, length, qt):
    """Key tiles the query tile qt of a chunk reaches (causal, within the request)."""
    end = min(prefix + (qt + 1) * BQ, prefix + length)
    return -(-end // BKV)


def units(kind, n_qt, hq):
    return n_qt * (hq // 2) if kind == 2 else ((n_qt + 1) // 2 if kind == 1 else n_qt) * hq


def reach_min(kind, prefix, length):
    n_qt = -(-length // BQ)
    return kv_tiles(prefix, length, min(1, n_qt - 1) if kind == 1 else 0)


# (chunks, Hq, Hkv) of the layer workloads: Qwen3-14B (G = 5), Qwen3-32B and Llama-3.1-8B (G = 8, 4)
def test_plans_of_the_layer_workloads(cf):
    p = cf.cf_prefill_plan([(2048, 16384)], 40, 8)
    # odd group: tile pairs; 320 units are fewer than 4 per SM of 152, so each is cut into 2
    assert p == {"kind": 1, "splits": [2], "cut_from": [0], "items": 640}
    p = cf.cf_prefill_plan([(4096, 28672)], 64, 8)
    # 32 tiles x 32 head pairs = 1024 whole units, more than two waves: the
    # last wave's worth (152 units) is cut into 4 key ranges
    assert p == {"kind": 2, "splits": [4], "cut_from": [1024 - 152], "items": 872 + 152 * 4}
    p = cf.cf_prefill_plan([(1024, 0)], 32, 8)
    # the first tile has one key tile: no cut
    assert p == {"kind": 2, "splits": [1], "cut_from": [128], "items": 128}
    # four chunks: units cut where each range keeps >= 16 key tiles
    p = cf.cf_prefill_plan([(1024, 0), (512, 4096), (256, 12288), (128, 2048)], 32, 8)
    assert p["kind"] == 2 and p["splits"] == [1, 2, 3, 1]
    assert p["cut_from"] == [128, 0, 0, 16]
    assert p["items"] == 16 * (8 * 1 + 4 * 2 + 2 * 3 + 1 * 1)
    # a long chunk without prefix ends on its lightest units: no tail cut
    p = cf.cf_prefill_plan([(8192, 0)], 32, 8)
    assert p == {"kind": 2, "splits": [1], "cut_from": [1024], "items": 1024}


def test_forced_modes(cf):
    chunks = [(2048, 16384)]
    assert cf.cf_prefill_plan(chunks, 40, 8, split_mode=1)["splits"] == [1]
    assert cf.cf_prefill_plan(chunks, 40, 8, split_mode=3)["splits"] == [3]
    assert cf.cf_prefill_plan(chunks, 40, 8, pairing_mode=1)["kind"] == 0
    assert cf.cf_prefill_plan(chunks, 40, 8, pairing_mode=2)["kind"] == 1
    with pytest.raises(cf.CfError):   # head pairs need an even GQA group
        cf.cf_prefill_plan(chunks, 40, 8, pairing_mode=3)
    assert cf.cf_prefill_plan(chunks, 32, 8, pairing_mode=3)["kind"] == 2
    for bad in ([], [(0, 5)], [(16, -1)]):
        with pytest.raises(cf.CfError):
            cf.cf_prefill_plan(bad, 32, 8)


@pytest.mark.parametrize("seed", range(40))
def test_random_chunk_lists_cover_every_unit(cf, seed):
    rng = random.Random(seed)
    hq, hkv = rng.choice([(32, 8), (40, 8), (64, 8), (4, 2), (28, 4)])
    n = rng.randint(1, 8)
    chunks = [(rng.choice([1, 17, 128, 200, 512, 1024, 2048, 4096]), rng.choice([0, 5, 128, 3000, 16384]))
              for _ in range(n)]
    sms = rng.choice([152, 148, 72, 7])
    mode = rng.choice([0, 0, 1, 2, 5])
    p = cf.cf_prefill_plan(chunks, hq, hkv, sms, split_mode=mode)
    kind, splits = p["kind"], p["splits"]
    assert kind in (0, 1, 2) and (kind != 2 or (hq // hkv) % 2 == 0)
    if (hq // hkv) % 2 == 0:
        assert kind == 2
    total, parts, tail_cut = 0, 0, False
    for (length, prefix), s, c in zip(chunks, splits, p["cut_from"]):
        n_qt = -(-length // BQ)
        u = units(kind, n_qt, hq)
        # every range of a cut unit keeps at least one key tile
        assert 1 <= s <= min(MAX_SPLITS, reach_min(kind, prefix, length))
        assert 0 <= c <= u and (s > 1 or c == u)
        if mode == 1:
            assert s == 1
        if mode >= 2:
            assert s <= mode and (s == 1 or c == 0)
        if s > 1 and c > 0:   # only the tail of a long queue is cut part-way
            assert mode == 0 and s <= 4 and 8 * s <= reach_min(kind, prefix, length)
            tail_cut = True
        total += c + (u - c) * s
        parts += 2 * (u - c) * s if s > 1 else 0
    assert p["items"] == total
    assert parts <= PART_TILES
    if tail_cut:   # at most one wave's worth of units is cut at the tail
        assert sum(u - c for (l, pf), c, s in zip(chunks, p["cut_from"], splits) if s > 1 for u in
                   [units(kind, -(-l // BQ), hq)]) <= sms
