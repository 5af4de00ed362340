"""CPU checks of the decode work plan (cf_decode_plan, the same formula the
decode kernels evaluate on the device): items are (request, KV head, chunk
of pages); the item count never exceeds the partial-output workspace the
engine sizes at creation (Decode Token Parallelism §4.4: split-K partials
with their log-sum-exp statistics)."""
import math
import random

import pytest

WARPS_PER_CTA = 8


@pytest.fixture(scope="module")
def cf():
    from co_prefill_decode_gb300 import build
    build.build()
    import co_prefill_decode_gb300 as cf
    cf.load_library()
    return cf


def pages_of(keys, stride):
    return min(stride, -(-keys // 16)) if keys > 0 else 0


def test_equal_lengths_take_fewer_longer_items(cf):
    # 16 requests at 8192 cached keys + the new one: 513 pages each, 8 KV heads, 152 CTAs x 8 warps
    p = cf.cf_decode_plan([8193] * 16, 513, 8)
    assert p["chunk"] == math.ceil(16 * 513 * 8 / (2 * 152 * WARPS_PER_CTA))      # 2 items per warp
    assert p["items"] == 16 * 8 * math.ceil(513 / p["chunk"])
    # the same total spread unequally: 4 items per warp, shorter chunks
    q = cf.cf_decode_plan([600, 30000, 5000, 7000], 2000, 8)
    tot = sum(pages_of(k, 2000) for k in (600, 30000, 5000, 7000))
    assert q["chunk"] == max(4, math.ceil(tot * 8 / (4 * 152 * WARPS_PER_CTA)))


def test_short_contexts_use_the_minimum_chunk_and_clamp_to_the_table(cf):
    p = cf.cf_decode_plan([18, 65, 101, 256], 17, 2)
    assert p["chunk"] == 4
    assert p["items"] == 2 * sum(math.ceil(pages_of(k, 17) / 4) for k in (18, 65, 101, 256))
    # a request with no keys has no items; one past its page table is clamped to the table
    p = cf.cf_decode_plan([0, 1000], 8, 8)
    assert p["items"] == 8 * math.ceil(8 / p["chunk"])


@pytest.mark.parametrize("seed", range(50))
def test_items_fit_the_workspace(cf, seed):
    rng = random.Random(seed)
    n = rng.randint(1, 256)
    hkv = rng.choice([1, 2, 4, 8])
    ctas = rng.choice([152, 148, 80, 16, 1])
    keys = [int(min(65536, max(1, math.exp(rng.gauss(math.log(6346), 1.2))))) for _ in range(n)]
    if rng.random() < 0.3:
        keys = [keys[0]] * n
    stride = max(pages_of(k, 1 << 30) for k in keys)
    p = cf.cf_decode_plan(keys, stride, hkv, ctas)
    assert p["chunk"] >= 4
    assert p["items"] == hkv * sum(math.ceil(pages_of(k, stride) / p["chunk"]) for k in keys)
    assert p["items"] <= p["max_items"]


def test_rejects_bad_arguments(cf):
    for args in ([], 8, 8), ([5], 0, 8), ([5], 8, 0):
        with pytest.raises(cf.CfError):
            cf.cf_decode_plan(*args)
