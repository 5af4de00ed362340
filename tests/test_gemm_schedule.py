"""CPU checks of the GEMM work split (cf_gemm_schedule): whole tiles for the
full waves, then the tiles of a partial last wave cut into equal k-chunks,
one chunk per CTA."""
import pytest

SHAPES = [  # (M, N, K, epilogue): the stacked token matrices of the layer workloads and small cases
    (1040, 6144, 4096, 0), (1040, 4096, 4096, 1), (1040, 14336, 4096, 3), (1040, 4096, 14336, 2),
    (384, 6144, 4096, 0), (384, 4096, 4096, 1), (384, 14336, 4096, 3), (384, 4096, 14336, 2),
    (2080, 7168, 5120, 0), (2080, 5120, 17408, 2), (4128, 5120, 25600, 2), (4128, 25600, 5120, 3),
    (1, 256, 64, 0), (200, 768, 4096, 0), (300, 256, 8192, 1), (68, 512, 256, 0), (4128, 2048, 256, 0),
    (128, 4096, 4096, 0),
]


@pytest.fixture(scope="module")
def cf():
    from co_prefill_decode_gb300 import build
    build.build()
    import co_prefill_decode_gb300 as cf
    cf.load_library()
    return cf


def units(G, tiles, dp_tiles, split, num_kb):
    """The units of every CTA under the documented rule: whole tiles c, c + G,
    ... below dp_tiles, then chunk c // R of tail tile dp_tiles + c % R."""
    R = tiles - dp_tiles
    out = []
    for c in range(G):
        us = [(t, 0, num_kb) for t in range(c, dp_tiles, G)]
        if c < R * split:
            s = c // R
            us.append((dp_tiles + c % R, s * num_kb // split, (s + 1) * num_kb // split))
        out.append(us)
    return out


@pytest.mark.parametrize("M,N,K,epi", SHAPES)
@pytest.mark.parametrize("ctas", [152, 148, 7])
@pytest.mark.parametrize("mode", [0, 1, 2, 5])
def test_schedule_covers_every_k_block_once(cf, M, N, K, epi, ctas, mode):
    s = cf.cf_gemm_schedule(M, N, K, epi, ctas, mode)
    num_m = -(-M // 128)
    num_n = N // 128 if epi == 3 else N // 256
    num_kb = K // 64
    assert s["tiles"] == num_m * num_n
    assert 1 <= s["grid"] <= ctas
    if s["split"] == 1:
        assert s["dp_tiles"] == s["tiles"] and s["grid"] == min(s["tiles"], ctas)
        return
    assert mode != 1 and 2 <= s["split"] <= num_kb
    assert mode < 2 or s["split"] <= mode
    G, R = s["grid"], s["tiles"] - s["dp_tiles"]
    assert s["dp_tiles"] % ctas == 0 and 0 < R < ctas and R * s["split"] <= G
    seen = set()
    for us in units(G, s["tiles"], s["dp_tiles"], s["split"], num_kb):
        for t, k0, k1 in us:
            assert 0 <= k0 < k1 <= num_kb
            for kb in range(k0, k1):
                assert (t, kb) not in seen
                seen.add((t, kb))
    assert len(seen) == s["tiles"] * num_kb


@pytest.mark.parametrize("M,N,K,epi", SHAPES)
def test_split_only_when_it_shortens_the_critical_path(cf, M, N, K, epi):
    G = 152
    s = cf.cf_gemm_schedule(M, N, K, epi, G)
    num_kb = K // 64
    whole = -(-s["tiles"] // G) * num_kb          # k-blocks on the busiest CTA, whole tiles only
    if s["split"] > 1:
        cut = s["dp_tiles"] // G * num_kb + -(-num_kb // s["split"])
        assert cut < whole
    off = cf.cf_gemm_schedule(M, N, K, epi, G, 1)
    assert off["split"] == 1 and off["dp_tiles"] == off["tiles"]


def test_schedule_cuts_the_small_batch_tails(cf):
    # FFN down projection of a 384-token batch: 48 tiles of 224 k-blocks
    # would keep 104 of 152 SMs idle; cut in 3 chunks they fill 144
    s = cf.cf_gemm_schedule(384, 4096, 14336, 2, 152)
    assert s["dp_tiles"] == 0 and s["split"] == 3 and s["grid"] == 144
    # 2080 tokens, FFN down: 2 full waves, then 36 tiles cut in 4
    s = cf.cf_gemm_schedule(2080, 5120, 17408, 2, 152)
    assert s["dp_tiles"] == 304 and s["split"] == 4 and s["grid"] == 152
    # 144 tiles on 152 SMs: one nearly full wave, nothing to gain
    s = cf.cf_gemm_schedule(1040, 4096, 4096, 1, 152)
    assert s["split"] == 1 and s["grid"] == 144
    # a 64-tile second wave of short (64 k-block) tiles: the fix-up would
    # cost about what the cut saves, so the tiles stay whole
    s = cf.cf_gemm_schedule(1040, 6144, 4096, 0, 152)
    assert s["split"] == 1


def test_schedule_rejects_bad_sizes(cf):
    for args in [(0, 256, 64, 0, 152), (128, 256, 64, 0, 0), (128, 256, 64, 9, 152), (128, -256, 64, 0, 152),
                 (128, 256, 64, 0, 152, -1)]:
        with pytest.raises(cf.CfError):
            cf.cf_gemm_schedule(*args)
