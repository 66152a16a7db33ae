"""The f32 GEMM's schedule, worked out on the host (phx_selftest_sgemm_schedule): no GPU.

On a 152-SM GPU with two 128 x 128 CTAs per SM (304 slots) the library picks, per shape:
whole tiles; a grid split along K into slices (added by a reduction); or stream-K blocks
that share the k tiles of the last partial wave -- or of a whole grid of less than one wave
-- evenly, written as partial tiles that a fix-up adds in k order.  These tests pin the
decisions the measurements in the design notes led to, and check on every plan that the
partial tiles the fix-up adds for a tile are, in k order, exactly the ones the stream-K
blocks write for it, covering its k tiles once, with at most two segments per block.
"""
import random

import pytest

from dense_gemm_04_gb300 import phx

CFG = "TILE_M=128 TILE_N=128 TILE_K=16 STAGES=4 FMA2=1"


@pytest.mark.parametrize("shape,want", [
    # whole waves, then the last partial wave spread over one block per slot
    ((4096, 4096, 4096), dict(whole_tiles=912, streamk_blocks=304, k_slices=1)),
    ((4096, 3840, 4096), dict(whole_tiles=912, streamk_blocks=304, k_slices=1)),
    ((4096, 4352, 512), dict(whole_tiles=912, streamk_blocks=304, k_slices=1)),
    # a whole grid of less than one wave, spread
    ((256, 256, 256), dict(whole_tiles=0, streamk_blocks=8, k_slices=1)),
    ((512, 512, 512), dict(whole_tiles=0, streamk_blocks=64, k_slices=1)),
    ((2048, 2048, 2048), dict(whole_tiles=0, streamk_blocks=304, k_slices=1)),
    ((1024, 1024, 16384), dict(whole_tiles=0, streamk_blocks=304, k_slices=1)),
    ((16384, 128, 4096), dict(whole_tiles=0, streamk_blocks=304, k_slices=1)),
    # split along K where that measured faster
    ((1024, 1024, 1024), dict(whole_tiles=64, streamk_blocks=0, k_slices=4)),
    ((300, 500, 3000), dict(whole_tiles=12, streamk_blocks=0, k_slices=8)),
    # tiles only: a short K, or a last wave already as good as spread
    ((2048, 2048, 256), dict(whole_tiles=256, streamk_blocks=0, k_slices=1)),
    ((4095, 4097, 4093), dict(whole_tiles=1056, streamk_blocks=0, k_slices=1)),
    ((8192, 8192, 1024), dict(whole_tiles=4096, streamk_blocks=0, k_slices=1)),
])
def test_documented_schedules(shape, want):
    got = phx.sgemm_schedule(CFG, *shape)
    for key, value in want.items():
        assert got[key] == value, (shape, key, got)
    assert got["bookkeeping_ok"] == 1 and got["max_segments"] <= 2, (shape, got)


def test_spread_covers_the_tail_exactly():
    # whole tiles + spread tiles = all tiles; every block gets at least 8 k tiles
    for shape in ((4096, 4096, 4096), (2304, 2304, 2048), (2300, 2310, 2000), (1000, 1000, 8000)):
        M, N, K = shape
        got = phx.sgemm_schedule(CFG, M, N, K)
        tiles = -(-M // 128) * -(-N // 128)
        k_tiles = -(-K // 16)
        tail = tiles - got["whole_tiles"]
        assert got["streamk_blocks"] > 0, shape
        assert got["streamk_k_tiles"] == tail * k_tiles, (shape, got)
        assert tail <= got["streamk_blocks"] <= 304, (shape, got)
        assert got["streamk_k_tiles"] // got["streamk_blocks"] >= 8, (shape, got)


def test_random_plans_are_consistent():
    # every tile configuration, random shapes and machine sizes
    rng = random.Random(7)
    names = [n for n in phx.config_names(phx.VARIANT_SGEMM) if n != "SKINNY"]
    spread = 0
    for _ in range(600):
        cfg = rng.choice(names)
        M, N, K = rng.randint(1, 20000), rng.randint(1, 20000), rng.randint(1, 40000)
        per_sm, sms = rng.choice((1, 2, 3, 4, 8)), rng.choice((1, 8, 66, 132, 148, 152, 160))
        got = phx.sgemm_schedule(cfg, M, N, K, per_sm, sms)
        assert got["bookkeeping_ok"] == 1, (cfg, M, N, K, per_sm, sms, got)
        assert got["max_segments"] <= 2, (cfg, M, N, K, per_sm, sms, got)
        assert got["streamk_blocks"] <= per_sm * sms
        assert got["streamk_blocks"] == 0 or got["k_slices"] == 1
        spread += got["streamk_blocks"] > 0
    assert spread > 50  # the random shapes do exercise the stream-K plans


def test_schedule_argument_checks():
    idx = phx.config_names(phx.VARIANT_SGEMM).index(CFG)
    out = (phx.ctypes.c_int64 * 6)()
    assert phx.phx_selftest_sgemm_schedule(idx, 64, 64, 64, 2, 152, out) == phx.PHX_OK
    skinny = phx.config_names(phx.VARIANT_SGEMM).index("SKINNY")
    for args in ((skinny, 64, 64, 64, 2, 152), (-1, 64, 64, 64, 2, 152), (idx, 0, 64, 64, 2, 152),
                 (idx, 64, 64, 64, 0, 152), (idx, 64, 64, 64, 2, 0), (idx, 1 << 31, 64, 64, 2, 152)):
        assert phx.phx_selftest_sgemm_schedule(*args, out) == phx.PHX_ERR_INVALID, args
    assert phx.phx_selftest_sgemm_schedule(idx, 64, 64, 64, 2, 152, None) == phx.PHX_ERR_INVALID
