"""The work planner behind tgemm_run (tile shape, split-K, narrow tail),
through tgemm_plan: host logic only, so it runs without a GPU.

The expected plans are worked out by hand from the rules the planner states:
CTA pairs with 256 x 256 tiles whenever those tiles fill every SM pair once
(clusters of two pairs sharing B, 512 x 256 tiles on 4 CTAs, only on request);
the tiles of a last partial wave cut in k into 2-4 ranges of at least 16
k-blocks when those pieces fit one wave, else into column parts that still
fit one wave; split-K of every tile only for problems with under half a wave
of tiles.
"""
import itertools
import os

import pytest

import gemm_epilogue_02_gb300 as tg

SMS = 152   # SMs of the GB300


@pytest.fixture(autouse=True)
def _no_overrides(monkeypatch):
    for v in ("TGEMM_FORCE_CFG", "TGEMM_SPLIT_K", "TGEMM_TAIL_SPLIT", "TGEMM_GROUP_M"):
        monkeypatch.delenv(v, raising=False)


def test_square_4096_pairs_with_a_k_split_tail():
    # 16 x 16 = 256 tiles on 76 pairs: 3 whole waves; the 28 tiles left have
    # their 64 k-blocks cut into 2 ranges (56 pieces <= 76; 3 would not fit).
    p = tg.tgemm_plan(4096, 4096, 4096, SMS)
    assert (p["bn"], p["cg"], p["tiles"], p["groups"]) == (256, 2, 256, 76)
    assert (p["split_k"], p["split_first"], p["narrow_first"], p["narrow_parts"]) == (2, 228, 228, 1)
    assert p["units"] == 2 * 28 + 228


def test_square_4096_narrow_tail_on_request(monkeypatch):
    # TGEMM_TAIL_SPLIT=1: the 28 tiles are cut into two column parts instead.
    monkeypatch.setenv("TGEMM_TAIL_SPLIT", "1")
    p = tg.tgemm_plan(4096, 4096, 4096, SMS)
    assert (p["split_k"], p["narrow_first"], p["narrow_parts"]) == (1, 228, 2)
    assert p["units"] == 228 + 2 * 28


def test_square_4096_shared_b_clusters_on_request(monkeypatch):
    # TGEMM_FORCE_CFG=256x4: 8 x 16 = 128 tiles of 512 x 256 on 38 clusters of
    # 4 CTAs: 3 whole waves; the 14 tiles left have their 64 k-blocks cut into
    # 2 ranges (28 pieces <= 38; 3 would not fit).
    monkeypatch.setenv("TGEMM_FORCE_CFG", "256x4")
    p = tg.tgemm_plan(4096, 4096, 4096, SMS)
    assert (p["bn"], p["cg"], p["tiles"], p["groups"]) == (256, 4, 128, 38)
    assert (p["split_k"], p["split_first"], p["narrow_first"], p["narrow_parts"]) == (2, 114, 114, 1)
    assert p["units"] == 2 * 14 + 114


def test_square_8192():
    # 32 x 32 = 1024 tiles: 13 waves of 76 and 36 tiles in two k ranges (72 <= 76).
    p = tg.tgemm_plan(8192, 8192, 8192, SMS)
    assert (p["bn"], p["cg"], p["tiles"]) == (256, 2, 1024)
    assert (p["split_k"], p["split_first"], p["narrow_parts"], p["units"]) == (2, 988, 1, 72 + 988)


def test_tail_ranges_capped_by_k_and_four(monkeypatch):
    # 20 x 8 = 160 single-CTA tiles, 8 left over: 19 ranges would fit, at most
    # 4 are used; each range keeps 16 k-blocks, so K = 2048 (32 k-blocks) gives
    # 2, and K = 1024 gives one, so the 8 tiles are cut into column parts.
    monkeypatch.setenv("TGEMM_FORCE_CFG", "256")
    p = tg.tgemm_plan(2560, 2048, 4096, SMS)
    assert (p["tiles"], p["split_k"], p["split_first"], p["units"]) == (160, 4, 152, 152 + 32)
    p = tg.tgemm_plan(2560, 2048, 2048, SMS)
    assert (p["split_k"], p["split_first"], p["units"]) == (2, 152, 152 + 16)
    p = tg.tgemm_plan(2560, 2048, 1024, SMS)
    assert (p["split_k"], p["narrow_first"], p["narrow_parts"]) == (1, 152, 4)


def test_decode_shape_splits_k():
    # M = 128 fits one CTA row; 128-wide tiles: 32 tiles, k cut into 4 ranges.
    p = tg.tgemm_plan(128, 4096, 8192, SMS)
    assert (p["bn"], p["cg"], p["tiles"]) == (128, 1, 32)
    assert (p["split_k"], p["split_first"], p["narrow_parts"], p["units"]) == (4, 0, 1, 128)


def test_whole_waves_are_not_cut():
    p = tg.tgemm_plan(256 * 4, 256 * 19, 512, SMS)   # 4 x 19 = 76 pair tiles: one whole wave
    assert (p["bn"], p["cg"], p["tiles"], p["narrow_parts"], p["units"]) == (256, 2, 76, 1, 76)


def test_overrides(monkeypatch):
    monkeypatch.setenv("TGEMM_TAIL_SPLIT", "0")
    p = tg.tgemm_plan(4096, 4096, 4096, SMS)
    assert (p["narrow_parts"], p["narrow_first"], p["units"]) == (1, 256, 256)
    monkeypatch.delenv("TGEMM_TAIL_SPLIT")
    monkeypatch.setenv("TGEMM_FORCE_CFG", "256")
    p = tg.tgemm_plan(2560, 2048, 512, SMS)           # 20 x 8 = 160 tiles: 8 left over
    assert (p["bn"], p["cg"], p["tiles"], p["narrow_first"], p["narrow_parts"]) == (256, 1, 160, 152, 4)
    monkeypatch.setenv("TGEMM_SPLIT_K", "3")
    p = tg.tgemm_plan(2560, 2048, 512, SMS)
    assert (p["split_k"], p["split_first"], p["units"]) == (3, 0, 480)


def test_invalid_arguments():
    for args in ((0, 64, 64, SMS), (64, -1, 64, SMS), (64, 64, 0, SMS), (64, 64, 64, 1), (2 ** 31, 64, 64, SMS)):
        with pytest.raises(tg.TgemmError):
            tg.tgemm_plan(*args)


SIZES = [1, 100, 128, 129, 255, 256, 1000, 2048, 4095, 4096, 6143, 8191, 12288]


@pytest.mark.parametrize("sms", [148, 152])
def test_plan_invariants(sms):
    for M, N, K in itertools.product(SIZES, SIZES, (16, 520, 4096)):
        p = tg.tgemm_plan(M, N, K, sms)
        bn, cg = p["bn"], p["cg"]
        assert bn in (64, 128, 192, 224, 256) and cg in (1, 2, 4)
        assert cg < 4 or bn == 256
        assert p["tiles"] == -(-M // (128 * cg)) * -(-N // bn)
        gmax = sms // cg
        assert 1 <= p["groups"] <= min(p["units"], gmax)
        parts, nf, sf, sk = p["narrow_parts"], p["narrow_first"], p["split_first"], p["split_k"]
        assert 0 <= nf <= sf <= p["tiles"]
        split_units = (p["tiles"] - sf) * sk if sk > 1 else 0
        assert p["units"] == split_units + nf + (sf - nf) * parts
        if sk > 1 and sf == 0:            # few tiles: every tile's k loop is cut
            assert p["tiles"] * 2 <= gmax
            assert -(-(-(-K // 64)) // sk) >= 1
        elif sk > 1:                        # the last partial wave's tiles are cut in k
            assert p["tiles"] >= gmax and sf == p["tiles"] - p["tiles"] % gmax and nf == sf
            assert 2 <= sk <= 4 and (p["tiles"] - sf) * sk <= gmax
            assert (-(-K // 64)) // sk >= 16 and parts == 1
        if parts > 1:
            assert parts in (2, 4) and sk == 1
            assert (bn // min(cg, 2) // parts) % 64 == 0     # B columns per CTA of a pair
            assert sf - nf == p["tiles"] % gmax and p["tiles"] >= gmax
            assert (sf - nf) * parts <= gmax       # the cut tiles still fit one wave
