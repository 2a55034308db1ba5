"""The persistent stream-K schedule, checked on the host (no GPU).

The stream-K kernel hands every CTA a sequence of segments (tile, K slices)
and, for tiles that several CTAs share, lets the last one to finish sum the
partial tiles from slots the others wrote.  Those index rules are restated
here from their definition and run for many plans the planner makes, so a
mistake in them -- a slice computed twice or never, two partials in one
slot, a ticket count that never completes -- shows up without a GPU.
"""
from __future__ import annotations

import itertools

import pytest

import dense_fp32_matrix_06_gb300 as sg
from dense_fp32_matrix_06_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sg.load_library()


def segments(g, G, dp_rounds, kt, U):
    """The (tile, k0, k1, first_run_segment) sequence CTA g works through."""
    out = []
    for r in range(dp_rounds):
        out.append((r * G + g, 0, kt, False))
    a, b = g * U // G, (g + 1) * U // G
    it = a
    while it < b:
        lt = it // kt
        k0 = it - lt * kt
        k1 = min(kt, k0 + (b - it))
        out.append((dp_rounds * G + lt, k0, k1, it == a))
        it += k1 - k0
    return out


def contributors(lt, G, kt, U):
    """First and last CTA of a shared tile, and the slot the first one used."""
    x0 = lt * kt
    g_first = ((x0 + 1) * G - 1) // U
    g_last = ((x0 + kt) * G - 1) // U
    slot0 = 2 * g_first + (0 if g_first * U // G == x0 else 1)
    return g_first, g_last, slot0


def check_schedule(tiles, kt, G, dp_rounds, U):
    dp_tiles = dp_rounds * G
    assert dp_tiles <= tiles and U == (tiles - dp_tiles) * kt
    if U:
        assert G <= U, "every run must be non-empty"
    covered = {}
    written = {}          # slot -> (tile, g)
    shared = {}           # tile -> list of CTAs that wrote a partial
    for g in range(G):
        for tile, k0, k1, first in segments(g, G, dp_rounds, kt, U):
            assert 0 <= tile < tiles and 0 <= k0 < k1 <= kt
            for k in range(k0, k1):
                assert (tile, k) not in covered, f"slice {k} of tile {tile} computed twice"
                covered[(tile, k)] = g
            if (k0, k1) != (0, kt):
                assert tile >= dp_tiles, "whole-K rounds never write partials"
                slot = 2 * g + (0 if first else 1)
                assert slot not in written, f"slot {slot} written twice"
                written[slot] = (tile, g)
                shared.setdefault(tile, []).append(g)
    assert len(covered) == tiles * kt, "some slice is never computed"
    for tile, gs in shared.items():
        lt = tile - dp_tiles
        g_first, g_last, slot0 = contributors(lt, G, kt, U)
        # the ticket target is g_last - g_first + 1: exactly the CTAs that wrote
        assert sorted(gs) == list(range(g_first, g_last + 1))
        # the reducer reads slot0, then 2h for the others: the slots they wrote
        assert written[slot0] == (tile, g_first)
        for h in range(g_first + 1, g_last + 1):
            assert written[2 * h] == (tile, h)
    return shared


@pytest.mark.parametrize("tiles,kt,G,dp", [
    (64, 64, 304, 0), (16, 32, 128, 0), (1, 7, 7, 0), (3, 5, 15, 0), (5, 1, 5, 0),
    (4096 - 12 * 304, 4, 304, 0), (997, 13, 304, 0), (7, 100, 97, 0),
    (700, 9, 304, 1), (2 * 304 + 17, 3, 304, 1), (10, 4, 40, 0),
])
def test_every_slice_once_and_every_partial_summed(tiles, kt, G, dp):
    U = (tiles - dp * G) * kt
    check_schedule(tiles, kt, G, dp, U)


def test_exhaustive_small_schedules():
    for tiles, kt in itertools.product(range(1, 9), range(1, 9)):
        for G in range(1, tiles * kt + 1):
            check_schedule(tiles, kt, G, 0, tiles * kt)


SHAPES = [
    (256, 256, 256), (1024, 1024, 1024), (1023, 777, 513), (1024, 2304, 768),
    (1024, 3072, 768), (1024, 768, 3072), (2048, 2048, 2048), (8192, 8192, 64),
    (1024, 1024, 16384), (4096, 4096, 4096), (1, 1, 1), (3, 5000, 7), (5000, 3, 20000),
    (129, 129, 129), (64, 64, 8192), (300, 4000, 33),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("min_slices", [None, 1, 3])
def test_planner_stream_k_plans_are_consistent(lib, tune, M, N, K, tile, min_slices):
    tune(schedule=1, tile=tile, sk_min_slices=min_slices)
    p = sg.gemm_plan_for_sms(M, N, K, K, N, N, sm_count=152)
    assert p.schedule == 1 and p.bm == tile
    # with A transposed first both operands are direct copies: K slices of
    # T/4 in three pages; otherwise K slices of T/8 in four
    if p.transpose_a:
        assert tile == 128 and p.bk == 32 and p.stages == 3
    else:
        assert p.bk == tile // 8 and p.stages == 4
    assert p.split_k == 1 and p.tail_split == 1
    # unchecked tiles only for whole tiles on the direct-copy kernel
    full = M % 128 == 0 and N % 128 == 0 and K % 32 == 0
    assert p.edge == (0 if (p.transpose_a and full) else 1)
    tiles = p.tiles_m * p.tiles_n
    kt = -(-K // p.bk)
    G = p.grid_ctas
    assert 1 <= G <= 152 * (8 if tile == 64 else 2)
    U = p.sk_iters
    sk_tiles = tiles - p.dp_rounds * G
    assert U == sk_tiles * kt
    parts = 2 * G * tile * tile * 4 if U else 0
    if U:
        assert sk_tiles <= 4096 and G <= sk_tiles * 16
    if p.transpose_a:
        at = (K * p.a_t_ld * 4 + 255) // 256 * 256
        assert p.a_t_ld == (M + 3) // 4 * 4
        assert p.workspace_bytes == 16384 + parts + at
    else:
        assert p.workspace_bytes == (16384 + parts if U else 0)
    if tiles * kt <= 200_000:
        check_schedule(tiles, kt, G, p.dp_rounds, U)


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (1024, 1024, 16384), (300, 4000, 36)])
def test_planner_stream_k_with_transposed_a(lib, tune, M, N, K):
    tune(schedule=1, tile=128, transpose_a=1)
    p = sg.gemm_plan_for_sms(M, N, K, K, N, N, sm_count=152)
    assert p.transpose_a == 1 and p.bk == 32 and p.stages == 3
    tiles = p.tiles_m * p.tiles_n
    check_schedule(tiles, -(-K // 32), p.grid_ctas, p.dp_rounds, p.sk_iters)


def test_planner_fills_whole_waves_before_stream_k(lib, tune):
    tune(schedule=1, tile=128, transpose_a=0)
    # 4096 tiles over 304 resident CTAs: 12 whole-K rounds, then 448 tiles
    p = sg.gemm_plan_for_sms(8192, 8192, 64, 64, 8192, 8192, sm_count=152)
    assert p.grid_ctas == 304 and p.dp_rounds == 12
    assert p.sk_iters == (4096 - 12 * 304) * 4
    # a grid of whole waves needs no stream-K part at all
    q = sg.gemm_plan_for_sms(128 * 16, 128 * 38, 512, 512, 128 * 38, 128 * 38, sm_count=152)
    assert q.tiles_m * q.tiles_n == 2 * 304 and q.dp_rounds == 2 and q.sk_iters == 0
    assert q.workspace_bytes == 0
