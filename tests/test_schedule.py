"""The persistent kernels' work schedule (WorkIter / ChainIter, the same integer code the GEMM
and chain kernels run), enumerated on the host through gemm_testing_schedule: every tile's
k-blocks are covered exactly once across the grid, split-K slices partition K, stream-K spans
are balanced, and every tile cut between two spans is started by one unit and ended by the
next, which publishes the flag slot the starter waits for.  No device needed."""
import collections

import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import build, gemm

TILE, EARLY, FINAL = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _all_pieces(chain, tiles_m, tiles_n, group_m, num_kb, splits, units, sk):
    tiles = tiles_m * (1 if chain else tiles_n)
    dp = (tiles // units - 1) * units if sk else 0
    out = {}
    for u in range(units):
        out[u] = gemm.gemm_testing_schedule(chain, tiles_m, tiles_n, group_m, num_kb, splits, dp, units if sk else 0,
                                            u, units)
    return out, dp


def _check(chain, tiles_m, tiles_n, group_m, num_kb, splits, units, sk):
    pieces, dp = _all_pieces(chain, tiles_m, tiles_n, group_m, num_kb, splits, units, sk)
    ntn = 1 if chain else tiles_n
    cover = collections.defaultdict(list)
    early, final = {}, {}
    for u, ps in pieces.items():
        for (tm, tn, kb0, kb1, role, slot) in ps:
            assert 0 <= tm < tiles_m and 0 <= tn < ntn and 0 <= kb0 < kb1 <= num_kb
            cover[(tm, tn)].append((kb0, kb1))
            if role == EARLY:
                assert kb0 > 0 and kb1 == num_kb and slot == u
                early[(tm, tn)] = u
            elif role == FINAL:
                assert kb0 == 0 and kb1 < num_kb and slot == u + 1
                final[(tm, tn)] = u
            else:
                assert role == TILE
        # stream-K: whole tiles first, then at most one piece that starts inside a tile (the
        # first of the span) and at most one that ends inside one (the last)
        roles = [p[4] for p in ps]
        assert roles.count(EARLY) <= 1 and roles.count(FINAL) <= 1
        if EARLY in roles:
            assert all(p[4] == TILE and p[2] == 0 and p[3] == num_kb for p in ps[:roles.index(EARLY)])
        if FINAL in roles:
            assert roles.index(FINAL) == len(roles) - 1
    # every tile once: its k-blocks partitioned by its pieces
    assert set(cover) == {(m, n) for m in range(tiles_m) for n in range(ntn)}
    for key, ranges in cover.items():
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == num_kb, key
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:])), (key, ranges)
        if not sk:
            assert len(ranges) == splits
            for s, (a, b) in enumerate(ranges):
                assert (a, b) == (s * num_kb // splits, (s + 1) * num_kb // splits)
        else:
            assert len(ranges) <= 2
    # a tile cut in two: started (FINAL) by unit u, ended (EARLY) by unit u + 1
    assert set(early) == set(final)
    for key in early:
        assert early[key] == final[key] + 1
    if sk:
        spans = [sum(p[3] - p[2] for p in ps[dp // units:]) for ps in pieces.values()]   # after the whole tiles
        total = (tiles_m * ntn - dp) * num_kb
        assert sum(spans) == total
        assert max(spans) - min(spans) <= 1
    return pieces


@pytest.mark.parametrize("tiles_m,tiles_n,group_m,num_kb,splits,units", [
    (32, 32, 12, 128, 1, 76),      # bf16 8192^3 pairs: 1024 tiles, 13.5 rounds
    (3, 2, 8, 33, 5, 152),         # few tiles, split-K slices
    (8, 3, 16, 9, 1, 152),         # fewer tiles than units
    (7, 11, 3, 17, 4, 19),         # ragged groups and slices
    (1, 1, 8, 1, 1, 1),
])
def test_gemm_schedule_covers_every_tile_once(tiles_m, tiles_n, group_m, num_kb, splits, units):
    pieces = _check(False, tiles_m, tiles_n, group_m, num_kb, splits, units, sk=False)
    # rasterisation: unit u takes work items u, u + units, ... of the (tile, K slice) list, the
    # slices of a tile consecutive, and the flat tile order visits group_m tile rows together,
    # column by column
    flat = []
    for t in range(tiles_m * tiles_n):
        g, r = divmod(t, group_m * tiles_n)
        first = g * group_m
        size = min(tiles_m - first, group_m)
        flat.append((first + r % size, r // size))
    for u, ps in pieces.items():
        want = [(*flat[w // splits], (w % splits) * num_kb // splits) for w in range(u, tiles_m * tiles_n * splits, units)]
        assert [(p[0], p[1], p[2]) for p in ps] == want


@pytest.mark.parametrize("tiles_m,tiles_n,group_m,num_kb,units", [
    (8, 10, 12, 64, 76),           # 80 pair tiles: every tile in a span
    (16, 11, 16, 65, 152),         # 176 single tiles: one whole round, then spans
    (9, 9, 4, 128, 19),            # four whole rounds, then spans
    (5, 7, 2, 3, 17),              # short K: spans of a few k-blocks, each at least one tile long
])
def test_gemm_stream_k_spans(tiles_m, tiles_n, group_m, num_kb, units):
    _check(False, tiles_m, tiles_n, group_m, num_kb, 1, units, sk=True)


@pytest.mark.parametrize("tiles,num_kb,units,sk", [
    (128, 64, 76, False),          # the chain workload in CTA pairs
    (128, 64, 76, True),
    (80, 16, 76, True),
    (176, 32, 76, True),           # one whole round, then spans
    (160, 16, 152, True),
    (3, 5, 8, False),
])
def test_chain_schedule(tiles, num_kb, units, sk):
    _check(True, tiles, 1, 1, num_kb, 1, units, sk)


def test_random_schedules():
    rng = np.random.default_rng(11)
    for _ in range(60):
        units = int(rng.integers(1, 160))
        tiles_m, tiles_n = int(rng.integers(1, 40)), int(rng.integers(1, 40))
        num_kb = int(rng.integers(1, 130))
        tiles = tiles_m * tiles_n
        sk = tiles > units and tiles % units != 0 and tiles < 4 * units and bool(rng.integers(2))
        splits = 1 if sk else int(rng.integers(1, min(num_kb, 8) + 1))
        _check(False, tiles_m, tiles_n, int(rng.integers(1, 20)), num_kb, splits, units, sk)
        chain_sk = tiles_m > units and tiles_m % units != 0 and tiles_m < 4 * units
        _check(True, tiles_m, 1, 1, num_kb, 1, units, chain_sk and bool(rng.integers(2)))


def test_schedule_rejects_bad_arguments():
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_testing_schedule(False, 4, 4, 8, 16, 1, 0, 0, 5, 5)        # unit outside the grid
    assert e.value.status == gemm.GEMM_ERR_INVALID_ARG
    with pytest.raises(gemm.GemmError):
        gemm.gemm_testing_schedule(False, 4, 4, 8, 16, 17, 0, 0, 0, 5)       # more slices than k-blocks
    with pytest.raises(gemm.GemmError):
        gemm.gemm_testing_schedule(False, 4, 4, 8, 16, 2, 0, 5, 0, 5)        # split-K with stream-K
    with pytest.raises(gemm.GemmError):
        gemm.gemm_testing_schedule(True, 10, 1, 1, 16, 1, 3, 5, 0, 5)        # whole tiles not whole rounds
