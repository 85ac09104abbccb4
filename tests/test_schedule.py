"""Host checks of the persistent work list (no GPU): the job list that
gemm_schedule_jobs returns is the one the kernel walks, so these invariants
hold for every launch.

- every (tile, k-block) is computed by exactly one job;
- every tile is stored by exactly one job (FULL or OWNER);
- a split tile's OWNER holds its last k-block and its WRITERs hold the rest,
  on the units just below the owner (unit-1, unit-2, ...), which is where the
  kernel's owner looks for them;
- each unit writes at most one partial and runs its jobs in the order
  WRITER, whole stream-K tiles, OWNER, whole round-robin tiles;
- stream-K shares are balanced: unit k-block counts differ by at most one
  over the stream-K tiles, and the whole tiles are dealt evenly.
"""
from __future__ import annotations

import itertools

import pytest

import dense_tiled_gemm_gb300 as dtg

FULL, WRITER, OWNER = dtg.GEMM_JOB_FULL, dtg.GEMM_JOB_WRITER, dtg.GEMM_JOB_OWNER


def sk_tiles_for(T, U):
    return T if T < 2 * U else U + T % U


def check_schedule(T, U, KB, S):
    cover = {}
    stores = {}
    writers_of = {}
    owner_of = {}
    per_unit_sk = []
    for u in range(U):
        jobs = dtg.gemm_schedule_jobs(T, U, KB, S, u)
        kinds = [j[3] for j in jobs]
        assert kinds.count(WRITER) <= 1 and kinds.count(OWNER) <= 1
        if WRITER in kinds:
            assert kinds[0] == WRITER
        # phase of each job: 0 writer, 1 whole stream-K tile, 2 owner, 3 round-robin tile
        phase = [0 if k == WRITER else 2 if k == OWNER else 1 if t < S else 3
                 for (t, _, _, k) in jobs]
        assert phase == sorted(phase)
        sk_blocks = 0
        for tile, k0, k1, kind in jobs:
            assert 0 <= tile < T and 0 <= k0 < k1 <= KB
            for k in range(k0, k1):
                assert (tile, k) not in cover, f"k-block {(tile, k)} computed twice"
                cover[(tile, k)] = u
            if tile < S:
                sk_blocks += k1 - k0
            if kind == FULL:
                assert (k0, k1) == (0, KB)
            if kind in (FULL, OWNER):
                assert tile not in stores, f"tile {tile} stored twice"
                stores[tile] = u
            if kind == OWNER:
                assert k1 == KB and k0 > 0
                owner_of[tile] = u
            if kind == WRITER:
                assert k1 < KB
                writers_of.setdefault(tile, []).append(u)
            if tile >= S:
                assert kind == FULL and (tile - S) % U == u
        per_unit_sk.append(sk_blocks)
    assert len(cover) == T * KB
    assert sorted(stores) == list(range(T))
    for tile, ws in writers_of.items():
        o = owner_of[tile]
        # the writers are exactly the units below the owner, down to the one holding
        # k-block 0, that have stream-K work (a unit whose share is empty writes nothing)
        assert sorted(ws) == [v for v in range(min(ws), o) if per_unit_sk[v] > 0]
        assert cover[(tile, 0)] == min(ws)
    assert set(owner_of) == set(writers_of)
    if S:
        assert max(per_unit_sk) - min(per_unit_sk) <= 1


@pytest.mark.parametrize("T,U,KB", [(304, 76, 64), (240, 76, 17), (1024, 76, 64), (16, 76, 8),
                                    (64, 76, 16), (3, 8, 5), (7, 3, 1), (1, 5, 3), (100, 7, 9),
                                    (2640, 76, 48)])
def test_planner_split(T, U, KB):
    check_schedule(T, U, KB, sk_tiles_for(T, U))


def test_data_parallel_only():
    for T, U in ((304, 76), (5, 8), (17, 4)):
        check_schedule(T, U, 4, 0)


def test_small_exhaustive():
    for T, U, KB in itertools.product(range(1, 9), range(1, 7), range(1, 6)):
        for S in sorted({0, T, sk_tiles_for(T, U)} | ({T - (T // U) * U} if T >= U else set())):
            if S and (T - S) % U:
                continue
            check_schedule(T, U, KB, S)


def test_two_waves_cut_each_tile_once():
    # with at least one full wave in the stream-K part, no tile has two writers
    for T, U, KB in ((240, 76, 17), (1024, 76, 64), (100, 7, 9), (13, 4, 6)):
        S = sk_tiles_for(T, U)
        assert S >= U
        writers = {}
        for u in range(U):
            for tile, k0, k1, kind in dtg.gemm_schedule_jobs(T, U, KB, S, u):
                if kind == WRITER:
                    writers[tile] = writers.get(tile, 0) + 1
        assert all(n == 1 for n in writers.values())


def test_invalid_arguments():
    for args in ((0, 1, 1, 0, 0), (4, 0, 1, 0, 0), (4, 2, 1, 0, 2), (4, 2, 0, 0, 0), (4, 2, 1, 5, 0),
                 (4, 2, 1, -1, 0)):
        with pytest.raises(dtg.GemmError):
            dtg.gemm_schedule_jobs(*args)
