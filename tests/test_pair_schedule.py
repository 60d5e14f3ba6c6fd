"""Work sharing of the BF16 paired-SM kernel, checked on the host through the
library's own schedule code (no GPU needed), for every schedule:

  * every k-slice of every output column of every tile is computed exactly
    once (whole tiles, 256 x 128 halves of a column-split last wave, or
    stream-K runs of k-slices);
  * tiles split along K are held by consecutive pairs in k order, and no
    two partial segments of one pair share a partial-sum slot;
  * each pair computes its stream-K range after its other units, and the
    work per pair is balanced.
"""
import collections

import pytest

from dense_gemm_07_gb300 import _abi

SCHEDULES = [_abi.SCHEDULE_AUTO, _abi.SCHEDULE_STREAM_K, _abi.SCHEDULE_COLUMN_SPLIT]


@pytest.fixture(scope="module")
def lib():
    return _abi.lib()


def tiles_of(M, N):
    return ((M + 255) // 256) * ((N + 255) // 256)


def all_units(M, N, K, P, sched):
    return {p: _abi.gemm_pair_units(M, N, K, P, p, sched) for p in range(P)}


CASES = [
    # (M, N, K, resident pairs)
    (4096, 4096, 4096, 76),     # 256 tiles: 3 whole waves + 28
    (8192, 8192, 8192, 76),     # 1024 tiles, 36 in the last wave
    (2048, 4096, 4096, 76),     # 128 tiles: one wave + 52
    (3001, 3000, 3000, 76),     # ragged edges, 144 tiles
    (1024, 1024, 4096, 76),     # 16 tiles: fewer tiles than pairs
    (512, 1024, 8192, 76),      # 8 tiles, long K
    (512, 512, 8192, 76),       # 4 tiles, long K
    (300, 700, 1000, 76),       # 6 tiles, 16 k-slices
    (1024, 4864, 512, 76),      # 76 tiles: exactly one wave
    (2560, 2304, 1024, 76),     # 90 tiles: one wave + 14
    (4096, 4096, 4096, 10),     # other resident counts
    (2560, 2304, 777, 7),
    (4096, 4096, 200, 76),      # 4 k-slices: too short to split along K
    (4096, 4096, 8192, 76),     # 3 whole waves, then 28 tiles halved along K
    (2560, 2048, 6200, 76),     # 1 whole wave, then 4 tiles halved (ragged K)
]


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("M,N,K,P", CASES)
def test_every_slice_exactly_once(lib, M, N, K, P, sched):
    nkb = (K + 63) // 64
    T = tiles_of(M, N)
    cover = collections.defaultdict(list)   # (tile, column half) -> k ranges
    for p, units in all_units(M, N, K, P, sched).items():
        for (tile, k0, k1, slot, qf, nseg, sk, n_off, width) in units:
            assert 0 <= tile < T
            assert 0 <= k0 < k1 <= nkb
            assert (n_off, width) in ((0, 256), (0, 128), (128, 128))
            for half in range(n_off // 128, (n_off + width) // 128):
                cover[(tile, half)].append((k0, k1, p))
    assert sorted(cover) == [(t, h) for t in range(T) for h in (0, 1)]
    for key, segs in cover.items():
        segs.sort()
        assert segs[0][0] == 0 and segs[-1][1] == nkb, (key, segs)
        for (a0, a1, _), (b0, b1, _) in zip(segs, segs[1:]):
            assert a1 == b0, (key, segs)


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("M,N,K,P", CASES)
def test_split_tiles_consecutive_pairs_and_slots(lib, M, N, K, P, sched):
    nkb = (K + 63) // 64
    T = tiles_of(M, N)
    by_tile = collections.defaultdict(list)
    for p, units in all_units(M, N, K, P, sched).items():
        slots = collections.Counter()
        for (tile, k0, k1, slot, qf, nseg, sk, n_off, width) in units:
            if k0 == 0 and k1 == nkb:
                assert (slot, qf, nseg) == (-1, p, 1)
                continue
            assert sk == 1 and (n_off, width) == (0, 256)
            assert slot in (0, 1)
            slots[slot] += 1
            by_tile[tile].append((k0, p, qf, nseg))
        assert all(c == 1 for c in slots.values()), (p, units)
    for tile, segs in by_tile.items():
        segs.sort()
        pairs = [p for (_, p, _, _) in segs]
        assert pairs == list(range(pairs[0], pairs[0] + len(pairs)))
        assert all(qf == pairs[0] and nseg == len(segs) for (_, _, qf, nseg) in segs)
        # each pair holds at least a tile's worth, or each tile is halved
        assert len(segs) == 2
    if sched == _abi.SCHEDULE_COLUMN_SPLIT:
        assert not by_tile


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("M,N,K,P", CASES)
def test_work_is_balanced(lib, M, N, K, P, sched):
    units = all_units(M, N, K, P, sched)
    T = tiles_of(M, N)
    sk_tiles = {u[0] for us in units.values() for u in us if u[6]}
    # the stream-K tiles are the last ones of the tile order
    if sk_tiles:
        assert sk_tiles == set(range(T - len(sk_tiles), T))
    sk_work = {}
    dp_cost = {}
    for p, us in units.items():
        flags = [u[6] for u in us]
        # each pair's stream-K range comes last, after its other units
        assert flags == sorted(flags), (p, us)
        sk_work[p] = sum(u[2] - u[1] for u in us if u[6])
        # in half-tile units of work
        dp_cost[p] = sum(u[8] // 128 for u in us if not u[6])
    busy = [w for w in sk_work.values() if w > 0]
    if busy:
        assert max(busy) - min(busy) <= 1, sk_work
    costs = [c for p, c in dp_cost.items() if units[p]]
    assert max(costs) - min(costs) <= 2


def _plan(M, N, K, c_addr=256):
    s, p = _abi.gemm_plan_bf16(M, N, K, 256, K, 256, N, c_addr, N)
    assert s == 0
    return (p.dp_tiles, p.sk_tiles, p.sk_pairs, p.pairs), p.workspace_bytes


def test_schedule_setting_and_plans(lib):
    prev = _abi.gemm_set_bf16_schedule(_abi.SCHEDULE_AUTO)
    try:
        # automatic: 3 whole waves, then each tile of the 28-tile last wave
        # of 4096^3 halved along K over 56 pairs (the halves are added in C)
        ws_4096 = 56 * 4 * 128 * 1024 + (28 * 8 + 56 * 16) * 8
        assert _plan(4096, 4096, 4096) == ((228, 28, 56, 76), ws_4096)
        # C not open to TMA stores: the halves would meet in the partial-sum
        # workspace, which costs more than the column split saves
        assert _plan(4096, 4096, 4096, c_addr=260) == ((256, 0, 0, 76), 0)
        assert _plan(2560, 2560, 4096, c_addr=260) == ((100, 0, 0, 76), 0)
        # few tiles and long K: on SM pairs each of the 20 tiles would be
        # halved along K; the automatic schedule runs 80 tiles of 128 x 128
        # there, and fewer (512 x 1024 x 8192: 32) on the narrow-N kernel
        sched, ws = _plan(1280, 1024, 4096)
        assert sched == (0, 20, 40, 40) and ws >= 40 * 4 * 128 * 1024
        assert _plan(512, 1024, 8192) == ((0, 0, 0, 0), 0)
        assert _plan(4096, 4096, 8192) == ((228, 28, 56, 76), ws_4096)
        assert _plan(5120, 5120, 4096)[0] == (380, 20, 40, 76)
        assert _plan(2560, 2560, 4096)[0] == (76, 24, 48, 76)
        assert _plan(8192, 8192, 8192)[0] == (988, 36, 72, 76)
        assert _plan(4096, 4096, 6144)[0] == (228, 28, 56, 76)
        # one whole wave, a last wave of 24 and 128 k-slices: every tile shared
        assert _plan(2560, 2560, 8192)[0] == (0, 100, 76, 76)
        assert _plan(2816, 2816, 6144)[0] == (0, 121, 76, 76)
        # one whole wave and a small last wave: every tile shared (stream-K)
        assert _plan(2560, 2048, 6200)[0] == (0, 80, 76, 76)
        assert _plan(2304, 2304, 8192)[0] == (0, 81, 76, 76)
        assert _plan(2560, 2048, 4096)[0] == (0, 80, 76, 76)
        # a last whole wave and a small partial one, but 32 k-slices: the
        # column split (48 k-slices: halved)
        assert _plan(4096, 4096, 2048)[0] == (256, 0, 0, 76)
        assert _plan(4096, 4096, 3072)[0] == (228, 28, 56, 76)
        # a last wave of 52 tiles is more than half the pairs: no split
        assert _plan(2048, 4096, 11008) == ((128, 0, 0, 76), 0)
        assert _plan(2048, 11008, 4096) == ((344, 0, 0, 76), 0)
        assert _abi.gemm_set_bf16_schedule(_abi.SCHEDULE_STREAM_K) == _abi.SCHEDULE_AUTO
        # stream-K: the last whole wave and the partial one are shared
        sched, ws = _plan(4096, 4096, 4096)
        assert sched == (152, 104, 76, 76)
        assert ws == 76 * 4 * 128 * 1024 + (104 * 8 + 76 * 16) * 8
        # one whole wave and 52 more tiles: all 128 are shared
        assert _plan(4096, 2048, 1024)[0] == (0, 128, 76, 76)
        assert _plan(2560, 2304, 1024)[0] == (0, 90, 76, 76)
        assert _abi.gemm_set_bf16_schedule(_abi.SCHEDULE_COLUMN_SPLIT) == _abi.SCHEDULE_STREAM_K
        assert _plan(512, 1024, 8192) == ((8, 0, 0, 16), 0)
        # a full last wave is never split
        for sched_ in SCHEDULES:
            _abi.gemm_set_bf16_schedule(sched_)
            assert _plan(1024, 4864, 512) == ((76, 0, 0, 76), 0)
        assert _abi.gemm_set_bf16_schedule(7) == -1
        assert _abi.gemm_set_bf16_schedule(-1) == -1
    finally:
        _abi.gemm_set_bf16_schedule(prev)


def test_pair_units_rejects_bad_arguments(lib):
    for args in [(-1, 4, 4, 76, 0), (4, 4, 0, 76, 0), (4, 4, 4, 0, 0),
                 (4, 4, 4, 76, 76), (4, 4, 4, 76, -1)]:
        with pytest.raises(ValueError):
            _abi.gemm_pair_units(*args)
    with pytest.raises(ValueError):
        _abi.gemm_pair_units(4, 4, 4, 76, 0, 3)
