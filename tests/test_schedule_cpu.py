"""CPU checks of the tensor-core attend kernel's work schedule, replayed on the host by
the library itself (ll_debug_attend_schedule runs the same walker the kernel runs)."""

import collections

import pytest

from windowed_sink_attention_ll_b300 import build_lib

SHAPES = [
    # Lq,   La,    Lb,  heads, max_ctas
    (4680, 18720, 4680, 12, 148),   # Wan-shaped steady state: 228 items on 148 SMs
    (4680, 0, 4680, 12, 148),       # first chunk: no cache
    (4680, 14040, 4680, 12, 148),   # warm-up chunk
    (48, 144, 48, 2, 148),          # tiny: fewer items than SMs
    (300, 1200, 300, 2, 148),
    (4680, 18720, 4680, 12, 7),     # few CTAs: several whole rounds plus a tail
    (4680, 18720, 4680, 12, 1),     # one CTA does everything
    (37000, 5000, 37000, 3, 148),   # long items
    (4680, 37440, 4680, 12, 148),   # longest sweep window (S=3, W=18)
]


@pytest.fixture(scope="module")
def ll():
    build_lib.build()
    import windowed_sink_attention_ll_b300 as mod

    mod._lib()
    return mod


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_schedule_covers_every_key_tile_once(ll, shape):
    Lq, La, Lb, H, max_ctas = shape
    grid, pieces, splits = ll.ll_debug_attend_schedule(Lq, La, Lb, H, max_ctas)
    nqb = -(-Lq // 256)
    items = nqb * H
    nkv = -(-La // 128) + -(-Lb // 128)
    assert 1 <= grid <= min(max_ctas, items)
    seen = collections.Counter()
    per_cta = collections.Counter()
    part_slots = {}
    for cta, item, j0, j1, partial, slot in pieces:
        assert 0 <= cta < grid and 0 <= item < items and 0 <= j0 < j1 <= nkv
        for j in range(j0, j1):
            seen[(item, j)] += 1
        per_cta[cta] += j1 - j0
        assert partial == (0 if (j0 == 0 and j1 == nkv) else 1)
        if partial:
            assert slot in (2 * cta, 2 * cta + 1)
            assert slot not in part_slots, "two parts share a scratch slot"
            part_slots[slot] = item
    assert len(seen) == items * nkv and set(seen.values()) == {1}
    # split items and their parts agree with the pieces that wrote partial results
    split_items = {}
    for item, slots in splits:
        assert len(slots) >= 2
        split_items[item] = sorted(slots)
    by_item = collections.defaultdict(list)
    for slot, item in part_slots.items():
        by_item[item].append(slot)
    assert {i: sorted(s) for i, s in by_item.items()} == split_items
    # balance: whole rounds are equal; the tail differs by at most one run boundary
    if grid == max_ctas and items > grid:
        lo, hi = min(per_cta.values()), max(per_cta.values())
        assert hi - lo <= max(1, nkv // 16) + 1, (lo, hi)


def test_schedule_splits_only_leftover_items(ll):
    grid, pieces, splits = ll.ll_debug_attend_schedule(4680, 18720, 4680, 12, 148)
    assert grid == 148
    # 228 items: round 0 = items 0..147 whole, items 148..227 shared by all 148 CTAs
    whole = {p[1] for p in pieces if not p[4]}
    assert set(range(148)) <= whole
    assert all(item >= 148 for item, _ in splits)


PREFILL = [
    # Lq,    La,   block, heads, max_ctas
    (18720, 0, 4680, 12, 148),      # Wan-shaped switch: 12 frames in blocks of 3 frames, 888 items
    (18720, 0, 1560, 12, 148),      # frame-causal blocks
    (14040, 4680, 4680, 12, 148),   # keep-sink switch: 9 window frames after 3 cached sink frames
    (144, 0, 48, 2, 148),           # tiny: fewer items than SMs
    (300, 100, 100, 2, 3),          # few CTAs, a cached prefix with a ragged last tile
]


@pytest.mark.parametrize("shape", PREFILL, ids=[str(s) for s in PREFILL])
def test_prefill_schedule_covers_every_item_once_and_balances(ll, shape):
    Lq, La, block, H, max_ctas = shape
    grid, pieces, splits = ll.ll_debug_attend_schedule(Lq, La, Lq, H, max_ctas, mode=1, block_tokens=block)
    nqb = -(-Lq // 256)
    items = nqb * H
    assert grid == min(max_ctas, items) and splits == []
    seen = collections.Counter()
    load = collections.Counter()
    for cta, item, j0, j1, partial, slot in pieces:
        assert 0 <= cta < grid and 0 <= item < items and j0 == 0 and partial == 0
        qb = nqb - 1 - item // H                       # last query block first
        last_row = min(Lq, (qb + 1) * 256) - 1
        kv_end = min(Lq, (last_row // block + 1) * block)
        assert j1 == -(-La // 128) + -(-kv_end // 128)  # every cached tile + the fresh tiles it may see
        seen[item] += 1
        load[cta] += j1
    assert len(seen) == items and set(seen.values()) == {1}
    # zigzag rounds over items sorted longest first: no CTA carries much more than the mean
    if items > grid:
        mean = sum(load.values()) / grid
        longest = max(j for _, _, _, j, _, _ in pieces)
        assert max(load.values()) <= mean + longest


def _check_attend(grid, pieces, splits, Lq, La, Lb, H, max_ctas):
    nqb = -(-Lq // 256)
    items = nqb * H
    nkv = -(-La // 128) + -(-Lb // 128)
    assert grid == min(max_ctas, 256, items)
    seen = collections.Counter()
    load = collections.Counter()
    part_slots = {}
    for cta, item, j0, j1, partial, slot in pieces:
        assert 0 <= cta < grid and 0 <= item < items and 0 <= j0 < j1 <= nkv
        for j in range(j0, j1):
            seen[(item, j)] += 1
        load[cta] += j1 - j0
        assert partial == (0 if (j0 == 0 and j1 == nkv) else 1)
        if partial:
            assert slot in (2 * cta, 2 * cta + 1) and slot not in part_slots
            part_slots[slot] = item
    assert len(seen) == items * nkv and set(seen.values()) == {1}
    by_item = collections.defaultdict(list)
    for slot, item in part_slots.items():
        by_item[item].append(slot)
    assert {i: sorted(s) for i, s in by_item.items()} == {i: sorted(s) for i, s in splits}
    assert all(len(s) >= 2 for _, s in splits)
    # whole rounds first: every CTA carries rounds * nkv tiles before the tail
    rounds, rem = divmod(items, grid)
    tail = rem * nkv
    # the tail goes to as many CTAs as runs of at least 16 tiles allow (all of them when
    # the tail is long): those CTAs differ by at most one tile, the others carry no tail
    tail_ctas = max(1, min(grid, tail // 16)) if tail else 0
    loads = [load[c] for c in range(grid)]
    assert min(loads) >= rounds * nkv
    assert sum(loads) == items * nkv
    if tail_ctas == grid:
        assert max(loads) - min(loads) <= 1
    elif tail:
        assert max(loads) - min(loads) <= -(-tail // tail_ctas)


def test_random_attend_schedules():
    import numpy as np
    import windowed_sink_attention_ll_b300 as ll

    build_lib.build()
    rng = np.random.default_rng(7)
    for _ in range(300):
        Lq = int(rng.integers(1, 12000))
        La = int(rng.choice([0, int(rng.integers(1, 60000))]))
        H = int(rng.integers(1, 25))
        max_ctas = int(rng.choice([1, 2, 3, 7, 64, 148, 160, 300]))
        shape = (Lq, La, Lq, H, max_ctas)
        grid, pieces, splits = ll.ll_debug_attend_schedule(*shape)
        _check_attend(grid, pieces, splits, *shape)
        # the frame-causal chunk (mode 2) runs the attend schedule unchanged
        block = int(rng.integers(1, Lq + 1))
        assert ll.ll_debug_attend_schedule(*shape, mode=2, block_tokens=block) == (grid, pieces, splits), shape


def test_random_prefill_schedules():
    import numpy as np
    import windowed_sink_attention_ll_b300 as ll

    build_lib.build()
    rng = np.random.default_rng(11)
    for _ in range(200):
        Lq = int(rng.integers(1, 20000))
        La = int(rng.choice([0, int(rng.integers(1, 10000))]))
        block = int(rng.integers(1, Lq + 1))
        H = int(rng.integers(1, 25))
        max_ctas = int(rng.choice([1, 3, 64, 148, 300]))
        grid, pieces, splits = ll.ll_debug_attend_schedule(Lq, La, Lq, H, max_ctas, mode=1, block_tokens=block)
        nqb = -(-Lq // 256)
        items = nqb * H
        assert grid == min(max_ctas, items) and splits == []
        seen = collections.Counter()
        load = collections.Counter()
        for cta, item, j0, j1, partial, slot in pieces:
            assert 0 <= cta < grid and 0 <= item < items and j0 == 0 and partial == 0
            qb = nqb - 1 - item // H
            last_row = min(Lq, (qb + 1) * 256) - 1
            kv_end = min(Lq, (last_row // block + 1) * block)
            assert j1 == -(-La // 128) + -(-kv_end // 128), (Lq, La, block, H, max_ctas, item)
            seen[item] += 1
            load[cta] += j1
        assert len(seen) == items and set(seen.values()) == {1}
        if items > grid:
            mean = sum(load.values()) / grid
            longest = max(p[3] for p in pieces)
            assert max(load.values()) <= mean + longest
