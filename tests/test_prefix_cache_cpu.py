"""Host bookkeeping of the prefix state cache (statecache.py, squad-0.8b,
StateCache: _bounds, _lookup, _evict), no GPU: the checkpoint schedule against
hand-worked cases and against its definition checked by brute force, the
longest-common-prefix lookup against a direct scan, and the LRU bounded in
MiB."""
import itertools

import numpy as np
import pytest

from gated_deltanet_recurrence_delta_gb300.prefix_cache import PrefixSchedule


def sched(**kw):
    return PrefixSchedule(ckpt_bytes=2**20, mb=kw.pop("mb", 64), **kw)


def test_bounds_hand_cases():
    s = sched(stride=2048, tail=16, align=64)
    # multiples of the stride below the state end, the end less the tail, the end
    assert s.bounds(0, 5000) == [2048, 4096, 4928, 4992]
    # the end less the tail rounds to the end itself: one position
    assert s.bounds(0, 100) == [64]
    # nothing above the restored position
    assert s.bounds(64, 100) == []
    assert s.bounds(4992, 5000) == []
    # restored at 2048: the stride multiple at 2048 is not above it
    assert s.bounds(2048, 5000) == [4096, 4928, 4992]
    # no stride: spans longer than the largest chunk (2048) get split points
    s0 = sched(stride=0, tail=16, align=64)
    assert s0.bounds(0, 9990) == [2048, 4096, 6144, 8192, 9920, 9984]
    assert s0.bounds(128, 4300) == [2176, 4224, 4288]
    # no tail
    st = sched(stride=1024, tail=0, align=64)
    assert st.bounds(0, 2100) == [1024, 2048]


def _definition(c, p, stride, tail, align, big=2048):
    """The schedule written from its definition: required positions, then the
    fewest split points (greedy, every largest-chunk step from the last one)."""
    down = lambda x: x - x % align
    e = down(p)
    req = set()
    if stride:
        req |= {k for k in range(stride, e, stride) if k > c}
    if tail and down(p - tail) > c:
        req.add(down(p - tail))
    if e > c:
        req.add(e)
    out, last = [], c
    for x in sorted(req):
        while x - last > big:
            last += big
            out.append(last)
        out.append(x)
        last = x
    return out


def test_bounds_properties_brute_force():
    rng = np.random.default_rng(3)
    for stride, tail in itertools.product((0, 256, 1024, 2048), (0, 16, 200)):
        s = sched(stride=stride, tail=tail, align=64)
        for _ in range(200):
            p = int(rng.integers(0, 9000))
            c = int(rng.integers(0, max(1, p // 64 + 1))) * 64
            b = s.bounds(c, p)
            assert b == _definition(c, p, stride, tail, 64)
            e = p - p % 64
            # ascending, above c, aligned, never past the state end, no span longer than 2048
            assert all(x % 64 == 0 and c < x <= e for x in b)
            assert b == sorted(set(b))
            assert all(y - x <= 2048 for x, y in zip([c] + b, b))
            if e > c:
                assert b[-1] == e


def test_stride_must_be_aligned():
    with pytest.raises(ValueError):
        sched(stride=1000, align=64)


def test_lookup_is_the_longest_common_prefix():
    s = sched(stride=128, tail=16, align=64)
    rng = np.random.default_rng(5)
    a = rng.integers(0, 50, 600)
    best, c0, pos = s.plan(a, 600)
    assert best is None and c0 == 0 and pos == s.bounds(0, 600)
    s.register(a, 600, pos, s.allocate(len(pos)), best, c0, 600)
    b = a.copy()
    b[300:] = rng.integers(50, 100, 300)  # shares 300 tokens
    usable = s.lookup(b[:576])
    assert sorted(c.pos for c in usable) == [p for p in pos if p <= 300]
    best, c0, pos_b = s.plan(b, 576)
    assert c0 == max(p for p in pos if p <= 300) == 256
    # a row with another first token shares nothing
    c = b.copy()
    c[0] = 99
    assert s.lookup(c[:500]) == []
    # the row itself again: its deepest checkpoint, nothing new to make
    best, c0, pos_a = s.plan(a, 600)
    assert c0 == 576 and pos_a == []


def test_lru_bounded_in_mib():
    # three checkpoints of 1 MiB fit in 3 MiB
    s = sched(mb=3, stride=64, tail=0, align=64)
    assert s.capacity == 3
    rows = [np.full(200, i) for i in range(3)]
    made = []
    for r in rows:
        best, c0, pos = s.plan(r, 128)
        slots = s.allocate(len(pos), keep=best)
        s.register(r, 128, pos, slots, best, c0, 128)
        made.append(list(zip(pos, slots)))
    # row 0 made [64, 128]; row 1's two pushed out row 0's oldest (64); row 2's
    # two pushed out row 0's 128 (its group goes with it) and row 1's 64
    assert s.bytes == 3 * 2**20 and len(s.ckpts) == 3 and len(s.groups) == 2
    assert s.stats["evicted"] == 3
    assert s.lookup(rows[0][:128]) == []
    assert [c.pos for c in s.lookup(rows[1][:128])] == [128]
    assert sorted(c.pos for c in s.lookup(rows[2][:128])) == [64, 128]
    # using row 1's checkpoint moves it to the back of the LRU order
    best, c0, pos = s.plan(rows[1], 128)
    assert c0 == 128 and pos == []
    s.register(rows[1], 128, pos, [], best, c0, 150)
    assert s.stats["hits"] == 1 and s.stats["tokens_reused"] == 128
    slots = s.allocate(2)
    assert id(best) in s.ckpts  # the recently used one survived; row 2's went
    assert len(slots) == 2 and s.stats["evicted"] == 5 and s.lookup(rows[2][:128]) == []
    with pytest.raises(ValueError):
        s.allocate(4)


def test_restore_source_is_never_evicted():
    s = sched(mb=2, stride=64, tail=0, align=64)
    r = np.arange(200)
    best, c0, pos = s.plan(r, 128)
    s.register(r, 128, pos, s.allocate(len(pos)), best, c0, 128)
    keep = max(s.lookup(r[:128]), key=lambda c: c.pos)
    keep_slot = keep.slot
    slots = s.allocate(1, keep=keep)
    assert id(keep) in s.ckpts and keep_slot not in slots
