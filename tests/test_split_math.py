"""The arithmetic two kernels rest on, checked on the CPU with the oracle's
offsets (no GPU): when the suffix products of two mixed radices over one
flat index lie on one divisibility chain, the offsets of a point split into
the offsets of its two digit groups.

* loop copy: the flat index of (thread t, slot s) under a loop layout is
  tflat(t) + sflat(s); when the loop's and the tile's radices nest,
  offset(tflat + sflat) = offset(tflat) + offset(sflat) on both sides;
* warp unit: lane + 32 j, when 32 lies on the chain of the unit's suffix
  products, has offsets offset(lane) + offset(32 j).
Random cases where the chain fails show that the split then fails too, so
the kernels' condition is needed, not only sufficient.
"""
import random

import numpy as np

from oracle import index_maps
from oracle.definition import Layout, paired_modes


def _offsets(modes, flat):
    idx = index_maps.unflatten(flat, [m[0] for m in modes])
    return (index_maps.project(idx, [m[1] for m in modes]), index_maps.project(idx, [m[2] for m in modes]))


def _chain(cuts):
    prev = 1
    for x in sorted(cuts):
        if x % prev:
            return False
        prev = x
    return True


def _suffixes(extents):
    out, c = [], 1
    for e in reversed(extents):
        if e == 1:
            continue
        c *= e
        out.append(c)
    return out


def _random_tile(rng):
    rank = rng.randint(1, 3)
    ext = [rng.choice([2, 3, 4, 6, 8]) for _ in range(rank)]
    order = list(range(rank))
    rng.shuffle(order)
    st, acc = [0] * rank, 1
    for m in reversed(order):
        st[m] = acc
        acc *= ext[m] + rng.choice([0, 0, 1])
    rm, acc = [0] * rank, 1
    for m in reversed(range(rank)):
        rm[m] = acc
        acc *= ext[m]
    return paired_modes(Layout(tuple(ext), tuple(rm)), Layout(tuple(ext), tuple(st)))


def _random_loop(rng, total):
    digits, rest = [], total
    for p in (2, 3, 5, 7):
        while rest % p == 0:
            digits.append(p)
            rest //= p
    rng.shuffle(digits)
    while len(digits) > 5:
        last = digits.pop()
        digits[rng.randrange(len(digits))] *= last
    loop, ts, ss = [None] * len(digits), 1, 1
    for k in rng.sample(range(len(digits)), len(digits)):
        if rng.random() < 0.5:
            loop[k], ts = (digits[k], ts, 0), ts * digits[k]
        else:
            loop[k], ss = (digits[k], 0, ss), ss * digits[k]
    return loop or [(1, 0, 0)]


def _parts(loop, flat):
    digits = index_maps.unflatten(flat, [m[0] for m in loop])
    weights, w = [], 1
    for e, _, _ in reversed(loop):
        weights.append(w)
        w *= e
    weights.reverse()
    t = sum(c * wt for c, wt, m in zip(digits, weights, loop) if m[1] > 0)
    s = sum(c * wt for c, wt, m in zip(digits, weights, loop) if m[2] > 0)
    return t, s


def test_loop_offsets_split_exactly_when_the_radices_nest():
    rng = random.Random(5)
    nested = not_nested = broke = 0
    for _ in range(300):
        modes = _random_tile(rng)
        total = int(np.prod([m[0] for m in modes]))
        loop = _random_loop(rng, total)
        chain = _chain(_suffixes([m[0] for m in loop]) + _suffixes([m[0] for m in modes]))
        splits = True
        for flat in range(total):
            t, s = _parts(loop, flat)
            assert t + s == flat
            a, b, c = _offsets(modes, flat), _offsets(modes, t), _offsets(modes, s)
            if a != (b[0] + c[0], b[1] + c[1]):
                splits = False
                break
        if chain:
            nested += 1
            assert splits, (modes, loop)
        else:
            not_nested += 1
            broke += not splits
    assert nested > 50 and not_nested > 20 and broke > 0


def test_warp_unit_offsets_split_exactly_when_32_nests():
    rng = random.Random(6)
    nested = not_nested = broke = 0
    for _ in range(300):
        rank = rng.randint(1, 3)
        ext = [rng.choice([2, 3, 4, 6, 8, 12, 16, 32, 48]) for _ in range(rank)]
        total = int(np.prod(ext))
        if total % 32 or total > 32 * 32:
            continue
        rm, acc = [0] * rank, 1
        for m in reversed(range(rank)):
            rm[m] = acc
            acc *= ext[m]
        order = list(range(rank))
        rng.shuffle(order)
        st, acc = [0] * rank, 1
        for m in reversed(order):
            st[m] = acc
            acc *= ext[m]
        extent, s_str, d_str, P = index_maps.permute_align(Layout(tuple(ext), tuple(rm)), Layout(tuple(ext), tuple(st)))
        modes = list(zip(extent, s_str, d_str))
        chain = _chain(_suffixes(list(extent)) + [32])
        splits = all(_offsets(modes, lane + 32 * j) ==
                     tuple(x + y for x, y in zip(_offsets(modes, lane), _offsets(modes, 32 * j)))
                     for lane in range(32) for j in range(P))
        if chain:
            nested += 1
            assert splits, modes
        else:
            not_nested += 1
            broke += not splits
    assert nested > 50 and not_nested > 5 and broke > 0


# ---------------------------------------------------------------------------
# the library's own decisions (lc_loop_plan, host only) against these facts
# ---------------------------------------------------------------------------

def _lib():
    import __graft_entry__
    __graft_entry__.build()
    import movement_primitives_gb300
    return movement_primitives_gb300


def test_loop_plan_decisions():
    M = _lib()
    L = lambda sh, st: dict(shape=sh, stride=st)
    got = M.loop_plan(L((32, 128, 128), (16384, 128, 1)), L((32, 128, 128), (128, 4096, 1)), 2,
                      [(64, 0, 8), (1024, 1, 0), (8, 0, 1)], 256)
    assert got == dict(num_threads=1024, slots_per_thread=512, points_per_tile=1 << 19, vec=8, split=1)
    got = M.loop_plan(L((3, 4), (4, 1)), L((3, 4), (1, 3)), 4, [(2, 1, 0), (6, 0, 1)], 2)
    assert (got["vec"], got["split"]) == (1, 0)  # suffix products 6 and 4 do not nest
    got = M.loop_plan(L((64, 128), (128, 1)), L((64, 128), (128, 1)), 4, [(16, 1, 0), (4, 0, 128), (128, 0, 1)], 2)
    assert (got["vec"], got["split"]) == (4, 1)
    got = M.loop_plan(L((8, 8), (8, 1)), L((8, 8), (1, 8)), 4, [(8, 0, 1), (8, 1, 0)])
    assert (got["vec"], got["split"]) == (1, 1)  # the innermost loop mode is a thread mode
    for n, split in [((1 << 31) - (1 << 14), 1), ((1 << 31) + (1 << 20), 0)]:  # the 2^31-byte cut-off
        got = M.loop_plan(L((n,), (1,)), L((n,), (1,)), 1, [(n >> 14, 0, 16), (1024, 1, 0), (16, 0, 1)], 2)
        assert (got["vec"], got["split"]) == (16, split)


def test_loop_plan_split_and_vectors_are_sound():
    """Random tiles and overrides: a split the library takes holds on the
    oracle's offsets, a nesting chain always gives one, and each vector of
    `vec` slots covers consecutive offsets on both sides."""
    M = _lib()
    rng = random.Random(9)
    splits = vectors = 0
    for _ in range(200):
        modes = _random_tile(rng)
        ext = tuple(m[0] for m in modes)
        src = dict(shape=ext, stride=tuple(m[1] for m in modes))
        dst = dict(shape=ext, stride=tuple(m[2] for m in modes))
        total = int(np.prod(ext))
        loop = _random_loop(rng, total)
        w = rng.choice([1, 2, 4])
        plan = M.loop_plan(src, dst, w, loop)
        if _chain(_suffixes([m[0] for m in loop]) + _suffixes(list(ext))):
            assert plan["split"] == 1, (modes, loop)
        if plan["split"]:
            splits += 1
            for flat in range(total):
                t, s = _parts(loop, flat)
                a, b, c = _offsets(modes, flat), _offsets(modes, t), _offsets(modes, s)
                assert a == (b[0] + c[0], b[1] + c[1]), (modes, loop, flat)
        v = plan["vec"]
        if v > 1:
            vectors += 1
            inner = next(m for m in reversed(loop) if m[0] > 1)
            assert inner[2] == 1 and inner[0] % v == 0, (loop, v)
            for flat in range(0, total, v):
                base = _offsets(modes, flat)
                for j in range(1, v):
                    assert _offsets(modes, flat + j) == (base[0] + j, base[1] + j), (modes, loop, v)
    assert splits > 50 and vectors > 10
