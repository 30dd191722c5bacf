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
