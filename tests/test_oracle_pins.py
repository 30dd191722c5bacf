"""Pins the oracle to what the pages and the mathematics fix (no GPU).

Each check below compares the oracle with something other than itself:
values the pages print (tests/golden/), closed forms worked out by hand,
library routines (numpy strided copies and transposes, memcpy), invariants
(bijection) and brute force over tiny layouts.  ``test_planted_mistakes``
then plants plausible mistakes in the oracle and checks that some pin fails.
"""
import itertools
import os
import random

import numpy as np
import pytest

import oracle
from oracle import banks, definition, index_maps
from oracle.definition import Layout

from conftest import GOLDEN

WORD_DTYPES = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64, 16: np.dtype("V16")}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _read_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]


def _numpy_strided_copy(src_bytes, src_l, dst_bytes, dst_l, w, n_tiles):
    """numpy's own strided assignment, one view per tile (independent of the oracle)."""
    dt = WORD_DTYPES[w]
    sw = src_bytes.view(dt)
    dw = dst_bytes.view(dt)
    s_nu = [(e, s) for e, s in zip(src_l.shape, src_l.stride) if e != 1]
    d_nu = [(e, s) for e, s in zip(dst_l.shape, dst_l.stride) if e != 1]
    shape = [e for e, _ in s_nu]
    isz = sw.itemsize
    s_span = 1 + sum((e - 1) * s for e, s in zip(src_l.shape, src_l.stride))
    d_span = 1 + sum((e - 1) * s for e, s in zip(dst_l.shape, dst_l.stride))
    sts = src_l.tile_stride or s_span
    dts = dst_l.tile_stride or d_span
    for t in range(n_tiles):
        sb = src_l.offset + t * sts
        db = dst_l.offset + t * dts
        sv = np.lib.stride_tricks.as_strided(sw[sb:], shape, [s * isz for _, s in s_nu])
        dv = np.lib.stride_tricks.as_strided(dw[db:], shape, [s * isz for _, s in d_nu])
        dv[...] = sv


def _dense_strides(extents, order, gaps=None):
    """Packed strides with mode order[-1] innermost; optional per-mode gap factors."""
    strides = [0] * len(extents)
    acc = 1
    for pos, m in enumerate(reversed(order)):
        acc *= (gaps[pos] if gaps else 1)
        strides[m] = acc
        acc *= extents[m]
    return tuple(strides)


def _tiny_layout_pairs(seed=0, count=300):
    """Random valid (injective-destination) tiny layout pairs, rank <= 3, extents <= 4."""
    rng = random.Random(seed)
    out = []
    for _ in range(count):
        rank = rng.randint(1, 3)
        ext = tuple(rng.randint(1, 4) for _ in range(rank))
        so = list(range(rank)); rng.shuffle(so)
        do = list(range(rank)); rng.shuffle(do)
        sg = [rng.choice([1, 1, 2, 3]) for _ in range(rank)]
        dg = [rng.choice([1, 1, 2]) for _ in range(rank)]
        src = Layout(ext, _dense_strides(ext, so, sg), rng.randint(0, 5), 0)
        dst = Layout(ext, _dense_strides(ext, do, dg), rng.randint(0, 5), 0)
        if rng.random() < 0.2:  # broadcast source mode
            st = list(src.stride); st[rng.randrange(rank)] = 0
            src = src._replace(stride=tuple(st))
        n_tiles = rng.randint(1, 3)
        out.append((src, dst, rng.choice([1, 2, 4, 8, 16]), n_tiles))
    return out


def _buffers(src_l, dst_l, w, n_tiles, seed):
    rng = np.random.default_rng(seed)
    ns = (src_l.offset + (n_tiles - 1) * (src_l.tile_stride or oracle.cosize(src_l))
          + oracle.cosize(src_l)) * w
    nd = (dst_l.offset + (n_tiles - 1) * (dst_l.tile_stride or oracle.cosize(dst_l))
          + oracle.cosize(dst_l)) * w
    src = rng.integers(0, 256, size=max(ns, 16), dtype=np.uint8)
    dst = np.full(max(nd, 16), 0xA5, dtype=np.uint8)
    return src, dst


# ---------------------------------------------------------------------------
# O4: the definition against library routines
# ---------------------------------------------------------------------------

def check_definition_vs_numpy(pairs=None):
    for i, (src_l, dst_l, w, n_tiles) in enumerate(pairs or _tiny_layout_pairs()):
        src, dst = _buffers(src_l, dst_l, w, n_tiles, i)
        want = dst.copy()
        _numpy_strided_copy(src, src_l, want, dst_l, w, n_tiles)
        got = dst.copy()
        oracle.copy(src, src_l, got, dst_l, w, n_tiles)
        assert np.array_equal(got, want), (src_l, dst_l, w, n_tiles)


def test_definition_matches_numpy_strided_copy():
    check_definition_vs_numpy()


def check_transpose_vs_numpy(shapes=((32, 32), (7, 13), (64, 48)), ws=(1, 2, 4, 8, 16)):
    for (r, c), w in itertools.product(shapes, ws):
        dt = WORD_DTYPES[w]
        rng = np.random.default_rng(r * 100 + c + w)
        a = rng.integers(0, 256, size=r * c * w, dtype=np.uint8)
        out = np.zeros_like(a)
        oracle.copy(a, Layout((r, c), (c, 1)), out, Layout((r, c), (1, r)), w)
        want = np.ascontiguousarray(a.view(dt).reshape(r, c).T).view(np.uint8).reshape(-1)
        assert np.array_equal(out, want), (r, c, w)


def test_transpose_matches_numpy_transpose():
    check_transpose_vs_numpy()


def test_identity_is_memcpy():
    rng = np.random.default_rng(7)
    for n, w in [(1, 1), (1000, 2), (4096, 4), (333, 16)]:
        a = rng.integers(0, 256, size=n * w, dtype=np.uint8)
        out = np.zeros_like(a)
        oracle.copy(a, Layout((n,), (1,)), out, Layout((n,), (1,)), w)
        assert out.tobytes() == a.tobytes()


def check_axis_permute_vs_numpy():
    # the (0,2,1,3) head/sequence swap, scaled down
    b, h, s, d = 2, 4, 8, 16
    rng = np.random.default_rng(5)
    x = rng.standard_normal((b, h, s, d)).astype(np.float32)
    src = x.reshape(-1).view(np.uint8)
    out = np.zeros_like(src)
    oracle.copy(src, Layout((b, h, s, d), (h * s * d, s * d, d, 1)), out,
                Layout((b, h, s, d), (h * s * d, d, h * d, 1)), 4)
    want = np.ascontiguousarray(x.transpose(0, 2, 1, 3)).reshape(-1).view(np.uint8)
    assert np.array_equal(out, want)


def test_axis_permute_matches_numpy():
    check_axis_permute_vs_numpy()


def test_untouched_bytes_and_bijection():
    """Each destination offset in the image is written once; the rest stay 0xA5."""
    for i, (src_l, dst_l, w, n_tiles) in enumerate(_tiny_layout_pairs(seed=3, count=120)):
        if 0 in src_l.stride:
            continue
        # source words carry distinct ids so that a double write would show
        n = definition.logical_size(src_l, dst_l, n_tiles)
        pts = np.arange(n)
        so, do = oracle.offsets_of(src_l, dst_l, n_tiles, pts)
        assert len(set(do.tolist())) == n  # injective destination
        src = np.zeros((int(so.max()) + 1) * 4, dtype=np.uint8)
        src.view(np.uint32)[so] = pts.astype(np.uint32) + 1
        dst = np.zeros((int(do.max()) + 1) * 4, dtype=np.uint8)
        oracle.copy(src, src_l, dst, dst_l, 4, n_tiles)
        vals = dst.view(np.uint32)
        written = vals[vals != 0]
        assert sorted(written.tolist()) == list(range(1, n + 1))
        assert np.array_equal(vals[do], pts.astype(np.uint32) + 1)


# ---------------------------------------------------------------------------
# "copy -> gmem_smem": the [outer, threads, vec] partition
# ---------------------------------------------------------------------------

def check_gmem_smem_table():
    rows = [ln.split() for ln in _read_golden("gmem_smem_partition.txt")]
    for row in rows:
        if row[0] != "dtype":
            continue
        _, name, w, vec, copy_bytes, outer = row
        w, vec, copy_bytes, outer = int(w), int(vec), int(copy_bytes), int(outer)
        part = index_maps.gmem_smem_partition((32, 32), (32, 1), (32, 1), w, 32)
        assert (part["vec"], part["vec"] * w, part["outer"]) == (vec, copy_bytes, outer), name
    ir = {row[1]: " ".join(row[2:]) for row in rows if row[0] == "ir"}
    part = index_maps.gmem_smem_partition((32, 32), (32, 1), (32, 1), 4, 32)
    seen = set()
    for f, tid, g_lin, s_lin, elems in index_maps.gmem_smem_replay(part, 32):
        env = {"f": f, "tid": tid}
        assert s_lin == eval(ir["s_lin"], {}, env)
        assert g_lin == eval(ir["g_lin"], {}, env)
        seen.update(g for g, _ in elems)
    assert seen == set(range(1024))


def test_gmem_smem_partition_matches_page():
    check_gmem_smem_table()


def check_gmem_smem_alignment_rule():
    # "both base offsets" must be multiples of vec: an 8-byte (2-float) base
    # offset rules out 16-byte vectors, leaving 64-bit ones (worked by hand).
    part = index_maps.gmem_smem_partition((32, 32), (32, 1), (32, 1), 4, 32, g_offset=2)
    assert (part["vec"], part["outer"]) == (2, 16)
    # a shared side that is transposed has no common contiguous tail: scalar copies
    part = index_maps.gmem_smem_partition((32, 32), (1, 32), (32, 1), 4, 32)
    assert part["vec"] == 1 and part["outer"] == 32
    # element count not a multiple of the thread count: the variant declines
    with pytest.raises(index_maps.Decline):
        index_maps.gmem_smem_partition((3, 7), (7, 1), (7, 1), 4, 32)


def check_gmem_smem_guarded():
    """Guarded partitions ("loop_mapping.py": counts below the thread count
    leave threads idle behind a guard), worked out by hand."""
    # 64 fp32 words, 128 threads: 16-byte vectors, one round, threads 0..15
    part = index_maps.gmem_smem_partition_guarded((64,), (1,), (1,), 4, 128)
    assert (part["vec"], part["outer"], part["total"], part["guarded"]) == (4, 1, 64, True)
    moved = {tid: [g for g, _ in el] for _f, tid, _g, _s, el in index_maps.gmem_smem_replay(part, 128)}
    assert sorted(moved) == list(range(16))
    assert all(moved[t] == [4 * t + v for v in range(4)] for t in range(16))
    # 64 eight-byte words, 128 threads: vectors of 2 words, threads 0..31
    part = index_maps.gmem_smem_partition_guarded((64,), (1,), (1,), 8, 128)
    assert (part["vec"], part["outer"]) == (2, 1)
    assert sorted({tid for _f, tid, _g, _s, _e in index_maps.gmem_smem_replay(part, 128)}) == list(range(32))
    # 100 fp32 words, 8 threads: vec 4, 25 vectors, rounds of 8: 4 rounds, the
    # last one with thread 0 alone (vector 24 = words 96..99)
    part = index_maps.gmem_smem_partition_guarded((100,), (1,), (1,), 4, 8)
    assert (part["vec"], part["outer"], part["guarded"]) == (4, 4, True)
    last = [(tid, g) for f, tid, g, _s, _e in index_maps.gmem_smem_replay(part, 8) if f == 3]
    assert last == [(0, 96)]
    # a 4-byte swizzle chunk caps the vector at one fp32 word
    part = index_maps.gmem_smem_partition_guarded((32, 32), (32, 1), (32, 1), 4, 32, chunk_bytes=4)
    assert (part["vec"], part["outer"], part["guarded"]) == (1, 32, False)
    part = index_maps.gmem_smem_partition_guarded((32, 32), (32, 1), (32, 1), 4, 32, chunk_bytes=16)
    assert part["vec"] == 4
    with pytest.raises(index_maps.Decline):
        index_maps.gmem_smem_partition_guarded((8,), (1,), (1,), 16, 32, chunk_bytes=8)


def test_gmem_smem_guarded_partition():
    check_gmem_smem_guarded()


def test_gmem_smem_guarded_agrees_with_the_page_where_exact():
    """Where the page's partition accepts (the count divides), the guarded one
    is the same partition (the dtype table of "copy -> gmem_smem" included)."""
    rng = np.random.default_rng(11)
    for _ in range(300):
        rank = int(rng.integers(1, 4))
        ext = [int(rng.choice([1, 2, 4, 8, 16, 3])) for _ in range(rank)]
        gs = list(np.cumprod([1] + ext[::-1][:-1])[::-1])
        ss = list(gs)
        if rng.random() < 0.5:
            perm = rng.permutation(rank)
            pe = [ext[i] for i in perm]
            st = list(np.cumprod([1] + pe[::-1][:-1])[::-1])
            ss = [0] * rank
            for k, i in enumerate(perm):
                ss[i] = st[k]
        w = int(rng.choice([1, 2, 4, 8, 16]))
        threads = int(rng.choice([1, 4, 8, 32]))
        try:
            exact = index_maps.gmem_smem_partition(ext, gs, ss, w, threads)
        except index_maps.Decline:
            continue
        guarded = index_maps.gmem_smem_partition_guarded(ext, gs, ss, w, threads)
        if exact["total"] % (threads * guarded["vec"]) == 0:
            assert (guarded["vec"], guarded["outer"], guarded["guarded"]) == (exact["vec"], exact["outer"], False)
            assert guarded["modes"] == exact["modes"]


def test_gmem_smem_guarded_replay_is_the_definition():
    """Brute force on small shapes with counts off the thread grid: the
    guarded replay moves every element exactly once, as the definition does."""
    rng = np.random.default_rng(12)
    for _ in range(200):
        rank = int(rng.integers(1, 4))
        ext = [int(rng.choice([1, 2, 3, 5, 7, 8])) for _ in range(rank)]
        gs = [int(x) for x in np.cumprod([1] + ext[::-1][:-1])[::-1]]
        perm = rng.permutation(rank)
        pe = [ext[i] for i in perm]
        st = [int(x) for x in np.cumprod([1] + pe[::-1][:-1])[::-1]]
        ss = [0] * rank
        for k, i in enumerate(perm):
            ss[i] = st[k]
        w = int(rng.choice([1, 2, 4, 8]))
        threads = int(rng.choice([8, 32, 128]))
        part = index_maps.gmem_smem_partition_guarded(ext, gs, ss, w, threads)
        seen = [s for _f, _t, _g, _s, el in index_maps.gmem_smem_replay(part, threads) for _gg, s in el]
        assert sorted(seen) == list(range(int(np.prod(ext))))
        total = int(np.prod(ext))
        src = rng.integers(0, 2 ** 31, total, dtype=np.int64).tolist()
        got = [None] * total
        index_maps.gmem_smem_copy(src, got, part, threads, g_is_src=True)
        want = np.empty(total * 8, np.uint8)
        definition.copy(np.asarray(src, np.int64).view(np.uint8), Layout(tuple(ext), tuple(gs)), want,
                        Layout(tuple(ext), tuple(ss)), 8)
        assert got == want.view(np.int64).tolist()


def check_xor_swizzle():
    """The shared-memory XOR swizzle: a bijection that keeps every chunk's
    bytes together and in order; the 128-byte form puts chunk c of row r at
    chunk c ^ (r % 8)."""
    for bits, c, r, span in [(3, 4, 7, 4096), (2, 2, 8, 2048), (5, 2, 7, 8192), (0, 4, 7, 1024), (1, 3, 4, 256)]:
        image = [index_maps.xor_swizzle(o, bits, c, r) for o in range(span)]
        assert sorted(image) == list(range(span))
        for o in range(0, span, 1 << c):
            assert image[o:o + (1 << c)] == list(range(image[o], image[o] + (1 << c)))
        if bits == 0:
            assert image == list(range(span))
    for row in range(16):
        for chunk in range(8):
            o = row * 128 + chunk * 16 + 5
            assert index_maps.xor_swizzle(o, 3, 4, 7) == row * 128 + (chunk ^ (row % 8)) * 16 + 5


def test_xor_swizzle():
    check_xor_swizzle()


def test_gmem_smem_alignment_rule():
    check_gmem_smem_alignment_rule()


def check_round_trip_identity():
    """The page's demonstration program: global -> shared -> global is the identity."""
    rng = np.random.default_rng(1)
    a = list(rng.uniform(-1, 1, 1024).astype(np.float32).view(np.uint32))
    smem = [None] * 1024
    b = [None] * 1024
    part = index_maps.gmem_smem_partition((32, 32), (32, 1), (32, 1), 4, 32)
    index_maps.gmem_smem_copy(a, smem, part, 32, g_is_src=True)
    index_maps.gmem_smem_copy(smem, b, part, 32, g_is_src=False)
    assert b == a


def test_round_trip_identity():
    check_round_trip_identity()


def test_gmem_smem_replay_matches_definition():
    """The replayed loop moves exactly what the definition moves, for tiny layouts."""
    rng = random.Random(11)
    for _ in range(60):
        rank = rng.randint(1, 3)
        ext = tuple(rng.choice([1, 2, 4, 8]) for _ in range(rank))
        total = int(np.prod(ext))
        threads = rng.choice([t for t in (1, 2, 4, 8, 16, 32) if total % t == 0])
        g_ord = list(range(rank)); rng.shuffle(g_ord)
        s_ord = list(range(rank)); rng.shuffle(s_ord)
        gs, ss = _dense_strides(ext, g_ord), _dense_strides(ext, s_ord)
        w = rng.choice([1, 2, 4])
        part = index_maps.gmem_smem_partition(ext, gs, ss, w, threads)
        src = list(range(1000, 1000 + total))
        got = [None] * total
        index_maps.gmem_smem_copy(src, got, part, threads, g_is_src=True)
        sb = np.array(src, dtype=np.uint32).view(np.uint8)
        want = np.zeros(total * 4, dtype=np.uint8)
        oracle.copy(sb, Layout(ext, gs), want, Layout(ext, ss), 4)
        assert got == want.view(np.uint32).tolist()


# ---------------------------------------------------------------------------
# TileLang default loop partition
# ---------------------------------------------------------------------------

def _parse_points(text):
    return [tuple(int(v) for v in p.strip("()").split(",") if v != "")
            for p in text.split()]


def check_loop_mapping_tables(plan_fn=None):
    for line in _read_golden("loop_mapping_t8_v2.txt"):
        ext_s, used, per, t0, t1 = [c.strip() for c in line.split("|")]
        extents = tuple(int(v) for v in ext_s.strip("()").split(",") if v.strip())
        pm = (plan_fn or index_maps.plan)(extents, 8, 2)
        assert len({t for t, _ in pm.values()}) == int(used)
        owned = {}
        for idx in sorted(pm, key=lambda i: index_maps.flatten(i, extents)):
            owned.setdefault(pm[idx][0], []).append(idx)
        assert all(len(v) == int(per) for v in owned.values())
        assert owned[0][:4] == _parse_points(t0)
        assert owned[1][:4] == _parse_points(t1)


def test_loop_mapping_tables_match_page():
    check_loop_mapping_tables()


def test_loop_mapping_levels():
    """lane -> thread -> serial replication, checked on the docstring's CLI examples."""
    for extents, T, V in [((128, 32), 128, 8), ((128, 32), 128, 4), ((64,), 128, 2)]:
        pm = index_maps.plan(extents, T, V)
        total = int(np.prod(extents))
        slots = set(pm.values())
        assert len(slots) == total  # (thread, slot) is a bijection
        for idx, (t, s) in pm.items():
            flat = index_maps.flatten(idx, extents)
            # consecutive vector_size iterations share a thread and consecutive slots
            if flat % V:
                prev = pm[index_maps.unflatten(flat - 1, extents)]
                assert prev == (t, s - 1)
        # fewer points than threads: some threads get nothing (the page's guard case)
        if total < T * V:
            assert len({t for t, _ in pm.values()}) < T


# ---------------------------------------------------------------------------
# loop_layout= override (reading: modes (extent, thread_stride, slot_stride)
# over the row-major flat index of the nest, an exact partition)
# ---------------------------------------------------------------------------

def _override_plan(extents, T, V):
    total = int(np.prod(extents))
    return index_maps.loop_layout_plan(extents, index_maps.default_loop_layout(total, T, V))


def check_default_override_tables():
    """The default plan written as an override reproduces the page's tables."""
    check_loop_mapping_tables(_override_plan)


def test_default_override_matches_page_tables():
    check_default_override_tables()


def check_override_hand_worked():
    """Three overrides whose owners were worked out by hand."""
    # blocked: thread t owns the 8 consecutive points 8t .. 8t + 7, in order
    pm = index_maps.loop_layout_plan((64,), [(8, 1, 0), (8, 0, 1)])
    assert [p for p in sorted(pm) if pm[p][0] == 0] == [(i,) for i in range(8)]
    assert [p for p in sorted(pm, key=lambda q: pm[q][1]) if pm[p][0] == 1] == [(i,) for i in range(8, 16)]
    # column per thread: point (i, j) goes to thread j, slot i
    pm = index_maps.loop_layout_plan((8, 8), [(8, 0, 1), (8, 1, 0)])
    assert pm[(0, 3)] == (3, 0) and pm[(5, 3)] == (3, 5) and pm[(7, 0)] == (0, 7)
    # (a, b, c) -> thread 4b + c, slot a
    pm = index_maps.loop_layout_plan((4, 4, 4), [(4, 0, 1), (4, 4, 0), (4, 1, 0)])
    assert pm[(2, 1, 3)] == (7, 2) and pm[(3, 0, 0)] == (0, 3) and pm[(0, 3, 1)] == (13, 0)
    # the default plan on 64 points, 8 threads, pairs: flat = 16 r + 2 t + v
    # gives thread t and slot 2 r + v
    pm = _override_plan((64,), 8, 2)
    for flat in range(64):
        r, rest = divmod(flat, 16)
        t, v = divmod(rest, 2)
        assert pm[(flat,)] == (t, 2 * r + v)


def test_override_hand_worked():
    check_override_hand_worked()


def check_override_sizes():
    """Compact thread and slot parts: T and L are the products of their
    extents; gaps, collisions and mixed modes are refused."""
    rng = random.Random(7)
    for _ in range(60):
        exts = [rng.choice([1, 2, 3, 4]) for _ in range(rng.randint(1, 4))]
        kinds = [rng.randint(0, 1) for _ in exts]
        loop, tstride, sstride = [None] * len(exts), 1, 1
        for i in rng.sample(range(len(exts)), len(exts)):  # compact, in a random order
            if kinds[i]:
                loop[i] = (exts[i], tstride, 0)
                tstride *= exts[i]
            else:
                loop[i] = (exts[i], 0, sstride)
                sstride *= exts[i]
        total = int(np.prod(exts))
        assert index_maps.loop_layout_sizes((total,), loop) == (tstride, sstride)
    for bad in ([(4, 2, 0), (4, 0, 1)],            # threads 0, 2, 4, 6: a gap
                [(4, 1, 0), (4, 1, 0)],            # two points per thread-slot pair
                [(4, 1, 1), (4, 0, 4)],            # a mode feeding both
                [(4, 0, 0), (4, 1, 0)],            # a mode feeding neither
                [(3, 0, 1), (4, 1, 0)]):           # 12 points for a 16-point nest
        with pytest.raises(index_maps.Decline):
            index_maps.loop_layout_sizes((16,), bad)
    with pytest.raises(index_maps.Decline):
        index_maps.default_loop_layout(60, 8, 2)   # the guarded case: 60 = 3 x 16 + 12


def test_override_sizes():
    check_override_sizes()


def test_override_replay_matches_definition():
    """Any exact override moves the same words as the definition; the trace
    records each (thread, slot) pair exactly once per tile."""
    cases = [
        (Layout((8, 8), (8, 1)), Layout((8, 8), (1, 8)), [(8, 0, 1), (8, 1, 0)], 1),
        (Layout((4, 16), (16, 1), 3), Layout((4, 16), (1, 4), 5), [(4, 1, 0), (8, 0, 2), (2, 0, 1)], 2),
        (Layout((2, 1, 4, 32), (128, 128, 32, 1)), Layout((2, 1, 4, 32), (128, 128, 1, 4)),
         index_maps.default_loop_layout(256, 64, 4), 3),
        (Layout((6, 5), (5, 1), 0, 40), Layout((6, 5), (1, 6), 1, 31), [(6, 0, 1), (5, 1, 0)], 2),
    ]
    for src_l, dst_l, loop, n_tiles in cases:
        n_src = src_l.offset + n_tiles * (src_l.tile_stride or definition.cosize(src_l)) + 64
        n_dst = dst_l.offset + n_tiles * (dst_l.tile_stride or definition.cosize(dst_l)) + 64
        src = list(range(1000, 1000 + n_src))
        got = [-1] * n_dst
        trace = index_maps.loop_layout_replay(src, got, src_l, dst_l, loop, n_tiles)
        want = np.full(n_dst * 4, 0xFF, np.uint8)
        definition.copy(np.asarray(src, np.uint32).view(np.uint8), src_l, want, dst_l, 4, n_tiles)
        assert np.asarray(got, np.int64)[np.asarray(got) >= 0].tolist() == \
            want.view(np.uint32)[np.asarray(got) >= 0].astype(np.int64).tolist()
        assert ((want.view(np.uint32) != 0xFFFFFFFF) == (np.asarray(got) >= 0)).all()
        extents = [m[0] for m in definition.paired_modes(src_l, dst_l)]
        T, L = index_maps.loop_layout_sizes(extents, loop)
        N = int(np.prod(extents))
        assert sorted(trace.values()) == sorted(list(range(T * L)) * n_tiles)
        assert len(trace) == n_tiles * N


def test_flatten_unflatten_roundtrip_and_order():
    for extents in [(3,), (2, 5), (4, 1, 3), (2, 3, 4, 5)]:
        total = int(np.prod(extents))
        pts = [index_maps.unflatten(f, extents) for f in range(total)]
        assert pts == list(itertools.product(*(range(e) for e in extents)))
        assert [index_maps.flatten(p, extents) for p in pts] == list(range(total))


# ---------------------------------------------------------------------------
# "permute_layout": worked example, replay and bank simulator
# ---------------------------------------------------------------------------

def _sf_example():
    g = {}
    for ln in _read_golden("permute_layout_sf_transpose.txt"):
        key, _, rest = ln.partition(" ")
        g[key] = rest
    ints = lambda s: tuple(int(v) for v in s.split())
    return g, ints


def check_sf_transpose_example():
    g, ints = _sf_example()
    shape = ints(g["shape"])
    stage = (1,) + shape[1:]
    src = Layout(stage, ints(g["src_stride"]))
    dst = Layout(stage, ints(g["dst_stride"]))
    extent, s_str, d_str, P = index_maps.permute_align(src, dst)
    assert P == int(g["P"])
    choice = banks.choose_xor_k(extent, s_str, d_str, int(g["elem_bytes"]))
    k, shift, mask = choice[:3]
    assert (shift, mask) == (int(g["shift"]), int(g["mask"]))
    for s in range(shape[0]):
        words = list(range(256))
        out = [None] * 256
        rec = index_maps.permute_replay(words, out, extent, s_str, d_str, P, k, shift,
                                        src_base=128 * s, dst_base=128 * s)
        for lane, r, _j, so, do in rec:
            env = {"s": s, "r": r, "tx": lane}
            assert so == eval(g["phase1"], {}, env)
            assert do == eval(g["phase2"], {}, env)
        # the stage's 4x32 block is transposed (numpy), the other stage untouched
        blk = np.array(words[128 * s:128 * s + 128]).reshape(4, 32)
        assert out[128 * s:128 * s + 128] == blk.T.reshape(-1).tolist()


def test_sf_transpose_worked_example():
    check_sf_transpose_example()


def check_bank_degrees_worked_example():
    """Bank degrees of the worked example, worked by hand.

    Phase 1 reads offset 32*j + lane: bank = lane, always 1-way.  Phase 2
    writes offset j + 4*lane: without a swizzle lanes l, l+8, l+16, l+24 hit
    the same bank with different words (4-way); one XOR bit can split them
    only in two (2-way); two bits taken from lane bits 3 and 4 (shift 3)
    split all four, and no other shift does.
    """
    ext, ss, ds = (4, 32), (32, 1), (1, 4)
    assert banks.phase_degrees(ext, ss, ds, 4, 0, 0) == (1, 4)
    assert min(max(banks.phase_degrees(ext, ss, ds, 4, 1, sh)) for sh in range(5)) == 2
    assert banks.phase_degrees(ext, ss, ds, 4, 2, 3) == (1, 1)
    for sh in (0, 1, 2):
        assert max(banks.phase_degrees(ext, ss, ds, 4, 2, sh)) > 1
    assert banks.choose_xor_k(ext, ss, ds, 4)[:3] == (2, 3, 3)


def test_bank_degrees_worked_example():
    check_bank_degrees_worked_example()


def check_access_degree_closed_forms():
    lanes = range(32)
    assert banks.access_degree([4 * l for l in lanes], 4) == 1          # consecutive words
    assert banks.access_degree([128 * l for l in lanes], 4) == 32       # one column
    assert banks.access_degree([0] * 32, 4) == 1                       # broadcast
    assert banks.access_degree([8 * l for l in lanes], 4) == 2         # stride 2 words
    assert banks.access_degree([8 * l for l in lanes], 8) == 1         # 64-bit, half-warps
    assert banks.access_degree([16 * l for l in lanes], 16) == 1       # 128-bit, quarter-warps
    assert banks.access_degree([32 * l for l in lanes], 16) == 2       # 128-bit, stride 2 chunks
    # stride-1 bytes: one word serves four lanes (hardware); distinct elements (strict)
    assert banks.access_degree(list(lanes), 1, "hardware") == 1
    assert banks.access_degree(list(lanes), 1, "strict") == 4
    assert banks.access_degree([2 * l for l in lanes], 2, "strict") == 2


def test_access_degree_closed_forms():
    check_access_degree_closed_forms()


def _dense_permute_cases():
    out = []
    for rank in (1, 2, 3):
        for ext in itertools.product((1, 2, 4, 8, 16, 32), repeat=rank):
            total = int(np.prod(ext))
            if total % 32 or total > 256:
                continue
            for so in itertools.permutations(range(rank)):
                for do in itertools.permutations(range(rank)):
                    out.append((ext, _dense_strides(ext, so), _dense_strides(ext, do)))
    return out


def test_four_byte_dense_transposes_admit_k():
    """The page's claim that 4-byte words always admit a conflict-free k (permute_layout, "How inputs change"),
    read on the op's stated use, a transpose: every dense rank-1/rank-2 case."""
    cases = [c for c in _dense_permute_cases() if len(c[0]) <= 2]
    assert len(cases) > 50
    for ext, ss, ds in cases:
        extent, s_str, d_str, _P = index_maps.permute_align(Layout(ext, ss), Layout(ext, ds))
        assert banks.choose_xor_k(extent, s_str, d_str, 4) is not None, (ext, ss, ds)


def test_three_d_counterexample_has_no_k():
    """Worked by hand: extent (2,2,16), src strides (16,32,1), dst (2,1,4), P = 2.

    Lane l handles c = l % 16, b = l >> 4 and a = j.  The read offset
    16*j + 32*b + c puts lanes l and l + 16 in one bank unless j follows lane
    bit 4; the write offset 2*j + b + 4*c puts lanes l and l + 8 in one bank
    unless j follows lane bit 3.  With P = 2 there is one XOR bit (k <= 1),
    so one phase stays 2-way for every (k, shift): the page's claim does not
    extend to this rank-3 permute.
    """
    ext, ss, ds = (2, 2, 16), (16, 32, 1), (2, 1, 4)
    want = {(0, 0): (2, 2), (1, 3): (2, 1), (1, 4): (1, 2)}
    for k, shift in [(0, 0)] + [(1, s) for s in range(5)]:
        got = banks.phase_degrees(ext, ss, ds, 4, k, shift)
        assert max(got) == 2
        if (k, shift) in want:
            assert got == want[(k, shift)]
    assert banks.choose_xor_k(ext, ss, ds, 4) is None


def test_sub_word_stride_one_reads_can_fail_strict():
    """Stride-1 sub-4-byte reads pack lanes into one bank: with nothing to swizzle
    (P = 1) the strict model fails, the hardware model does not."""
    ext, ss, ds = (32,), (1,), (1,)
    assert banks.choose_xor_k(ext, ss, ds, 1, "strict") is None
    assert banks.choose_xor_k(ext, ss, ds, 2, "strict") is None
    assert banks.choose_xor_k(ext, ss, ds, 1, "hardware")[:3] == (0, 0, 0)


def test_permute_replay_matches_definition():
    """Every admissible (k, shift) moves exactly what the definition moves."""
    for ext, ss, ds in _dense_permute_cases()[::7]:
        extent, s_str, d_str, P = index_maps.permute_align(Layout(ext, ss), Layout(ext, ds))
        total = 32 * P
        src = list(range(500, 500 + total))
        want = np.zeros(total * 4, dtype=np.uint8)
        oracle.copy(np.array(src, dtype=np.uint32).view(np.uint8), Layout(ext, ss),
                    want, Layout(ext, ds), 4)
        kmax = P.bit_length() - 1 if P & (P - 1) == 0 else 0
        for k in range(kmax + 1):
            for shift in range(0, 6 - k):
                out = [None] * total
                rec = index_maps.permute_replay(src, out, extent, s_str, d_str, P, k, shift)
                assert sorted(l + 32 * j for l, _r, j, _s, _d in rec) == list(range(total))
                assert out == want.view(np.uint32).tolist()


def test_permute_replay_in_place():
    """The warp barrier between the phases makes src == dst safe."""
    ext, ss, ds = (4, 32), (32, 1), (1, 4)
    buf = list(range(128))
    index_maps.permute_replay(buf, buf, ext, ss, ds, 4, 2, 3)
    assert buf == np.arange(128).reshape(4, 32).T.reshape(-1).tolist()


def test_chosen_k_is_conflict_free():
    for ext, ss, ds in _dense_permute_cases()[::3]:
        extent, s_str, d_str, _P = index_maps.permute_align(Layout(ext, ss), Layout(ext, ds))
        for w in (4, 8, 16):
            c = banks.choose_xor_k(extent, s_str, d_str, w)
            if c is None:
                continue
            k, shift, _m, rd, wd = c
            assert (rd, wd) == (1, 1)
            assert banks.phase_degrees(extent, s_str, d_str, w, k, shift) == (1, 1)


# ---------------------------------------------------------------------------
# planted mistakes: every plausible slip must trip at least one pin
# ---------------------------------------------------------------------------

ALL_PINS = [check_definition_vs_numpy, check_transpose_vs_numpy, check_axis_permute_vs_numpy,
            check_gmem_smem_table, check_gmem_smem_alignment_rule, check_round_trip_identity,
            check_gmem_smem_guarded, check_xor_swizzle,
            check_loop_mapping_tables, check_default_override_tables, check_override_hand_worked,
            check_override_sizes, check_sf_transpose_example,
            check_bank_degrees_worked_example, check_access_degree_closed_forms]


def _some_pin_fails():
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, IndexError, KeyError, ValueError, TypeError,
                index_maps.Decline):
            return True
    return False


def _mut_unflatten_transposed(flat, extents):
    coords = []
    for e in extents:  # peels the FIRST coordinate first: a transposed order
        flat, c = divmod(flat, e)
        coords.append(c)
    return tuple(coords)


def _mut_swizzle_dropped(lane, r, k, shift):
    return r


def _mut_swizzle_wrong_sign(lane, r, k, shift):
    return r ^ ((lane << shift) & ((1 << k) - 1))


def _mut_paired_swapped(src, dst):
    return [(e, d, s) for e, s, d in definition.__dict__["_orig_paired"](src, dst)]


@pytest.mark.parametrize("mutation", [
    "unflatten_transposed", "swizzle_dropped", "swizzle_shift_wrong_way",
    "pairing_swapped", "plan_thread_slot_swapped", "vec_ignores_offsets",
    "bank_counts_lanes_not_words", "project_drops_last_term",
    "override_thread_slot_swapped", "override_digits_column_major",
    "guard_drops_last_round", "swizzle_xors_chunk_into_row",
])
def test_planted_mistakes(monkeypatch, mutation):
    assert not _some_pin_fails()  # the unmutated oracle passes every pin
    if mutation == "unflatten_transposed":
        monkeypatch.setattr(index_maps, "unflatten", _mut_unflatten_transposed)
        monkeypatch.setattr(banks, "unflatten", _mut_unflatten_transposed)
    elif mutation == "swizzle_dropped":
        monkeypatch.setattr(index_maps, "swizzled_iteration", _mut_swizzle_dropped)
        monkeypatch.setattr(banks, "swizzled_iteration", _mut_swizzle_dropped)
    elif mutation == "swizzle_shift_wrong_way":
        monkeypatch.setattr(index_maps, "swizzled_iteration", _mut_swizzle_wrong_sign)
        monkeypatch.setattr(banks, "swizzled_iteration", _mut_swizzle_wrong_sign)
    elif mutation == "pairing_swapped":
        monkeypatch.setitem(definition.__dict__, "_orig_paired", definition.paired_modes)
        monkeypatch.setattr(definition, "paired_modes", _mut_paired_swapped)
        monkeypatch.setattr(index_maps, "paired_modes", _mut_paired_swapped)
    elif mutation == "plan_thread_slot_swapped":
        orig = index_maps.plan

        def bad_plan(extents, num_thread, vector_size):
            return {k: (s, t) for k, (t, s) in orig(extents, num_thread, vector_size).items()}
        monkeypatch.setattr(index_maps, "plan", bad_plan)
    elif mutation == "vec_ignores_offsets":
        orig = index_maps.gmem_smem_partition

        def bad_part(shape, g, s, w, T, g_offset=0, s_offset=0):
            return orig(shape, g, s, w, T, 0, 0)
        monkeypatch.setattr(index_maps, "gmem_smem_partition", bad_part)
    elif mutation == "bank_counts_lanes_not_words":
        def bad_degree(addrs, w, model="hardware"):
            per = banks.wavefront_lanes(w)
            worst = 0
            for st in range(0, len(addrs), per):
                cnt = {}
                for a in addrs[st:st + per]:
                    cnt[(a // 4) % 32] = cnt.get((a // 4) % 32, 0) + 1
                worst = max([worst] + list(cnt.values()))
            return worst
        monkeypatch.setattr(banks, "access_degree", bad_degree)
    elif mutation == "project_drops_last_term":
        def bad_project(idx, strides):
            return sum(i * s for i, s in zip(idx[:-1], strides[:-1]))
        monkeypatch.setattr(index_maps, "project", bad_project)
        monkeypatch.setattr(banks, "project", bad_project)
    elif mutation == "override_thread_slot_swapped":
        orig = index_maps.loop_layout_plan

        def bad_override(extents, loop):
            return {k: (s, t) for k, (t, s) in orig(extents, loop).items()}
        monkeypatch.setattr(index_maps, "loop_layout_plan", bad_override)
    elif mutation == "override_digits_column_major":
        def bad_override(extents, loop):
            out = {}
            for flat in range(int(np.prod(extents))):
                digits = _mut_unflatten_transposed(flat, [m[0] for m in loop])
                out[index_maps.unflatten(flat, extents)] = (
                    sum(c * m[1] for c, m in zip(digits, loop)),
                    sum(c * m[2] for c, m in zip(digits, loop)))
            return out
        monkeypatch.setattr(index_maps, "loop_layout_plan", bad_override)
    elif mutation == "guard_drops_last_round":
        orig = index_maps.gmem_smem_partition_guarded

        def bad_guarded(*args, **kw):  # rounds rounded down: the partial round is lost
            part = dict(orig(*args, **kw))
            part["outer"] -= 1 if part["guarded"] else 0
            return part
        monkeypatch.setattr(index_maps, "gmem_smem_partition_guarded", bad_guarded)
    elif mutation == "swizzle_xors_chunk_into_row":
        def bad_swizzle(o, bits, c, r):
            return o ^ (((o >> c) & ((1 << bits) - 1)) << r)
        monkeypatch.setattr(index_maps, "xor_swizzle", bad_swizzle)
    assert _some_pin_fails(), mutation
