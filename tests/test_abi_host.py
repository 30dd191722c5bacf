"""The C-ABI library on the host (no GPU): symbols, planner, bank simulator,
[outer, threads, vec] partition and validation, against the oracle."""
import itertools
import os
import random
import re

import numpy as np
import pytest

import oracle
from oracle import banks, index_maps
from oracle.definition import Layout

from conftest import ROOT


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import movement_primitives_gb300
    return movement_primitives_gb300


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(lc_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(M):
    import ctypes
    names = _declared_functions()
    assert len(names) >= 10
    handle = ctypes.CDLL(M._lib.LIB_PATH)
    for n in names:
        assert hasattr(handle, n), n
    assert set(names) == set(M._lib.PROTOTYPES), "binding and header disagree"


def test_status_and_kernel_names(M):
    lib = M._lib.lib()
    for code in range(17):
        assert lib.lc_status_string(code) and lib.lc_status_string(code) != b"unknown status"
    assert lib.lc_kernel_name(2) == b"warp_permute"


# ---------------------------------------------------------------------------
# planner on the workloads and the pages' worked examples
# ---------------------------------------------------------------------------

def test_plan_scale_factor_transpose(M):
    """'permute_layout' demonstration: P = 4, shift = 3, mask = 3 (k = 2)."""
    import workloads
    c = workloads.config(2)
    p = M.plan(c["src"], c["dst"], 4, c["n_tiles"], "warp_permute")
    assert p["kernel_name"] == "warp_permute"
    assert (p["P"], p["k"], p["shift"], p["mask"]) == (4, 2, 3, 3)
    assert (p["conflicts_read"], p["conflicts_write"]) == (1, 1)
    assert p["modes"][-2:] == [(4, 32, 1), (32, 1, 4)]
    # the automatic choice moves the same (4, 32) blocks through warp shuffles:
    # V = 4 words per 16-byte chunk, 32 / 4 = 8 blocks of 4 x 4 words per unit
    a = M.plan(c["src"], c["dst"], 4, c["n_tiles"])
    assert a["kernel_name"] == "warp_shuffle"
    assert (a["vec"], a["units_per_chunk"]) == (4, 8)
    assert (a["conflicts_read"], a["conflicts_write"]) == (0, 0)  # no shared memory


def test_plan_workloads(M):
    import workloads
    expect = {1: "smem_transpose", 3: "tile_transpose", 5: "tma_copy"}
    for cfg, kname in expect.items():
        c = workloads.config(cfg)
        assert M.plan(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"])["kernel_name"] == kname
    for w in (1, 2, 4, 8, 16):
        c = workloads.config(4, w)
        p = M.plan(c["src"], c["dst"], w, 1)
        assert p["kernel_name"] == "tile_transpose"
        if w == 1:
            # 64 MiB a side: the direct form, warp tiles of 4 chunks (64 bytes) x 8 blocks of 16 rows
            assert (p["tile_form"], p["stages"], p["tile_cols"], p["tile_rows"]) == (1, 0, 64, 128)
        elif w == 2:
            # 128 MiB: the ring's short boxes, 128-byte rows (swizzled, line stores), 3 stages
            assert (p["tile_form"], p["stages"], p["tile_cols"] * w, p["tile_rows"]) == (0, 3, 128, 128)
        elif w == 4:
            # TMA stores: swizzled boxes of 128-byte rows x 256 rows in, 32 x 256-word tiles out
            assert (p["tile_form"], p["tile_cols"], p["tile_rows"], p["stages"]) == (2, 32, 256, 3)
        else:
            # 512 MiB and 1 GiB: the ring with thread stores, box rows of 256 / 128 bytes
            assert p["tile_form"] == 0 and p["stages"] > 0 and p["tile_cols"] * w == (256 if w == 8 else 128)
    p = M.plan(workloads.config(5)["src"], workloads.config(5)["dst"], 2)
    assert (p["vec"], p["run"]) == (8, 128)  # the vector fallback: 16-byte vectors over 256-byte runs
    # TMA boxes: the 128-word run, its 32 rows, 2 of the next mode (16 KiB)
    assert (p["tile_cols"], p["tile_rows"], p["stages"]) == (128, 32, 6)


def test_plan_tile_direct_form(M):
    """The tile transpose takes its direct form (stages 0) for 1- and 2-byte
    words when both extents are whole V x V blocks and the copy is at most
    256 MiB a side; ragged extents, wider words and larger copies keep the
    TMA ring."""
    def plan(shape_src, stride_src, stride_dst, w, n_tiles=1):
        p = M.plan(dict(shape=shape_src, stride=stride_src), dict(shape=shape_src, stride=stride_dst), w,
                   n_tiles, "tile_transpose")
        assert p["kernel_name"] == "tile_transpose"
        return p["stages"]
    for w in (1, 2):
        V = 16 // w
        assert plan((V, V), (V, 1), (1, V), w) == 0
        assert plan((9 * V, 5 * V), (5 * V + V, 1), (1, 9 * V + V), w) == 0        # padded rows
        assert plan((3, 4 * V, 2 * V), (8 * V * V, 2 * V, 1), (8 * V * V, 1, 4 * V), w, 2) == 0  # batch, tiles
        assert plan((9 * V, 5 * V - 1), (5 * V, 1), (1, 9 * V), w) > 0             # ragged Y
        assert plan((9 * V - 1, 5 * V), (5 * V, 1), (1, 9 * V), w) > 0             # ragged X
        big = (16384, 16384 + V) if w == 1 else (8192, 16384 + V)                  # past 256 MiB a side
        assert plan(big, (big[1], 1), (1, big[0]), w) > 0
    for w in (4, 8, 16):
        assert plan((64, 64), (64, 1), (1, 64), w) > 0


def test_plan_tile_store_forms(M):
    """The tile transpose's form by word width and size a side, where the
    destination rows are whole 16-byte chunks: TMA tensor stores (tile_form
    2) for 4-byte words at every size, 8- and 16-byte words up to 256 MiB,
    1- and 2-byte words above it; the direct form (1) for whole blocks of 1-
    and 2-byte words up to 96 / 64 MiB; thread stores (0) otherwise, and for
    every destination row that ends inside a 16-byte chunk."""
    def form(shape, s_stride, d_stride, w, kernel="tile_transpose"):
        p = M.plan(dict(shape=shape, stride=s_stride), dict(shape=shape, stride=d_stride), w, 1, kernel)
        assert p["kernel_name"] == "tile_transpose"
        return p["tile_form"]
    assert form((64, 36), (36, 1), (1, 64), 4) == 2
    assert form((61, 36), (36, 1), (1, 64), 4) == 0            # destination rows of 61 words
    assert form((64, 35), (36, 1), (1, 64), 4) == 2            # ragged source rows: clipped per row
    assert form((8192, 8200), (8200, 1), (1, 8192), 4) == 2    # past 256 MiB a side
    assert form((64, 64), (64, 1), (1, 64), 8) == 2
    assert form((63, 64), (64, 1), (1, 64), 8) == 0
    assert form((8192, 8192), (8192, 1), (1, 8192), 8) == 0    # 512 MiB
    assert form((64, 64), (64, 1), (1, 64), 16) == 2
    assert form((8192, 4160), (4160, 1), (1, 8192), 16) == 0   # past 256 MiB
    assert form((64, 64), (64, 1), (1, 64), 2) == 1
    assert form((64, 60), (64, 1), (1, 64), 2) == 0
    assert form((8192, 8192), (8192, 1), (1, 8192), 2) == 0    # 128 MiB: the ring's short boxes
    assert form((12288, 12288), (12288, 1), (1, 12288), 2) == 2  # 288 MiB
    assert form((16384, 16384), (16384, 1), (1, 16384), 2) == 0  # 512 MiB, destination rows 32 KiB apart
    assert form((16000, 16000), (16000, 1), (1, 16000), 2) == 2
    assert form((8192, 8192), (8192, 1), (1, 8192), 1) == 1    # 64 MiB
    assert form((11520, 11520), (11520, 1), (1, 11520), 1) == 0  # 126 MiB
    assert form((16384, 16640), (16640, 1), (1, 16384), 1) == 2  # 260 MiB
    p = M.plan(dict(shape=(64, 64), stride=(64, 1)), dict(shape=(64, 64), stride=(64, 1)), 4, 1)
    assert p["tile_form"] == 0                                 # not a tile transpose


def test_gmem_smem_partition_table(M):
    """'copy -> gmem_smem' dtype table: fp32 vec 4 / outer 8, fp16 8 / 4, u8 16 / 2."""
    for w, vec, outer in [(4, 4, 8), (2, 8, 4), (1, 16, 2)]:
        assert M.gmem_smem_partition(M.TileLayout((32, 32)), M.TileLayout((32, 32)), w, 32) == (vec, outer)


def test_gmem_smem_partition_matches_oracle(M):
    rng = random.Random(3)
    for _ in range(300):
        rank = rng.randint(1, 3)
        ext = tuple(rng.choice([1, 2, 4, 8, 16]) for _ in range(rank))
        go = list(range(rank)); rng.shuffle(go)
        so = list(range(rank)); rng.shuffle(so)

        def st(order):
            s, acc = [0] * rank, 1
            for m in reversed(order):
                s[m] = acc
                acc *= ext[m]
            return tuple(s)
        g, s = st(go), st(so)
        w = rng.choice([1, 2, 4, 8, 16])
        T = rng.choice([1, 2, 4, 8, 32])
        goff, soff = rng.choice([0, 0, 2, 4]), rng.choice([0, 0, 8])
        try:
            want = index_maps.gmem_smem_partition(ext, g, s, w, T, goff, soff)
        except index_maps.Decline:
            with pytest.raises(M.LayoutCopyError):
                M.gmem_smem_partition(M.TileLayout(ext, g, goff), M.TileLayout(ext, s, soff), w, T)
            continue
        got = M.gmem_smem_partition(M.TileLayout(ext, g, goff), M.TileLayout(ext, s, soff), w, T)
        assert got == (want["vec"], want["outer"]), (ext, g, s, w, T)


# ---------------------------------------------------------------------------
# bank simulator / XOR choice against the oracle's
# ---------------------------------------------------------------------------

def _swizzle_cases():
    cases = []
    for rank in (1, 2, 3):
        for ext in itertools.product((1, 2, 4, 8, 16, 32), repeat=rank):
            total = int(np.prod(ext))
            if total % 32 or total > 256:
                continue
            for so in itertools.permutations(range(rank)):
                for do in itertools.permutations(range(rank)):
                    def st(order):
                        s, acc = [0] * rank, 1
                        for m in reversed(order):
                            s[m] = acc
                            acc *= ext[m]
                        return tuple(s)
                    cases.append((ext, st(so), st(do)))
    return cases


def test_choose_swizzle_matches_oracle(M):
    cases = _swizzle_cases()
    for i, (ext, ss, ds) in enumerate(cases[::5]):
        for w in ((1, 2, 4, 8, 16) if i % 7 == 0 else (4,)):
            got = M.choose_swizzle(M.TileLayout(ext, ss), M.TileLayout(ext, ds), w)
            e, s_str, d_str, _P = index_maps.permute_align(Layout(ext, ss), Layout(ext, ds))
            want = banks.choose_xor_k(e, s_str, d_str, w)
            if want is None:
                assert not got["ok"]
            else:
                assert got["ok"]
                assert (got["k"], got["shift"], got["mask"], got["conflicts_read"],
                        got["conflicts_write"]) == want, (ext, ss, ds, w)


def test_swizzle_conflicts_match_oracle(M):
    rng = random.Random(9)
    cases = _swizzle_cases()
    for _ in range(150):
        ext, ss, ds = rng.choice(cases)
        w = rng.choice([1, 2, 4, 8, 16])
        e, s_str, d_str, P = index_maps.permute_align(Layout(ext, ss), Layout(ext, ds))
        kmax = P.bit_length() - 1 if P & (P - 1) == 0 else 0
        k = rng.randint(0, kmax)
        shift = rng.randint(0, 5 - k) if k else 0
        got = M.swizzle_conflicts(M.TileLayout(ext, ss), M.TileLayout(ext, ds), w, k, shift)
        assert got == banks.phase_degrees(e, s_str, d_str, w, k, shift)


def test_choose_swizzle_worked_example(M):
    sl = M.TileLayout((1, 1, 4, 32), (128, 128, 32, 1))
    dl = M.TileLayout((1, 1, 4, 32), (128, 128, 1, 4))
    assert M.choose_swizzle(sl, dl, 4) == dict(ok=True, k=2, shift=3, mask=3,
                                               conflicts_read=1, conflicts_write=1)
    assert M.swizzle_conflicts(sl, dl, 4, 0, 0) == (1, 4)


# ---------------------------------------------------------------------------
# validation (host-side status codes; no launch happens on these paths)
# ---------------------------------------------------------------------------

def test_validation_codes(M):
    S = M.STATUS
    T = M.TileLayout

    def code(src, dst, w=4, n=1):
        try:
            M.plan(src, dst, w, n)
            return 0
        except M.LayoutCopyError as e:
            return e.status

    assert code(T((4, 5), (5, 1)), T((5, 4), (4, 1))) == S["LC_ERR_EXTENT_MISMATCH"]
    assert code(T((4, 4), (4, 1)), T((4, 4), (1, 4)), w=3) == S["LC_ERR_ELEM_BYTES"]
    assert code(T((4, 4), (4, -1)), T((4, 4), (1, 4))) == S["LC_ERR_BAD_STRIDE"]
    assert code(T((4, 4), (4, 1)), T((4, 4), (0, 4))) == S["LC_ERR_BAD_STRIDE"]
    assert code(T((4, 4), (4, 1)), T((4, 4), (1, 1))) == S["LC_ERR_NOT_INJECTIVE"]
    assert code(T((4, 4), (4, 1)), T((4, 4), (2, 1))) == S["LC_ERR_NOT_INJECTIVE"]
    assert code(T((4, 4), (4, 1)), T((4, 4), (4, 1)), n=-1) == S["LC_ERR_SHAPE"]
    assert code(T((-1, 4), (4, 1)), T((-1, 4), (4, 1))) == S["LC_ERR_SHAPE"]
    assert code(T((2,) * 9, (1,) * 9), T((2,) * 9, (1,) * 9)) == S["LC_ERR_RANK"]
    assert code(T((4, 4), (4, 1), -1), T((4, 4), (1, 4))) == S["LC_ERR_BAD_STRIDE"]
    assert code(T((1 << 40, 1 << 30), (1 << 30, 1)), T((1 << 40, 1 << 30), (1, 1 << 40))) \
        == S["LC_ERR_OVERFLOW"]
    # injective but not nested: proved by enumeration
    assert code(T((2, 3), (3, 2)), T((2, 3), (3, 2))) == 0
    # tiles that overlap on the destination
    assert code(T((4,), (1,)), T((4,), (1,), 0, 2), n=3) == S["LC_ERR_NOT_INJECTIVE"]
    # over 2^24 words and not nested: offsets k + 2^23 (2i + 3j) are distinct
    # (the dense inner mode stays below the other strides' gcd 2^23, and
    # 2i + 3j is one-to-one on 3 x 2); on 4 x 3, 2i + 3j collides (3,0)/(0,2)
    big = (3, 2, 1 << 23)
    assert code(T(big, (2 << 23, 1 << 23, 1)), T(big, (1 << 24, 3 << 23, 1)), w=1) == 0
    big = (4, 3, 1 << 23)
    assert code(T(big, (3 << 23, 1 << 23, 1)), T(big, (1 << 24, 3 << 23, 1)), w=1) == S["LC_ERR_NOT_INJECTIVE"]
    # no stride split settles 3i + 5j and 2^25 words are too many to enumerate
    assert code(T((1 << 13, 1 << 12), (1 << 12, 1)), T((1 << 13, 1 << 12), (3, 5)), w=1) == S["LC_ERR_UNDECIDED"]
    # zero-size copies are fine
    assert code(T((0, 4), (4, 1)), T((0, 4), (1, 4))) == 0
    assert code(T((4, 4), (4, 1)), T((4, 4), (1, 4)), n=0) == 0


def test_forced_kernel_unsupported(M):
    T = M.TileLayout
    with pytest.raises(M.LayoutCopyError) as e:
        M.plan(T((100,), (1,)), T((100,), (1,)), 4, 1, kernel="tile_transpose")
    assert e.value.status == M.STATUS["LC_ERR_UNSUPPORTED"]
    with pytest.raises(M.LayoutCopyError):
        M.plan(T((40, 40), (40, 1)), T((40, 40), (1, 40)), 4, 1, kernel="warp_permute")


def test_pointer_checks_before_launch(M):
    """NULL / misaligned / overlapping pointers are refused before any CUDA call."""
    T = M.TileLayout
    lay = T((16, 16), (16, 1))
    for args, status in [((0, lay, 4096, lay, 4), "LC_ERR_NULL"),
                         ((4098, lay, 1 << 20, lay, 4), "LC_ERR_ALIGN"),
                         ((4096, lay, 4096 + 512, lay, 4), "LC_ERR_OVERLAP")]:
        with pytest.raises(M.LayoutCopyError) as e:
            M.layout_copy_ptr(*args, stream=0)
        assert e.value.status == M.STATUS[status]


# ---------------------------------------------------------------------------
# loop-layout override
# ---------------------------------------------------------------------------

def test_loop_layout_default_matches_oracle(M):
    for total, T, V in [(64, 8, 2), (256, 64, 4), (1 << 19, 1024, 8), (12, 1, 1), (0, 4, 2), (32, 32, 1)]:
        assert M.loop_layout_default(total, T, V) == index_maps.default_loop_layout(total, T, V)
    for total, T, V in [(60, 8, 2), (7, 2, 1)]:  # the guarded case
        with pytest.raises(index_maps.Decline):
            index_maps.default_loop_layout(total, T, V)
        with pytest.raises(M.LayoutCopyError) as e:
            M.loop_layout_default(total, T, V)
        assert e.value.status == M.STATUS["LC_ERR_SHAPE"]


def _random_loops(rng, n):
    strides = [0, 0, 1, 1, 2, 3, 4, 6, 8, 12, 16]
    for _ in range(n):
        r = rng.randint(1, 4)
        yield [(rng.choice([1, 2, 2, 3, 4]), rng.choice(strides), rng.choice(strides)) for _ in range(r)]
    for _ in range(n):  # exact partitions, in random mode orders
        exts = [rng.choice([1, 2, 3, 4]) for _ in range(rng.randint(1, 5))]
        loop, ts, ss = [None] * len(exts), 1, 1
        for i in rng.sample(range(len(exts)), len(exts)):
            if rng.random() < 0.5:
                loop[i], ts = (exts[i], ts, 0), ts * exts[i]
            else:
                loop[i], ss = (exts[i], 0, ss), ss * exts[i]
        yield loop


def test_loop_layout_info_matches_oracle(M):
    """Accept / refuse and (T, L) agree with the oracle's brute-force check."""
    rng = random.Random(11)
    accepted = refused = 0
    for loop in _random_loops(rng, 400):
        total = int(np.prod([m[0] for m in loop]))
        try:
            want = index_maps.loop_layout_sizes((total,), loop)
        except index_maps.Decline:
            want = None
        try:
            got = M.loop_layout_info(loop, total)
        except M.LayoutCopyError:
            got = None
        assert got == want, loop
        accepted += want is not None
        refused += want is None
    assert accepted > 300 and refused > 100
    with pytest.raises(M.LayoutCopyError) as e:
        M.loop_layout_info([(2048, 1, 0)], 2048)
    assert e.value.status == M.STATUS["LC_ERR_LOOP_LAYOUT"]  # over 1024 threads
    with pytest.raises(M.LayoutCopyError) as e:
        M.loop_layout_info([(4, 1, 0)], 8)
    assert e.value.status == M.STATUS["LC_ERR_SHAPE"]


def test_layout_copy_loop_checks_before_launch(M):
    """Refusals of lc_layout_copy_loop come before any CUDA call."""
    T = M.TileLayout
    src, dst = T((8, 8), (8, 1)), T((8, 8), (1, 8))
    col = [(8, 0, 1), (8, 1, 0)]
    cases = [((0, src, 1 << 20, dst, 4, col), "LC_ERR_NULL"),
             ((4096, src, 4096 + 128, dst, 4, col), "LC_ERR_OVERLAP"),
             ((4096, src, 1 << 20, dst, 4, [(4, 0, 1), (8, 1, 0)]), "LC_ERR_SHAPE"),
             ((4096, src, 1 << 20, dst, 4, [(8, 2, 0), (8, 0, 1)]), "LC_ERR_LOOP_LAYOUT"),
             ((4096, src, 1 << 20, dst, 4, [(8, 1, 1), (8, 0, 8)]), "LC_ERR_BAD_STRIDE"),
             ((4096, src, 1 << 20, T((8, 7), (7, 1)), 4, col), "LC_ERR_EXTENT_MISMATCH"),
             ((4098, src, 1 << 20, dst, 4, col), "LC_ERR_ALIGN")]
    for args, status in cases:
        with pytest.raises(M.LayoutCopyError) as e:
            M.layout_copy_loop_ptr(*args, stream=0)
        assert e.value.status == M.STATUS[status], (args, status)
    with pytest.raises(M.LayoutCopyError) as e:  # a misaligned trace
        M.layout_copy_loop_ptr(4096, src, 1 << 20, dst, 4, col, 1, trace_ptr=(1 << 22) + 4)
    assert e.value.status == M.STATUS["LC_ERR_ALIGN"]
    # nothing to move: no launch, no error
    M.layout_copy_loop_ptr(4096, src, 1 << 20, dst, 4, col, n_tiles=0)
    M.layout_copy_loop_ptr(4096, T((0, 8), (8, 1)), 1 << 20, T((0, 8), (1, 8)), 4, [(0, 1, 0)])


def test_layout_conversion_cache(M):
    """Layouts are converted to their C struct once per distinct value: a
    changed dict gives a fresh struct, equal values share one, and the
    bounded cache stays correct when it is cleared."""
    d = {"shape": (4, 8), "stride": (8, 1), "offset": 3, "tile_stride": 0}
    a = M._c_layout(d)
    assert M._c_layout(dict(d)) is a
    assert (a.rank, list(a.shape)[:2], list(a.stride)[:2], a.offset) == (2, [4, 8], [8, 1], 3)
    d["offset"] = 5
    b = M._c_layout(d)
    assert b is not a and b.offset == 5 and a.offset == 3
    assert M._c_layout(M.TileLayout((4, 8), (8, 1), 5)).offset == 5
    for i in range(M._LAYOUT_CACHE_MAX + 10):  # overflow clears the cache
        assert M._c_layout({"shape": (i + 1,), "stride": (1,)}).shape[0] == i + 1
    assert M._c_layout(d).offset == 5
    assert M.plan(M.TileLayout((32, 32)), M.TileLayout((32, 32), (1, 32)), 4)["kernel_name"] == "smem_transpose"


def test_fastdiv_host_mirror():
    """The invariant-divisor division used by the vector copy, re-derived here
    from the published method and checked against integer division."""
    def make(d):
        s = 0
        while (1 << s) < d:
            s += 1
        m = ((1 << 32) * ((1 << s) - d)) // d + 1
        return m & 0xFFFFFFFF, s
    rng = random.Random(1)
    ds = [1, 2, 3, 5, 7, 31, 32, 33, 128, 1000, 65535, 65536, (1 << 31) - 1, 1 << 31, (1 << 32) - 1]
    ds += [rng.randrange(1, 1 << 32) for _ in range(200)]
    for d in ds:
        m, s = make(d)
        for n in [0, 1, d - 1, d, d + 1, (1 << 32) - 1, (1 << 31)] + [rng.randrange(1 << 32) for _ in range(50)]:
            n &= 0xFFFFFFFF
            q = (((n * m) >> 32) + n) >> s
            assert q == n // d, (n, d)


def test_overlaps_other_than_exact_unit_alias_are_refused(M):
    """Only an exact in-place permute of dense units may alias; every other
    overlap is refused before anything is launched."""
    T = M.TileLayout
    p = 1 << 20
    cases = [
        # a 64 x 64 transpose in place: units would exceed 32 words per lane
        (p, T((64, 64), (64, 1)), p, T((64, 64), (1, 64)), 4, 1),
        # unit permute with the destination shifted by one unit: ranges overlap
        (p, T((4, 32), (32, 1)), p + 512, T((4, 32), (1, 4)), 4, 8),
        # equal bases but different tile strides
        (p, T((4, 32), (32, 1), 0, 128), p, T((4, 32), (1, 4), 0, 256), 4, 8),
        # identical layouts through the vector copy
        (p, T((4096,), (1,)), p, T((4096,), (1,)), 4, 1),
    ]
    for sp, sl, dp, dl, w, n in cases:
        with pytest.raises(M.LayoutCopyError) as e:
            M.layout_copy_ptr(sp, sl, dp, dl, w, n, stream=0)
        assert e.value.status == M.STATUS["LC_ERR_OVERLAP"], (sl, dl)


def test_smem_transpose_swizzle_is_conflict_free_by_the_oracle(M):
    """The shared-memory transpose's chunk swizzle, checked with the oracle's
    own bank model.  A tile is TX rows of RB bytes; chunk k (C bytes) of row x
    sits in slot k ^ ((x >> shift) & mask).  Copy 1: thread t of 256 writes
    chunk t % NC of row t // NC (+ 256 // NC per round).  Copy 2: 32 lanes read
    word y of 32 consecutive rows (rows without lead-in bytes).  Every warp
    access must be 1-way."""
    T = M.TileLayout
    geometry = {1: (4, 256, 64, 252), 2: (4, 256, 64, 124), 4: (4, 256, 64, 64),
                8: (8, 512, 64, 64), 16: (16, 512, 32, 32)}
    for w, (C, RB, TX, TYW) in geometry.items():
        p = M.plan(T((37, 555), (555, 1)), T((37, 555), (1, 37)), w, 1, kernel="smem_transpose")
        assert p["kernel_name"] == "smem_transpose"
        assert (p["tile_rows"], p["tile_cols"]) == (TX, TYW)
        shift, mask = p["shift"], p["mask"]
        NC = RB // C
        sw = lambda x: (x >> shift) & mask
        for x in range(TX):
            assert sorted(k ^ sw(x) for k in range(NC)) == list(range(NC))  # each row a permutation
        for r in range(TX * NC // 256):
            for t0 in range(0, 256, 32):
                writes = [(t // NC + r * (256 // NC)) * RB + ((t % NC) ^ sw(t // NC + r * (256 // NC))) * C
                          for t in range(t0, t0 + 32)]
                assert banks.access_degree(writes, C) == 1, (w, r, t0)
        for y in range(TYW):
            for base in range(0, TX, 32):
                reads = [(base + l) * RB + ((y * w) ^ (sw(base + l) * C)) for l in range(32)]
                assert banks.access_degree(reads, w) == 1, (w, y)
        assert (p["conflicts_read"], p["conflicts_write"]) == (1, 1)


def test_tma_copy_plans(M):
    """The TMA tensor copy takes layouts whose innermost mode is contiguous on
    both sides (at least 64 bytes, 16-byte multiples), at most 5 modes, all
    other strides 16-byte multiples; everything else stays on other classes."""
    T = M.TileLayout
    perm = lambda w: M.plan(T((8, 3, 64), (192, 64, 1)), T((8, 3, 64), (64, 512, 1)), w)
    for w in (1, 2, 4, 8, 16):
        p = perm(w)
        assert p["kernel_name"] == "tma_copy", w
        eb = w if w < 16 else 8  # 16-byte words travel as two 8-byte TMA elements
        assert p["tile_cols"] * eb == min(64 * w, 256 * eb)  # the whole 64-word run
        assert p["tile_cols"] * eb * p["tile_rows"] <= 16384
    # 48-byte runs: too short; 40 one-byte words: not a 16-byte multiple
    assert M.plan(T((8, 3, 24), (72, 24, 1)), T((8, 3, 24), (24, 192, 1)), 2)["kernel_name"] == "vec_copy"
    assert M.plan(T((8, 3, 40), (120, 40, 1)), T((8, 3, 40), (40, 320, 1)), 1)["kernel_name"] == "vec_copy"
    # odd outer strides (not 16-byte multiples)
    assert M.plan(T((8, 3, 64), (193, 64, 1)), T((8, 3, 64), (64, 512, 1)), 2)["kernel_name"] == "vec_copy"
    # six modes after coalescing: beyond a tensor map's five dimensions
    sh = (2, 2, 2, 2, 2, 64)
    st = (64 * 32, 64 * 16, 64 * 8, 64 * 4, 64 * 2, 1)
    dt = (64 * 2, 64 * 4, 64 * 8, 64 * 16, 64 * 32, 1)
    assert M.plan(T(sh, st), T(sh, dt), 4)["kernel_name"] == "vec_copy"
    # a single contiguous mode (an identity copy) stays on the vector copy
    assert M.plan(T((4096,), (1,)), T((4096,), (1,)), 4)["kernel_name"] == "vec_copy"
    # the forced class declines what it cannot take
    with pytest.raises(M.LayoutCopyError):
        M.plan(T((8, 3, 24), (72, 24, 1)), T((8, 3, 24), (24, 192, 1)), 2, kernel="tma_copy")
    # runs under 256 bytes: the 16 KiB box splits between the destination's
    # next mode (S) and the source's (H): 32 x 16 x 16 two-byte words for a
    # (B, S, H, 32) -> (B, H, S, 32) permute; 256-byte runs keep the
    # destination's next mode whole (32 rows)
    p = M.plan(T((4, 64, 32, 32), (65536, 1024, 32, 1)), T((4, 64, 32, 32), (65536, 32, 2048, 1)), 2)
    assert (p["kernel_name"], p["tile_cols"], p["tile_rows"]) == ("tma_copy", 32, 16)
    p = M.plan(T((4, 64, 32, 128), (262144, 4096, 128, 1)), T((4, 64, 32, 128), (262144, 128, 8192, 1)), 2)
    assert (p["kernel_name"], p["tile_cols"], p["tile_rows"]) == ("tma_copy", 128, 64)


def test_unaligned_transposes_plan_the_smem_transpose(M):
    T = M.TileLayout
    for w in (1, 2, 4, 8):  # single tiles past the 32 KiB small-tile rule
        p = M.plan(T((137, 555), (555, 1)), T((137, 555), (1, 137)), w, 1)
        assert p["kernel_name"] == "smem_transpose", w
    # aligned ones keep the TMA path
    assert M.plan(T((128, 128), (128, 1)), T((128, 128), (1, 128)), 4, 1)["kernel_name"] == "tile_transpose"


def _unit_point(modes, flat):
    """(source, destination) word offsets of logical index `flat` of a unit
    whose modes (extent, src_stride, dst_stride) are listed outermost first."""
    so = do = 0
    for e, ss, ds in reversed(modes):
        so += (flat % e) * ss
        do += (flat % e) * ds
        flat //= e
    return so, do


def test_warp_unit_lane_digits_split_where_32_nests(M):
    """The identity behind the warp permute's offsets without stored
    tables: when every suffix product of the unit's extents divides 32 or is
    a multiple of it, the logical index lane + 32 j has disjoint lane and j
    digits, so its offset on either side is the offset of lane plus that of
    32 j, for every lane and every j < P; where 32 does not nest (48 = 3 x 16
    words after a 16) some pair breaks it."""
    T = M.TileLayout

    def nests(modes):
        suffix = 1
        for e, _, _ in reversed(modes):
            suffix *= e
            if suffix % 32 and 32 % suffix:
                return False
        return True

    cases = [((32, 32), (1, 0), True), ((16, 32), (1, 0), True), ((8, 4, 32), (2, 1, 0), True),
             ((128, 8), (1, 0), True), ((4, 32), (1, 0), True), ((6, 48), (1, 0), False),
             ((2, 3, 16), (2, 1, 0), False)]
    for sh, perm, expect in cases:
        r = len(sh)
        st = [1] * r
        for i in range(r - 2, -1, -1):
            st[i] = st[i + 1] * sh[i + 1]
        psh = [sh[q] for q in perm]
        pst = [1] * r
        for i in range(r - 2, -1, -1):
            pst[i] = pst[i + 1] * psh[i + 1]
        dst = [0] * r
        for j, q in enumerate(perm):
            dst[q] = pst[j]
        _, info = M.warp_unit_plan(T(sh, tuple(st)), T(sh, tuple(dst)), 4)
        modes, P = info["modes"], info["P"]
        assert nests(modes) == expect, sh
        split = all(_unit_point(modes, lane + 32 * j) ==
                    tuple(a + b for a, b in zip(_unit_point(modes, lane), _unit_point(modes, 32 * j)))
                    for lane in range(32) for j in range(P))
        assert split == expect, sh


def test_batched_small_planes_plan(M):
    """Batches of small transposed planes: the warp permute for units up to
    32 words a lane, except 16-byte words past 8 a lane (their words alone
    take 128 registers); planes of 4-byte words and wider of at most 16 KiB
    that the warp permute does not take go to the shared-memory transpose,
    larger ones and narrower words to the TMA tile."""
    T = M.TileLayout
    tr = lambda r, c: (T((r, c), (c, 1)), T((r, c), (1, r)))
    cases = [((32, 32), 4, "warp_permute"), ((32, 32), 2, "warp_permute"), ((32, 32), 1, "warp_permute"),
             ((32, 32), 8, "warp_permute"), ((128, 8), 4, "warp_permute"),
             # (16, 16) 16-byte units: no conflict-free swizzle, so not the warp permute
             ((16, 16), 16, "smem_transpose"), ((32, 32), 16, "smem_transpose"), ((64, 32), 4, "smem_transpose"), ((64, 64), 4, "smem_transpose"),
             ((32, 64), 2, "tile_transpose"), ((64, 128), 4, "tile_transpose")]
    for (r, c), w, name in cases:
        p = M.plan(*tr(r, c), w, 4096)
        assert p["kernel_name"] == name, ((r, c), w, p["kernel_name"])
        if name == "warp_permute":
            assert p["P"] <= 32 and not (w == 16 and p["P"] > 8)
    # forced, the warp permute still takes 16-byte units of 32 words a lane
    assert M.plan(*tr(32, 32), 16, 4096, kernel="warp_permute")["P"] == 32


def test_small_single_tiles_plan_by_word_size(M):
    """Single tiles of at most 32 KiB: the shared-memory transpose for words
    of 4 bytes and more, the tile transpose for narrower words, the vector
    copy where neither plans; never the warp classes or the staged copy."""
    T = M.TileLayout
    tr = lambda r, c: (T((r, c), (c, 1)), T((r, c), (1, r)))
    cases = [(tr(32, 32), 4, "smem_transpose"), (tr(64, 64), 4, "smem_transpose"),
             (tr(90, 90), 4, "smem_transpose"), (tr(64, 64), 8, "smem_transpose"),
             (tr(32, 32), 16, "smem_transpose"), (tr(128, 128), 2, "tile_transpose"),
             (tr(128, 256), 1, "tile_transpose"), (tr(37, 55), 2, "vec_copy"),
             ((T((8, 16, 32), (512, 32, 1)), T((8, 16, 32), (16, 1, 128))), 4, "smem_transpose")]
    for (s, d), w, name in cases:
        assert M.plan(s, d, w, 1)["kernel_name"] == name, (s, w)
    # a layout with no contiguous mode on either side: the vector copy
    assert M.plan(T((16, 16), (32, 2)), T((16, 16), (3, 48)), 4, 1)["kernel_name"] == "vec_copy"
    # past 32 KiB the general rules apply again
    assert M.plan(*tr(96, 96), 4, 1)["kernel_name"] not in ("smem_staged", "vec_copy")
    # the staged copy still plans when forced
    assert M.plan(*tr(32, 32), 4, 1, kernel="smem_staged")["kernel_name"] == "smem_staged"


def test_warp_unit_plan_matches_the_page_and_the_oracle(M):
    """P4's shared-buffer op, planned on the host: the worked example's shard
    alignment and swizzle, and for random dense and strided units the same
    alignment as the oracle's permute_align and the bank degrees the
    oracle's simulator gives at the chosen (k, shift)."""
    T = M.TileLayout
    _, info = M.warp_unit_plan(T((4, 32), (32, 1)), T((4, 32), (1, 4)), 4)
    assert info["modes"] == [(4, 32, 1), (32, 1, 4)]
    assert (info["P"], info["k"], info["shift"], info["mask"]) == (4, 2, 3, 3)
    assert info["conflict_free"] and (info["src_cosize"], info["dst_cosize"]) == (128, 128)
    # the hand-worked rank-3 case with no conflict-free choice still plans
    _, info = M.warp_unit_plan(T((2, 2, 16), (16, 32, 1)), T((2, 2, 16), (2, 1, 4)), 4)
    assert not info["conflict_free"] and max(info["conflicts_read"], info["conflicts_write"]) == 2
    rng = random.Random(11)
    for _ in range(60):
        rank = rng.randint(1, 3)
        while True:
            ext = [rng.choice([1, 2, 4, 8, 16, 32]) for _ in range(rank)]
            total = int(np.prod(ext))
            if total % 32 == 0 and total // 32 <= 32:
                break
        order_s, order_d = list(range(rank)), list(range(rank))
        rng.shuffle(order_s)
        rng.shuffle(order_d)

        def strides(order, gap):
            st, acc = [0] * rank, 1
            for m in reversed(order):
                st[m] = acc
                acc *= ext[m] + gap
            return st

        src = T(ext, strides(order_s, rng.choice([0, 0, 1])))
        dst = T(ext, strides(order_d, rng.choice([0, 0, 3])))
        w = rng.choice([1, 2, 4, 8, 16])
        _, info = M.warp_unit_plan(src, dst, w)
        extent, sstr, dstr, P = index_maps.permute_align(src, dst)
        assert info["modes"] == list(zip(extent, sstr, dstr)) and info["P"] == P
        rd, wd = banks.phase_degrees(extent, sstr, dstr, w, info["k"], info["shift"])
        assert (rd, wd) == (info["conflicts_read"], info["conflicts_write"])
        assert info["conflict_free"] == (rd == 1 and wd == 1)
    # P need not be a power of two (then only k = 0); shapes the op does not take
    _, info = M.warp_unit_plan(T((3, 32), (32, 1)), T((3, 32), (1, 3)), 4)
    assert (info["P"], info["k"]) == (3, 0)
    for bad in [(T((33,), (1,)), T((33,), (1,))),               # not a multiple of 32
                (T((64, 32), (32, 1)), T((64, 32), (1, 64))),   # P = 64 > LC_WARP_UNIT_MAX_P
                (T((4, 32), (32, 1)), T((4, 32), (1, 2)))]:     # destination not injective
        with pytest.raises(M.LayoutCopyError):
            M.warp_unit_plan(*bad, 4)


def test_build_compiles_every_source():
    """Every translation unit under csrc/ is in the build, every header it
    includes is tracked for rebuilds, and the library exports no undefined
    symbol of its own."""
    import glob
    import subprocess
    from movement_primitives_gb300 import build as b
    csrc = os.path.join(ROOT, "movement_primitives_gb300", "csrc")
    units = sorted(os.path.basename(p) for p in glob.glob(os.path.join(csrc, "*.cu")) +
                   glob.glob(os.path.join(csrc, "*.cpp")))
    assert sorted(b.SOURCES) == units
    headers = sorted(os.path.basename(p) for p in glob.glob(os.path.join(csrc, "*.h")) +
                     glob.glob(os.path.join(csrc, "*.cuh")))
    assert sorted(b.HEADERS) == headers
    out = subprocess.run(["nm", "-D", "--undefined-only", b.LIB_PATH], capture_output=True, text=True).stdout
    own = [line for line in out.splitlines() if "lc_" in line.split()[-1] or "_ZN2lc" in line]
    assert not own, own


def test_planner_is_thread_safe(M):
    """Plans from many host threads at once (the plan cache is shared)
    equal the plans made one at a time."""
    from concurrent.futures import ThreadPoolExecutor
    import workloads
    cfgs = [workloads.config(c, w, scale="small") for c, w in
            [(1, None), (2, None), (3, None), (4, 1), (4, 8), (5, None), (6, 2)]]
    args = [(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"]) for c in cfgs] * 20
    serial = [M.plan(*a) for a in args]
    with ThreadPoolExecutor(16) as ex:
        parallel = list(ex.map(lambda a: M.plan(*a), args))
    assert parallel == serial


def test_destination_injectivity_matches_brute_force(M):
    """The planner's one-to-one decision (stride splits, then enumeration)
    against a plain set of all destination offsets, on random small layouts."""
    import itertools
    import random
    rng = random.Random(17)
    T = M.TileLayout
    for _ in range(3000):
        rank = rng.randint(1, 4)
        ext = [rng.randint(1, 5) for _ in range(rank)]
        dst = [rng.choice([1, 2, 3, 4, 5, 6, 8, 9, 12, 16, 20, 24, 36]) for _ in range(rank)]
        src = []
        acc = 1
        for e in reversed(ext):
            src.insert(0, acc)
            acc *= e
        offs = [sum(i * d for i, d in zip(idx, dst)) for idx in itertools.product(*[range(e) for e in ext])]
        want = len(set(offs)) == len(offs)
        try:
            M.plan(T(tuple(ext), tuple(src)), T(tuple(ext), tuple(dst)), 4, 1)
            got = True
        except M.LayoutCopyError as e:
            assert e.status == M.STATUS["LC_ERR_NOT_INJECTIVE"], (ext, dst, e.status)
            got = False
        assert got == want, (ext, dst)


def test_gmem_smem_plan_matches_the_oracle(M):
    """lc_gmem_smem_plan (guarded partition, vector capped by the swizzle
    chunk) against oracle.index_maps.gmem_smem_partition_guarded."""
    import random
    from oracle import index_maps
    rng = random.Random(31)
    T = M.TileLayout
    checked = 0
    for _ in range(2000):
        rank = rng.randint(1, 4)
        ext = [rng.choice([1, 2, 3, 4, 8, 16, 5]) for _ in range(rank)]
        gs, acc = [0] * rank, 1
        order = list(range(rank))
        rng.shuffle(order)
        for i in reversed(order):
            gs[i] = acc
            acc *= ext[i] + rng.choice([0, 0, 2])
        ss, acc = [0] * rank, 1
        for i in reversed(range(rank)):
            ss[i] = acc
            acc *= ext[i]
        w = rng.choice([1, 2, 4, 8, 16])
        threads = rng.choice([1, 32, 96, 128, 1024])
        goff = rng.choice([0, 0, 1, 4, 16])
        swz = rng.choice([None, (2, 2, 7), (3, 4, 7), (5, 2, 7), (1, 3, 8)])
        chunk = None if swz is None else 1 << swz[1]
        try:
            want = index_maps.gmem_smem_partition_guarded(ext, gs, ss, w, threads, goff, 0, chunk)
        except index_maps.Decline:
            with pytest.raises(M.LayoutCopyError) as e:
                M.gmem_smem_plan(T(ext, gs, goff), T(ext, ss), w, threads, swz)
            assert e.value.status == M.STATUS["LC_ERR_BAD_STRIDE"]
            continue
        got = M.gmem_smem_plan(T(ext, gs, goff), T(ext, ss), w, threads, swz)
        assert got["modes"] == [tuple(m) for m in want["modes"]], (ext, gs, ss)
        assert (got["vec"], got["outer"], got["total"], got["guarded"]) == \
            (want["vec"], want["outer"], want["total"], want["guarded"]), (ext, gs, w, threads, swz)
        checked += 1
    assert checked > 1500


def test_gmem_smem_plan_refusals(M):
    T = M.TileLayout
    S = M.STATUS

    def code(*args, **kw):
        try:
            M.gmem_smem_plan(*args, **kw)
            return 0
        except M.LayoutCopyError as e:
            return e.status
    assert code(T((8,), (1,)), T((8,), (1,)), 4, 0) == S["LC_ERR_SHAPE"]
    assert code(T((8,), (1,)), T((8,), (1,)), 4, 1025) == S["LC_ERR_SHAPE"]
    assert code(T((8,), (1,)), T((8,), (1,)), 3, 32) == S["LC_ERR_ELEM_BYTES"]
    assert code(T((8,), (1,)), T((9,), (1,)), 4, 32) == S["LC_ERR_EXTENT_MISMATCH"]
    assert code(T((8,), (1,)), T((8,), (1,)), 4, 32, (3, 4, 6)) == S["LC_ERR_BAD_STRIDE"]  # not one-to-one
    assert code(T((8,), (1,)), T((8,), (1,)), 16, 32, (2, 2, 7)) == S["LC_ERR_BAD_STRIDE"]  # splits an element
    assert code(T((1 << 16, 1 << 15), (1 << 15, 1)), T((1 << 16, 1 << 15), (1 << 15, 1)), 1, 32) == S["LC_ERR_SHAPE"]


def test_mapped_copy_refusals_need_no_gpu(M):
    """lc_layout_copy_mapped refuses before launching anything: null
    pointers, layouts that do not pair, and memory the device cannot
    address (plain pageable host memory) -- each with its own status."""
    import ctypes
    import numpy as np
    lib = M._lib.lib()
    a = np.zeros(64 * 48 * 4, np.uint8)
    b = np.zeros(64 * 48 * 4, np.uint8)
    sl = M.TileLayout((64, 48), (48, 1)).to_c()
    dl = M.TileLayout((64, 48), (1, 64)).to_c()
    bad = M.TileLayout((64, 47), (48, 1)).to_c()

    def call(src, s, dst, d, w=4):
        return lib.lc_layout_copy_mapped(ctypes.c_void_p(src), ctypes.byref(s), ctypes.c_void_p(dst),
                                         ctypes.byref(d), w, 1, ctypes.c_void_p(0))
    names = M._lib.STATUS_NAMES
    assert names[call(0, sl, b.ctypes.data, dl)] == "LC_ERR_NULL"
    assert names[call(a.ctypes.data, sl, 0, dl)] == "LC_ERR_NULL"
    assert names[call(a.ctypes.data, bad, b.ctypes.data, dl)] == "LC_ERR_EXTENT_MISMATCH"
    assert names[call(a.ctypes.data, sl, b.ctypes.data, dl, 3)] == "LC_ERR_ELEM_BYTES"
    assert names[call(a.ctypes.data, sl, b.ctypes.data, dl)] == "LC_ERR_NOT_MAPPED"
    assert lib.lc_status_string(18).decode() == "a byte range is not memory the device can address"


def test_plan_tile_forms_at_their_size_boundaries(M):
    """The tile transpose's size table at its edges (bytes a side, whole
    blocks, destination rows of whole 16-byte chunks): 1-byte words direct up
    to 96 MiB, 2-byte words up to 64 MiB, then the ring up to 256 MiB, then
    TMA stores (2-byte words not with destination rows a multiple of 32 KiB
    apart); 8- and 16-byte words TMA stores up to 256 MiB, the ring above;
    4-byte words TMA stores at every size."""
    def form(rows, cols, w):
        p = M.plan(dict(shape=(rows, cols), stride=(cols, 1)), dict(shape=(rows, cols), stride=(1, rows)), w, 1,
                   "tile_transpose")
        return p["tile_form"]
    MiB = 1 << 20
    # 1-byte words: 96 MiB = 8192 x 12288
    assert form(8192, 12288, 1) == 1 and 8192 * 12288 == 96 * MiB
    assert form(8192, 12288 + 16, 1) == 0
    assert form(16384, 16384, 1) == 0 and 16384 * 16384 == 256 * MiB
    assert form(16384, 16384 + 16, 1) == 2
    # 2-byte words: 64 MiB = 4096 x 8192 words
    assert form(4096, 8192, 2) == 1 and 4096 * 8192 * 2 == 64 * MiB
    assert form(4096, 8192 + 8, 2) == 0
    assert form(8192, 16384, 2) == 0 and 8192 * 16384 * 2 == 256 * MiB
    assert form(8192 + 8, 16384, 2) == 2                      # rows 16400 bytes apart
    assert form(16384, 8192 + 8, 2) == 0                      # rows 32 KiB apart
    # 8- and 16-byte words: 256 MiB
    assert form(4096, 8192, 8) == 2 and 4096 * 8192 * 8 == 256 * MiB
    assert form(4096, 8192 + 2, 8) == 0
    assert form(4096, 4096, 16) == 2 and 4096 * 4096 * 16 == 256 * MiB
    assert form(4096, 4096 + 1, 16) == 0
    # 4-byte words at both ends
    assert form(64, 64, 4) == 2 and form(16384, 16384, 4) == 2
