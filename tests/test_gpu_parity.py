"""GPU parity: the CUDA path against the oracle, bit for bit (raw words).

Every case builds seeded host bytes, prefills the destination with the
sentinel 0xA5, runs the oracle on the host and the library on cuda:0 through
the C ABI, and compares the WHOLE destination buffer byte for byte (so
untouched bytes are checked too), then checks the device error word.
"""
import random

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def lc():
    import movement_primitives_gb300
    return movement_primitives_gb300


def _footprint(layout, n_tiles):
    return workloads.footprint_elems(layout, n_tiles)


def run_case(src_l, dst_l, w, n_tiles=1, kernel="auto", seed=0, src_pad=0, dst_pad=0,
             src_shift=0, dst_shift=0):
    """Oracle vs GPU on one copy; returns the planner's kernel name.

    ``*_shift`` moves the base pointer by that many bytes (alignment cases);
    ``*_pad`` adds slack bytes after the footprint.
    """
    ns = _footprint(src_l, n_tiles) * w + src_pad + src_shift
    nd = _footprint(dst_l, n_tiles) * w + dst_pad + dst_shift
    g = torch.Generator().manual_seed(seed)
    src_h = torch.randint(0, 256, (max(ns, 1),), generator=g, dtype=torch.uint8)
    dst_h = torch.full((max(nd, 1),), workloads.SENTINEL, dtype=torch.uint8)
    want = dst_h.numpy().copy()
    oracle.copy(src_h.numpy()[src_shift:].copy(), src_l, want[dst_shift:], dst_l, w, n_tiles)
    src_d = src_h.cuda()
    dst_d = dst_h.cuda()
    lc().layout_copy_ptr(src_d.data_ptr() + src_shift, src_l, dst_d.data_ptr() + dst_shift, dst_l,
                         w, n_tiles, kernel=kernel, stream=torch.cuda.current_stream().cuda_stream)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    got = dst_d.cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError("%d bytes differ, first at %d (got %d want %d); kernel %s"
                             % (bad.size, bad[0], got[bad[0]], want[bad[0]], kernel))
    return lc().plan(src_l, dst_l, w, n_tiles, kernel)["kernel_name"]


def L(shape, stride, offset=0, tile_stride=0):
    return dict(shape=tuple(shape), stride=tuple(stride), offset=offset, tile_stride=tile_stride)


def row_major(shape):
    st, acc = [], 1
    for e in reversed(shape):
        st.append(acc)
        acc *= e
    return tuple(reversed(st))


def permuted(shape, perm):
    """Strides of a row-major tensor of shape[perm] seen through the axes of `shape`."""
    out_shape = [shape[p] for p in perm]
    ost = row_major(out_shape)
    st = [0] * len(shape)
    for j, p in enumerate(perm):
        st[p] = ost[j]
    return tuple(st)


# ---------------------------------------------------------------------------
# the five workloads, reduced (several tiles and a ragged tail), every class
# ---------------------------------------------------------------------------

SMALL = [(1, None), (2, None), (3, None), (4, 1), (4, 2), (4, 4), (4, 8), (4, 16), (5, None),
         (6, 1), (6, 2), (6, 4), (6, 8)]


@pytest.mark.parametrize("cfg,w", SMALL)
def test_workload_small_auto(cfg, w):
    c = workloads.config(cfg, w, scale="small")
    name = run_case(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"], seed=cfg)
    expect = {1: "smem_transpose", 2: "warp_shuffle", 3: "tile_transpose", 4: "tile_transpose",
              5: "tma_copy", 6: "smem_transpose"}[cfg]
    assert name == expect


@pytest.mark.parametrize("cfg,w", SMALL)
def test_workload_small_vec_copy(cfg, w):
    c = workloads.config(cfg, w, scale="small")
    run_case(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"], kernel="vec_copy", seed=10 + cfg)


@pytest.mark.parametrize("cfg", [1, 2])
def test_workload_warp_permute_forced(cfg):
    c = workloads.config(cfg, scale="small")
    run_case(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"], kernel="warp_permute", seed=cfg)


@pytest.mark.parametrize("cfg", [1, 2])
def test_workload_warp_shuffle_or_refused(cfg):
    # workload 2's (4, 32) blocks are the shuffle's shape; workload 1's 32 x 32
    # tile is not (neither contiguous mode spans exactly 16 bytes)
    c = workloads.config(cfg, scale="small")
    if cfg == 2:
        run_case(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"], kernel="warp_shuffle", seed=cfg)
    else:
        with pytest.raises(RuntimeError):
            run_case(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"], kernel="warp_shuffle", seed=cfg)


def _shuffle_cases(w):
    """Layout pairs of the warp-shuffle class for w-byte words: V = 16 / w."""
    V = 16 // w
    out = []
    for C in sorted({V, 3 * V, 8 * V, 32 * V // min(V, 8)}):
        out.append((L((V, C), (C, 1)), L((V, C), (1, V)), 1))            # the page's shape, one block row
        out.append((L((V, C), (C, 1)), L((V, C), (1, V)), 37))           # tiles back to back, ragged count
        out.append((L((C, V), (V, 1)), L((C, V), (1, C)), 23))           # the mirror
    # gaps: source rows and destination columns padded, tiles spaced out
    out.append((L((V, 4 * V), (6 * V, 1), V, 6 * V * V + 2 * V), L((V, 4 * V), (1, 2 * V), 3 * V, 10 * V * V), 5))
    out.append((L((4 * V, V), (3 * V, 1), 0, 0), L((4 * V, V), (1, 5 * V), 2 * V, 0), 9))
    # batch modes in both orders, around the block
    out.append((L((3, V, 2, 2 * V), (4 * V * V, 2 * V, 2 * V * V, 1)),
                L((3, V, 2, 2 * V), (4 * V * V, 1, 2 * V * V, V)), 2))
    out.append((L((V, 5, 2 * V), (2 * V, 2 * V * V, 1)), L((V, 5, 2 * V), (1, 2 * V * V, V)), 3))
    return out


@pytest.mark.parametrize("w", [1, 2, 4, 8])
def test_warp_shuffle_shapes(w):
    for i, (src_l, dst_l, nt) in enumerate(_shuffle_cases(w)):
        assert lc().plan(src_l, dst_l, w, nt, "warp_shuffle")["kernel_name"] == "warp_shuffle", (src_l, dst_l)
        if nt > 1:  # (single tiles of 32 KiB and less take the small-tile rule)
            assert lc().plan(src_l, dst_l, w, nt)["kernel_name"] == "warp_shuffle", (src_l, dst_l)
        run_case(src_l, dst_l, w, nt, kernel="warp_shuffle", seed=100 * w + i)
        run_case(src_l, dst_l, w, nt, seed=200 * w + i)  # the automatic choice
    # a source base off the 16-byte grid: the planner takes another class,
    # and the copy is still exact
    V = 16 // w
    src_l, dst_l = L((V, 4 * V), (4 * V, 1)), L((V, 4 * V), (1, V))
    run_case(src_l, dst_l, w, 7, src_shift=w, seed=300 + w)
    with pytest.raises(RuntimeError):
        run_case(src_l, dst_l, w, 7, src_shift=w, kernel="warp_shuffle", seed=300 + w)


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_tile_transpose_ragged(w):
    # row strides of 16-byte multiples (TMA), extents off the tile grid
    for r, c in [(1008, 1104), (48, 560), (272, 144), (256, 128), (16, 16)]:
        assert run_case(L((r, c), (c, 1)), L((r, c), (1, r)), w, kernel="tile_transpose",
                        seed=r + c) == "tile_transpose"
    # strides TMA cannot take: the automatic choice still gets it right
    for r, c in [(37, 555), (257, 129), (3, 1000)]:
        run_case(L((r, c), (c, 1)), L((r, c), (1, r)), w, seed=r * c)


@pytest.mark.parametrize("w", [1, 2])
def test_tile_transpose_direct_form(w):
    """Whole V x V blocks of 1- and 2-byte words: the direct form of the tile
    transpose (plan stages 0; 16-byte loads straight into registers, no TMA,
    no shared memory).  Extents off the warp tile, padded rows, offsets, tile
    strides with gaps and up to three batch modes, each against the oracle;
    ragged extents beside them keep the TMA ring."""
    V = 16 // w

    def check(src_l, dst_l, n_tiles=1, direct=True, seed=0):
        p = lc().plan(src_l, dst_l, w, n_tiles, "tile_transpose")
        assert (p["stages"] == 0) == direct, (src_l, dst_l, p["stages"])
        # sentinel bytes after the destination catch writes past its last row
        assert run_case(src_l, dst_l, w, n_tiles, kernel="tile_transpose", seed=seed,
                        dst_pad=1024) == "tile_transpose"

    for r, c in [(V, V), (V, 3 * V), (9 * V, 5 * V), (144, 80), (1024, 1040), (2000, 336), (128 + V, 64 + V)]:
        check(L((r, c), (c, 1)), L((r, c), (1, r)), seed=r + c)
        check(L((r, c), (c + V, 1), 3 * V), L((r, c), (1, r + 2 * V), 5 * V), seed=r * c)  # padded rows, offsets
    # tiles with gaps between them; a batch mode; three batch modes that do not merge
    check(L((48, 32), (32, 1), V, 48 * 32 + 4 * V), L((48, 32), (1, 48), 0, 48 * 32 + 2 * V), n_tiles=3, seed=5)
    sh = (3, 4 * V, 6 * V)
    check(L(sh, row_major(sh)), L(sh, permuted(sh, (0, 2, 1))), seed=6)
    sh = (2, 3, 5, 2 * V, 3 * V)
    check(L(sh, row_major(sh)), L(sh, permuted(sh, (2, 1, 0, 4, 3))), seed=7)
    # ragged extents with 16-byte rows: the TMA ring
    for r, c in [(9 * V, 5 * V - 1), (9 * V - 1, 5 * V), (100 + V // 2, 77)]:
        check(L((r, c), (((c + V - 1) // V) * V, 1)), L((r, c), (1, ((r + V - 1) // V) * V)), direct=False,
              seed=r + 3 * c)


def test_tile_transpose_tma_store_form():
    """4-byte transposes whose destination rows are whole 16-byte chunks: the
    ring whose output tiles leave by TMA tensor stores (tile_form 2), with
    ragged source rows, extents off the 256 x 32 tile, padded rows, offsets,
    tile strides with gaps and up to three batch modes; sentinel bytes after
    the destination catch any write past its last row.  Destination rows
    that end inside a 16-byte chunk keep thread stores (form 0)."""
    w = 4

    def check(src_l, dst_l, n_tiles=1, form=2, seed=0):
        p = lc().plan(src_l, dst_l, w, n_tiles, "tile_transpose")
        assert p["tile_form"] == form, (src_l, dst_l, p["tile_form"])
        assert run_case(src_l, dst_l, w, n_tiles, kernel="tile_transpose", seed=seed,
                        dst_pad=4096) == "tile_transpose"

    for r, c in [(4, 4), (64, 36), (256, 32), (300, 33), (1024, 70), (520, 1000)]:
        check(L((r, c), (((c + 3) // 4) * 4, 1)), L((r, c), (1, r)), seed=r + c)
        check(L((r, c), (((c + 3) // 4) * 4 + 8, 1), 12), L((r, c), (1, r + 4), 8), seed=r * c)
    check(L((48, 30), (32, 1), 4, 48 * 32 + 16), L((48, 30), (1, 48), 0, 48 * 30 + 8), n_tiles=3, seed=5)
    sh = (3, 260, 40)
    check(L(sh, row_major(sh)), L(sh, permuted(sh, (0, 2, 1))), seed=6)
    sh = (2, 3, 5, 36, 20)
    check(L(sh, row_major(sh)), L(sh, permuted(sh, (2, 1, 0, 4, 3))), seed=7)
    for r, c in [(61, 36), (257, 33), (3, 40)]:
        check(L((r, c), (((c + 3) // 4) * 4, 1)), L((r, c), (1, ((r + 3) // 4) * 4)), form=0, seed=r + 3 * c)
    # the automatic choice on a whole-chunk case
    assert run_case(L((1024, 520), (520, 1)), L((1024, 520), (1, 1024)), w, dst_pad=4096, seed=9) == "tile_transpose"


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_smem_transpose_any_alignment(w):
    # whole tiles and ragged edges in both modes; aligned and unaligned rows
    for r, c in [(37, 555), (257, 129), (3, 1000), (32, 32), (64, 96), (65, 63), (2, 3),
                 (130, 250), (129, 241), (256, 240), (200, 61), (130, 600), (64, 252), (128, 124),
                 (70, 505)]:
        run_case(L((r, c), (c, 1)), L((r, c), (1, r)), w, kernel="smem_transpose", seed=r + c)
    # a single non-unit mode has nothing to transpose: the forced class declines
    with pytest.raises(lc().LayoutCopyError):
        run_case(L((1, 2), (2, 1)), L((1, 2), (1, 1)), w, kernel="smem_transpose")
    # offsets off every alignment grid, tile strides with gaps, batch modes
    run_case(L((45, 70), (71, 1), 3, 3300), L((45, 70), (1, 47), 5, 3400), w, n_tiles=3,
             kernel="smem_transpose", seed=w)
    sh = (3, 5, 33, 31)
    run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (1, 0, 3, 2))), w, kernel="smem_transpose", seed=9)
    # misaligned base pointers: the automatic choice takes one of the
    # transpose classes (or, for a small single tile of narrow words that
    # the tile transpose cannot take, the vector copy)
    assert run_case(L((64, 96), (96, 1)), L((64, 96), (1, 64)), w, src_shift=w if w < 16 else 0,
                    dst_shift=0) in ("smem_transpose", "tile_transpose", "vec_copy")


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_tma_copy_layouts(w):
    # axis permutes that keep the last axis: boxes of whole runs, ragged outer modes
    for sh, perm in [((8, 3, 64), (1, 0, 2)), ((5, 37, 3, 96), (2, 0, 1, 3)), ((7, 9, 48), (1, 0, 2)),
                     ((3, 4, 5, 2, 64), (3, 2, 0, 1, 4))]:
        if (sh[-1] * w) % 16 or sh[-1] * w < 64:
            continue
        assert run_case(L(sh, row_major(sh)), L(sh, permuted(sh, perm)), w, kernel="tma_copy",
                        seed=sum(sh)) == "tma_copy"
    # runs longer than one box (boxes of 256 elements, several per run)
    sh = (6, 1024)
    run_case(L(sh, (1040, 1)), L(sh, (1024 + 16, 1)), w, kernel="tma_copy", seed=w)
    # strided slices with offsets and tiles spaced apart on both sides
    run_case(L((10, 64), (96, 1), 32, 1280), L((10, 64), (80, 1), 16, 1024), w, n_tiles=5,
             kernel="tma_copy", seed=3 * w)
    # the automatic choice takes it for a head permute (B, S, H, D) -> (B, H, S, D)
    sh = (2, 33, 6, 64)
    assert run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (0, 2, 1, 3))), w, seed=7) == "tma_copy"


# ---------------------------------------------------------------------------
# layouts beyond the workloads
# ---------------------------------------------------------------------------

def test_batched_transposes_with_batch_modes():
    # (B, M, N) -> (B, N, M): one batch mode on the tile path
    for w in (1, 2, 4, 8, 16):
        sh = (3, 80, 144)  # 16-byte row strides for every width
        assert run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (0, 2, 1))), w, seed=w) \
            == "tile_transpose"
        sh = (3, 70, 130)  # unaligned rows: correctness only
        run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (0, 2, 1))), w, seed=w)
    # three batch modes (rank 5)
    sh = (2, 3, 2, 40, 72)
    run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (0, 1, 2, 4, 3))), 2, kernel="tile_transpose")
    # batch modes in swapped order on the destination
    sh = (4, 5, 64, 48)
    run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (1, 0, 3, 2))), 4, kernel="tile_transpose")


def test_warp_permute_units_with_gaps_and_tiles():
    # 4x32 units, tiles spaced apart (tile_stride > cosize) on both sides
    sh = (4, 32)
    run_case(L(sh, (32, 1), 16, 256), L(sh, (1, 4), 32, 160), 4, n_tiles=37, kernel="warp_permute")
    # units whose destination order is a 3-D permutation
    sh = (2, 4, 16)
    for w in (1, 2, 4, 8, 16):
        run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (2, 0, 1))), w, n_tiles=9,
                 kernel="warp_permute", seed=w)


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_warp_permute_large_nested_units(w):
    """Units of 16 and 32 words a lane whose radix nests 32 (offsets formed
    by shuffles as they are used): 999 tiles packed back to back (an odd
    last group), and tiles with chunk-sized gaps between them (units found
    by division), against the oracle."""
    for i, sh in enumerate([(16, 32), (32, 32), (8, 4, 32), (32, 16)]):
        perm = tuple(reversed(range(len(sh))))
        src_l, dst_l = L(sh, row_major(sh)), L(sh, permuted(sh, perm))
        assert lc().plan(src_l, dst_l, w, 999, "warp_permute")["kernel_name"] == "warp_permute"
        run_case(src_l, dst_l, w, n_tiles=999, kernel="warp_permute", seed=40 * w + i)
        n = 1
        for e in sh:
            n *= e
        v = 16 // w  # words per 16-byte chunk: units start on chunks
        gap_s, gap_d = L(sh, row_major(sh), 2 * v, n + 5 * v), L(sh, permuted(sh, perm), v, n + 3 * v)
        run_case(gap_s, gap_d, w, n_tiles=7, kernel="warp_permute", seed=41 * w + i)


@pytest.mark.parametrize("w", [1, 2, 4])
def test_warp_permute_prefetch_cycles_slots(w):
    """Enough 32 x 32 units that every warp of the bulk-prefetch form takes
    about three groups (4 KiB each): its two slots alternate and each slot's
    barrier completes more than one phase; the whole batch against the
    oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    warps = sms * 3 * 8  # 3 CTAs of 8 warps a SM at most
    units_per_group = 4096 // (1024 * w)
    n_tiles = 3 * warps * units_per_group + 5  # and a ragged last group
    sh = (32, 32)
    src_l, dst_l = L(sh, row_major(sh)), L(sh, permuted(sh, (1, 0)))
    assert run_case(src_l, dst_l, w, n_tiles=n_tiles, seed=70 + w) == "warp_permute"


def test_axis_permutes_auto():
    rng = random.Random(5)
    for _ in range(25):
        rank = rng.randint(2, 5)
        sh = tuple(rng.choice([1, 2, 3, 5, 8, 16, 33]) for _ in range(rank))
        perm = list(range(rank))
        rng.shuffle(perm)
        w = rng.choice([1, 2, 4, 8, 16])
        run_case(L(sh, row_major(sh)), L(sh, permuted(sh, perm)), w, seed=rng.randrange(1000))


def _random_layout_pair(rng):
    rank = rng.randint(1, 4)
    ext = [rng.choice([1, 2, 3, 4, 7, 8, 16, 32, 33]) for _ in range(rank)]
    so = list(range(rank)); rng.shuffle(so)
    do = list(range(rank)); rng.shuffle(do)

    def strides(order, gap_p):
        st = [0] * rank
        acc = 1
        for m in reversed(order):
            acc *= rng.choice([1, 2]) if rng.random() < gap_p else 1
            st[m] = acc
            acc *= ext[m]
        return st

    ss = strides(so, 0.3)
    if rng.random() < 0.15:
        ss[rng.randrange(rank)] = 0  # broadcast read
    ds = strides(do, 0.3)
    n_tiles = rng.choice([1, 1, 2, 5])
    src = L(ext, ss, rng.randint(0, 9), 0)
    dst = L(ext, ds, rng.randint(0, 9), rng.choice([0, 0, None]) or 0)
    return src, dst, rng.choice([1, 2, 4, 8, 16]), n_tiles


@pytest.mark.parametrize("seed", range(6))
def test_random_layouts(seed):
    rng = random.Random(1000 + seed)
    for i in range(40):
        src, dst, w, n_tiles = _random_layout_pair(rng)
        run_case(src, dst, w, n_tiles, seed=i)
        run_case(src, dst, w, n_tiles, kernel="vec_copy", seed=i)


@pytest.mark.parametrize("seed", range(8))
def test_tile_transpose_fuzz(seed):
    """Seeded transposes through the three forms of the tile class: the
    direct form (1- and 2-byte words, whole V x V blocks), the swizzled ring
    with line stores (short boxes of 1-, 2- and 4-byte words) and the plain
    ring (8- and 16-byte words), with ragged extents, padded rows, offsets,
    tile strides and up to two batch modes, forced and automatic, each
    against the oracle."""
    rng = random.Random(4242 + seed)

    def up(n, m):
        return (n + m - 1) // m * m

    for i in range(24):
        w = rng.choice([1, 2, 4, 8, 16])
        V = 16 // w
        whole = rng.random() < 0.5
        if whole:
            r, c = V * rng.randint(2 if V == 1 else 1, 40), V * rng.randint(2 if V == 1 else 1, 40)
        else:
            r, c = rng.randint(2, 40 * V), rng.randint(2, 40 * V)
        sc = up(c, V) + V * rng.randint(0, 2)        # source row stride (16-byte multiple)
        dr = up(r, V) + V * rng.randint(0, 2)        # destination row stride
        batch = [rng.randint(2, 3) for _ in range(rng.randint(0, 2))]
        sh = tuple(batch) + (r, c)
        sst, acc = [sc, 1], r * sc + V * rng.randint(0, 1)
        for e in reversed(batch):
            sst.insert(0, acc)
            acc *= e
        order = list(range(len(batch)))
        rng.shuffle(order)                           # batch modes in another order on the destination
        dst_batch = [0] * len(batch)
        dacc = c * dr
        for k in reversed(order):
            dst_batch[k] = dacc
            dacc *= batch[k]
        dst_st = tuple(dst_batch) + (1, dr)
        n_tiles = rng.choice([1, 1, 2])
        src_l = L(sh, tuple(sst), V * rng.randint(0, 3), acc + V if n_tiles > 1 else 0)
        dst_l = L(sh, dst_st, V * rng.randint(0, 3), dacc + 2 * V if n_tiles > 1 else 0)
        p = lc().plan(src_l, dst_l, w, n_tiles, "tile_transpose")
        direct = w <= 2 and r % V == 0 and c % V == 0
        assert (p["stages"] == 0) == direct, (sh, w, p["stages"])
        tstore = (r * w) % 16 == 0 and w >= 4                # small copies: 4-, 8- and 16-byte words
        assert p["tile_form"] == (1 if direct else 2 if tstore else 0), (sh, w, p["tile_form"])
        assert run_case(src_l, dst_l, w, n_tiles, kernel="tile_transpose", seed=i, dst_pad=1024) == "tile_transpose"
        run_case(src_l, dst_l, w, n_tiles, seed=100 + i, dst_pad=1024)  # the automatic choice


def test_edge_cases():
    # empty copies launch nothing and touch nothing
    run_case(L((0, 4), (4, 1)), L((0, 4), (1, 4)), 4)
    run_case(L((4, 4), (4, 1)), L((4, 4), (1, 4)), 4, n_tiles=0)
    # one word
    run_case(L((1,), (1,)), L((1,), (1,)), 16)
    # unit modes ignored when pairing, different ranks
    run_case(L((1, 5, 1, 7), (99, 7, 3, 1)), L((5, 7), (1, 5)), 2)
    # rank 8
    sh = (2, 2, 2, 2, 2, 2, 2, 3)
    run_case(L(sh, row_major(sh)), L(sh, permuted(sh, (7, 6, 5, 4, 3, 2, 1, 0))), 4)
    # broadcast source (stride 0 everywhere)
    run_case(L((6, 9), (0, 0), 3), L((6, 9), (9, 1)), 8)
    # identity copies of every width, odd sizes
    for w in (1, 2, 4, 8, 16):
        for n in (1, 15, 4097):
            run_case(L((n,), (1,)), L((n,), (1,)), w, seed=n)


@pytest.mark.parametrize("w,rows,cols,form", [(1, 16384, 16640, 2), (1, 16383, 16640, 0), (2, 8192, 16640, 2),
                                               (2, 8191, 16640, 0), (4, 8192, 8320, 2), (4, 8191, 8320, 0)])
def test_tile_transpose_tall_boxes(w, rows, cols, form):
    """Transposes just past 256 MiB a side: with destination rows of whole
    16-byte chunks the TMA-store form, with rows that end inside one the
    ring's 256-row boxes (and the 64-bit index path); whole buffer against
    the oracle."""
    pitch = (rows + 15) // 16 * 16
    src_l, dst_l = L((rows, cols), (cols, 1)), L((rows, cols), (1, pitch))
    assert rows * cols * w > 256 << 20
    p = lc().plan(src_l, dst_l, w, 1)
    assert p["kernel_name"] == "tile_transpose" and p["tile_form"] == form and p["tile_rows"] == 256
    c = dict(src=src_l, dst=dst_l, elem_bytes=w, n_tiles=1, kind="bytes", seed=700 + w, cfg=4, name="tall")
    src_h = workloads.make_src(c)
    src_d = src_h.cuda()
    dst_d = workloads.make_dst(c, device="cuda")
    lc().layout_copy(src_d, src_l, dst_d, dst_l, elem_bytes=w)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    _assert_same_bytes(dst_d.cpu().numpy(), _oracle_full(c, src_h.numpy()), "tall w=%d" % w)


@pytest.mark.parametrize("w,side,form", [(1, 11520, 0), (2, 12288, 2), (8, 4096, 2), (16, 4096, 2)])
def test_tile_transpose_forms_at_size(w, side, form):
    """The tile transpose's form chosen by width and size, at sizes no other
    test reaches: 1-byte words at 126 MiB a side (the swizzled ring), 2-byte
    words at 288 MiB (TMA stores), 8- and 16-byte words at 128 and 256 MiB
    (TMA stores); whole buffer against the oracle."""
    src_l, dst_l = L((side, side), (side, 1)), L((side, side), (1, side))
    p = lc().plan(src_l, dst_l, w, 1)
    assert p["kernel_name"] == "tile_transpose" and p["tile_form"] == form
    c = dict(src=src_l, dst=dst_l, elem_bytes=w, n_tiles=1, kind="bytes", seed=800 + w, cfg=4, name="forms")
    src_h = workloads.make_src(c)
    src_d = src_h.cuda()
    dst_d = workloads.make_dst(c, device="cuda")
    lc().layout_copy(src_d, src_l, dst_d, dst_l, elem_bytes=w)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    _assert_same_bytes(dst_d.cpu().numpy(), _oracle_full(c, src_h.numpy()), "forms w=%d" % w)


def test_injective_destination_beyond_enumeration():
    # 2^25 + 2^24 one-byte words whose destination strides do not nest:
    # offsets k + 2^23 (2i + 3j), one-to-one by the stride split (the planner
    # enumerates only the 3 x 2 quotient)
    big = (3, 2, 1 << 23)
    run_case(L(big, (2 << 23, 1 << 23, 1)), L(big, (1 << 24, 3 << 23, 1)), 1, seed=77)


def test_misaligned_bases_still_exact():
    # base pointers off the 16-byte grid: the planner must pick narrower paths
    for w, shift in [(1, 1), (2, 2), (4, 4), (8, 8)]:
        run_case(L((64, 96), (96, 1)), L((64, 96), (1, 64)), w, src_shift=shift)
        run_case(L((64, 96), (96, 1)), L((64, 96), (1, 64)), w, dst_shift=shift)
        run_case(L((4, 32), (32, 1)), L((4, 32), (1, 4)), w, n_tiles=11, src_shift=shift)
        run_case(L((8, 256), (256, 1)), L((8, 256), (256, 1)), w, dst_shift=shift)


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------

FULL = [(1, None), (2, None), (3, None), (4, 1), (4, 2), (4, 4), (4, 8), (4, 16), (5, None),
        (6, 1), (6, 2), (6, 4), (6, 8)]


def _oracle_full(c, src_np):
    """The oracle over the whole workload, split over the host's cores (tiles,
    or slabs of the outermost mode, each its own oracle copy)."""
    import bench
    want = workloads.make_dst(c).numpy()
    bench.run_oracle(c, src_np, want, bench.host_cores())
    return want


def _assert_same_bytes(got, want, what):
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError("%s: %d bytes differ, first at %d (got %d want %d)"
                             % (what, bad.size, bad[0], got[bad[0]], want[bad[0]]))


@pytest.mark.parametrize("cfg,w", FULL)
def test_workload_full_size_exact(cfg, w):
    """Full size, the benchmark's launch: the WHOLE destination buffer equals
    the oracle's byte for byte (sentinel bytes included), then 2^20 sampled
    points are checked once more against the oracle's offsets."""
    c = workloads.config(cfg, w)
    src_h = workloads.make_src(c)
    src_d = src_h.cuda()
    dst_d = workloads.make_dst(c, device="cuda")
    lc().layout_copy(src_d, c["src"], dst_d, c["dst"], n_tiles=c["n_tiles"], elem_bytes=c["elem_bytes"])
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    want = _oracle_full(c, src_h.numpy())
    _assert_same_bytes(dst_d.cpu().numpy(), want, c["name"])
    del want
    wbytes = c["elem_bytes"]
    n = workloads.logical_elems(c)
    rng = np.random.default_rng(cfg * 100 + wbytes)
    pts = rng.integers(0, n, size=min(n, 1 << 20), dtype=np.int64)
    pts[:2] = [0, n - 1]
    so, do = oracle.offsets_of(c["src"], c["dst"], c["n_tiles"], pts)
    sv, dv = src_d.view(-1, wbytes), dst_d.view(-1, wbytes)
    assert torch.equal(sv[torch.from_numpy(so).cuda()], dv[torch.from_numpy(do).cuda()])
    del src_d, dst_d, sv, dv


# ---------------------------------------------------------------------------
# errors and the bounded-wait failure path
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_recovers():
    lc().debug_wait_timeout(200_000)  # 0.2 ms on a barrier nothing arrives at
    st, detail = lc().last_device_error()
    assert st == 12 and (detail & 0xff) == 12
    assert lc().last_device_error() == (0, 0)  # cleared; the context still works
    run_case(L((32, 32), (32, 1)), L((32, 32), (1, 32)), 4)


def test_pointer_errors():
    M = lc()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    l4 = L((16, 16), (16, 1))
    with pytest.raises(M.LayoutCopyError) as e:
        M.layout_copy_ptr(p, l4, p + 512, l4, 4)  # ranges [0,1024) and [512,1536)
    assert e.value.status == M.STATUS["LC_ERR_OVERLAP"]
    with pytest.raises(M.LayoutCopyError) as e:
        M.layout_copy_ptr(p + 2, l4, p + 4096, l4, 4)
    assert e.value.status == M.STATUS["LC_ERR_ALIGN"]
    with pytest.raises(M.LayoutCopyError) as e:
        M.layout_copy_ptr(0, l4, p, l4, 4)
    assert e.value.status == M.STATUS["LC_ERR_NULL"]
    with pytest.raises(ValueError):
        M.layout_copy(buf[:100], l4, buf[1000:], l4, elem_bytes=4)  # tensor too small


# ---------------------------------------------------------------------------
# in place: P4's aliasing case (the destination image is the source image)
# ---------------------------------------------------------------------------

def run_in_place(lay_src, lay_dst, w, n_tiles, seed=0):
    n = _footprint(lay_src, n_tiles) * w
    g = torch.Generator().manual_seed(seed)
    buf_h = torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8)
    want = buf_h.numpy().copy()                    # untouched bytes keep their values
    oracle.copy(buf_h.numpy().copy(), lay_src, want, lay_dst, w, n_tiles)  # reads see the snapshot
    buf = buf_h.cuda()
    lc().layout_copy_ptr(buf.data_ptr(), lay_src, buf.data_ptr(), lay_dst, w, n_tiles,
                         stream=torch.cuda.current_stream().cuda_stream)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    assert np.array_equal(buf.cpu().numpy(), want)


def test_in_place_unit_permutes():
    sh = (2, 1, 4, 32)
    run_in_place(L(sh, (128, 128, 32, 1)), L(sh, (128, 128, 1, 4)), 4, n_tiles=(1 << 12) + 3, seed=1)
    # gapped tiles (same tile stride on both sides), every width
    for w in (1, 2, 4, 8, 16):
        run_in_place(L((4, 32), (32, 1), 32, 192), L((4, 32), (1, 4), 32, 192), w, n_tiles=57, seed=w)
    # one 32 x 32 tile transposed in place
    run_in_place(L((32, 32), (32, 1)), L((32, 32), (1, 32)), 4, n_tiles=1, seed=7)


# ---------------------------------------------------------------------------
# host buffers through the pipelined entry point
# ---------------------------------------------------------------------------

def run_host_case(src_l, dst_l, w, n_tiles, seed=0, staging_bytes=None):
    ns = _footprint(src_l, n_tiles) * w
    nd = _footprint(dst_l, n_tiles) * w
    g = torch.Generator().manual_seed(seed)
    src_h = torch.randint(0, 256, (ns,), generator=g, dtype=torch.uint8).pin_memory()
    dst_h = torch.full((nd,), workloads.SENTINEL, dtype=torch.uint8).pin_memory()
    want = dst_h.numpy().copy()
    oracle.copy(src_h.numpy(), src_l, want, dst_l, w, n_tiles)
    staging = None
    if staging_bytes is not None:
        staging = torch.empty(staging_bytes, dtype=torch.uint8, device="cuda")
    lc().layout_copy_host(src_h, src_l, dst_h, dst_l, n_tiles=n_tiles, elem_bytes=w, staging=staging)
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(dst_h.numpy(), want)


def test_host_buffers_pipelined():
    c = workloads.config(2, scale="small")
    run_host_case(c["src"], c["dst"], 4, c["n_tiles"], seed=1)
    # a small staging buffer: more, smaller chunks
    run_host_case(c["src"], c["dst"], 4, c["n_tiles"], seed=2, staging_bytes=1 << 16)
    # destination with holes between tiles: bytes outside the image survive
    run_host_case(L((4, 32), (32, 1)), L((4, 32), (1, 4), 8, 200), 2, 301, seed=3)
    # one tile (no chunking): a transpose and an axis permute
    c = workloads.config(3, scale="small")
    run_host_case(c["src"], c["dst"], 2, 1, seed=4)
    c = workloads.config(5, scale="small")
    run_host_case(c["src"], c["dst"], 2, 1, seed=5)
    # batches of transposes chunked over a small staging buffer, through the
    # tile transpose's TMA-store form (4-byte words) and direct form (1-byte)
    for w, form, (r, cc) in [(4, 2, (64, 48)), (1, 1, (64, 96))]:
        src_l, dst_l = L((r, cc), (cc, 1)), L((r, cc), (1, r))
        assert lc().plan(src_l, dst_l, w, 37, "tile_transpose")["tile_form"] == form
        run_host_case(src_l, dst_l, w, 37, seed=6 + w, staging_bytes=1 << 20)


def run_mapped_case(src_l, dst_l, w, n_tiles=1, seed=0, dst_pad=256):
    ns = _footprint(src_l, n_tiles) * w
    nd = _footprint(dst_l, n_tiles) * w + dst_pad
    g = torch.Generator().manual_seed(seed)
    src_h = torch.randint(0, 256, (ns,), generator=g, dtype=torch.uint8).pin_memory()
    dst_h = torch.full((nd,), workloads.SENTINEL, dtype=torch.uint8).pin_memory()
    want = dst_h.numpy().copy()
    oracle.copy(src_h.numpy(), src_l, want, dst_l, w, n_tiles)
    lc().layout_copy_mapped(src_h, src_l, dst_h, dst_l, n_tiles=n_tiles, elem_bytes=w)
    torch.cuda.current_stream().synchronize()
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    _assert_same_bytes(dst_h.numpy(), want, "mapped")


@pytest.mark.parametrize("cfg,w", SMALL)
def test_mapped_host_buffers_workloads(cfg, w):
    """lc_layout_copy_mapped: the kernels read and write pinned host memory
    directly; every reduced workload (TMA classes replaced by plain-load
    ones) against the oracle, sentinel bytes after the destination."""
    c = workloads.config(cfg, w, scale="small")
    run_mapped_case(c["src"], c["dst"], c["elem_bytes"], c["n_tiles"], seed=cfg + (w or 0))


@pytest.mark.parametrize("seed", range(2))
def test_mapped_host_buffers_random_layouts(seed):
    """Seeded random layout pairs (ranks 1-4, gaps, broadcasts, tiles) between
    pinned host buffers through lc_layout_copy_mapped, against the oracle."""
    rng = random.Random(5000 + seed)
    for i in range(40):
        src, dst, w, n_tiles = _random_layout_pair(rng)
        run_mapped_case(src, dst, w, n_tiles, seed=i)


def test_mapped_host_buffers_edges():
    M = lc()
    # ragged transposes and batch modes through the shared-memory transpose,
    # whole 1-byte blocks through the tile transpose's direct form
    run_mapped_case(L((300, 33), (36, 1)), L((300, 33), (1, 304)), 4, seed=1)
    run_mapped_case(L((3, 64, 96), (96 * 64, 96, 1)), L((3, 64, 96), (96 * 64, 1, 64)), 1, seed=2)
    run_mapped_case(L((45, 70), (71, 1), 3, 3300), L((45, 70), (1, 47), 5, 3400), 2, n_tiles=3, seed=3)
    # a device source and a pinned host destination: both addressable
    src_l, dst_l = L((64, 48), (48, 1)), L((64, 48), (1, 64))
    src_d = torch.randint(0, 256, (64 * 48 * 4,), dtype=torch.uint8, device="cuda")
    dst_h = torch.full((64 * 48 * 4,), workloads.SENTINEL, dtype=torch.uint8).pin_memory()
    st = _lib_call_mapped(src_d.data_ptr(), src_l, dst_h.data_ptr(), dst_l, 4)
    assert st == 0
    torch.cuda.synchronize()
    want = dst_h.numpy().copy()
    oracle.copy(src_d.cpu().numpy(), src_l, want, dst_l, 4, 1)
    _assert_same_bytes(dst_h.numpy(), want, "device to mapped")
    # two device buffers: the ordinary copy (TMA classes allowed)
    dst_d = torch.full((64 * 48 * 4,), workloads.SENTINEL, dtype=torch.uint8, device="cuda")
    assert _lib_call_mapped(src_d.data_ptr(), src_l, dst_d.data_ptr(), dst_l, 4) == 0
    torch.cuda.synchronize()
    _assert_same_bytes(dst_d.cpu().numpy(), want, "device to device through the mapped entry")
    # pageable host memory is refused before anything is launched
    a = torch.zeros(64 * 48 * 4, dtype=torch.uint8)
    b = torch.zeros(64 * 48 * 4, dtype=torch.uint8).pin_memory()
    with pytest.raises(M.LayoutCopyError, match="LC_ERR_NOT_MAPPED"):
        M.layout_copy_mapped(a, src_l, b, dst_l, elem_bytes=4)
    with pytest.raises(M.LayoutCopyError, match="LC_ERR_NOT_MAPPED"):
        M.layout_copy_mapped(b, src_l, a, dst_l, elem_bytes=4)
    assert _lib_call_mapped(a.data_ptr(), src_l, b.data_ptr(), dst_l, 4) == 18


def _lib_call_mapped(src_ptr, src_l, dst_ptr, dst_l, w, n_tiles=1):
    import ctypes
    M = lc()
    sl, dl = M.TileLayout(**src_l).to_c(), M.TileLayout(**dst_l).to_c()
    return M._lib.lib().lc_layout_copy_mapped(ctypes.c_void_p(src_ptr), ctypes.byref(sl), ctypes.c_void_p(dst_ptr),
                                             ctypes.byref(dl), w, n_tiles,
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_mapped_host_buffers_full_size():
    """The benchmark's workload (2^20 scale-factor tiles, 1 GiB a side) host to
    host through lc_layout_copy_mapped: the whole destination against the
    oracle."""
    c = workloads.config(2)
    src_h = workloads.make_src(c).pin_memory()
    dst_h = workloads.make_dst(c).pin_memory()
    lc().layout_copy_mapped(src_h, c["src"], dst_h, c["dst"], n_tiles=c["n_tiles"], elem_bytes=c["elem_bytes"])
    torch.cuda.current_stream().synchronize()
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    _assert_same_bytes(dst_h.numpy(), _oracle_full(c, src_h.numpy()), "mapped full size")


def test_host_buffers_errors():
    M = lc()
    lay = L((16, 16), (16, 1))
    a = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    b = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.LayoutCopyError) as e:
        M.layout_copy_host(a, lay, b, L((16, 16), (1, 16)), elem_bytes=4, staging=small)
    assert e.value.status == M.STATUS["LC_ERR_STAGING"]
    with pytest.raises(M.LayoutCopyError) as e:
        M.layout_copy_host(a, lay, a, L((16, 16), (1, 16)), elem_bytes=4)
    assert e.value.status == M.STATUS["LC_ERR_OVERLAP"]


# ---------------------------------------------------------------------------
# window sum (cooperative fetch + stencil), against the oracle, bit for bit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("window", [1, 2, 3, 4, 5, 6, 7, 64])
def test_window_sum_matches_oracle(window):
    from oracle import stencil
    rng = np.random.default_rng(window)
    for n in (1, 5, 1024, 2047, 2048, 2049, 100003, 1 << 20):
        a_h = rng.standard_normal(n + window - 1).astype(np.float32)
        want = stencil.window_sum_f32(a_h, n, window)
        a = torch.from_numpy(a_h).cuda()
        b = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        lc().window_sum(a, b, window)
        got = b.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (n, window)


def test_window_sum_unaligned_and_page_shape():
    from oracle import stencil
    a_h = np.random.default_rng(0).standard_normal(1027 + 3).astype(np.float32)
    a = torch.from_numpy(a_h).cuda()
    b = torch.empty(1024 + 1, dtype=torch.float32, device="cuda")
    # the page's shapes (1027 -> 1024), from a base that is not 16-byte aligned
    lc().window_sum(a[1:1028], b[1:], 3)
    assert np.array_equal(b[1:].cpu().numpy(), stencil.window_sum_f32(a_h[1:1028], 1024, 3))
    # aligned input, output off the 16-byte grid (scalar stores), and the reverse
    for win in (3, 5, 9):
        n = 5000
        a2_h = np.random.default_rng(win).standard_normal(n + win).astype(np.float32)
        a2 = torch.from_numpy(a2_h).cuda()
        b2 = torch.empty(n + 1, dtype=torch.float32, device="cuda")
        lc().window_sum(a2[:n + win - 1], b2[1:], win)
        assert np.array_equal(b2[1:].cpu().numpy().view(np.uint32),
                              stencil.window_sum_f32(a2_h[:n + win - 1], n, win).view(np.uint32))
        lc().window_sum(a2[1:n + win], b2[:n], win)
        assert np.array_equal(b2[:n].cpu().numpy().view(np.uint32),
                              stencil.window_sum_f32(a2_h[1:n + win], n, win).view(np.uint32))
    with pytest.raises(lc().LayoutCopyError):
        lc().window_sum(a, a[:1000], 3)  # overlapping ranges


# ---------------------------------------------------------------------------
# P4's warp-scope permute between shared-memory buffers (lc_warp_unit_run)
# ---------------------------------------------------------------------------

def _unit_layouts(rng):
    rank = rng.randint(1, 3)
    while True:
        ext = [rng.choice([1, 2, 4, 8, 16, 32, 3]) for _ in range(rank)]
        total = int(np.prod(ext))
        if total % 32 == 0 and 1 <= total // 32 <= 32:
            break
    so, do = list(range(rank)), list(range(rank))
    rng.shuffle(so)
    rng.shuffle(do)

    def strides(order, gap):
        st, acc = [0] * rank, 1
        for m in reversed(order):
            st[m] = acc
            acc *= ext[m] + gap
        return st

    return L(ext, strides(so, rng.choice([0, 0, 1]))), L(ext, strides(do, rng.choice([0, 0, 2])))


@pytest.mark.parametrize("in_place", [False, True])
def test_warp_unit_on_shared_buffers(in_place):
    M = lc()
    rng = random.Random(21 + in_place)
    done = 0
    while done < 40:
        src_l, dst_l = _unit_layouts(rng)
        w = rng.choice([1, 2, 4, 8, 16])
        plan, info = M.warp_unit_plan(src_l, dst_l, w)
        scos, dcos = info["src_cosize"], info["dst_cosize"]
        if max(scos, dcos) * w > 8192 or (in_place and scos < dcos):
            continue
        n = rng.choice([1, 3, 37])
        g = torch.Generator().manual_seed(done)
        src_h = torch.randint(0, 256, (n * scos * w,), generator=g, dtype=torch.uint8)
        if in_place:  # the destination buffer starts as the source buffer
            start = np.concatenate([src_h.numpy()[i * scos * w:(i * scos + dcos) * w] for i in range(n)])
        else:
            start = np.full(n * dcos * w, workloads.SENTINEL, np.uint8)
        want = start.copy()
        oracle.copy(src_h.numpy(), dict(src_l, tile_stride=scos), want, dict(dst_l, tile_stride=dcos), w, n)
        src_d = src_h.cuda()
        dst_d = torch.from_numpy(start.copy()).cuda()
        M.warp_unit_run(src_d, dst_d, plan, w, n, in_place=in_place,
                        stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        got = dst_d.cpu().numpy()
        assert np.array_equal(got, want), (src_l, dst_l, w, n, info)
        done += 1


@pytest.mark.parametrize("shape", [(6, 48), (2, 3, 16), (3, 32), (32, 32), (4, 8, 32)])
def test_warp_units_whose_radix_does_or_does_not_nest_32(shape):
    """Lane offsets come from shuffles where 32 lies on the divisibility chain
    of the unit's suffix products ((3, 32), (32, 32), (4, 8, 32)) and from a
    per-step unflatten where it does not ((6, 48): 48; (2, 3, 16): 48): both,
    in the global warp permute and in the shared-buffer op, against the
    oracle."""
    M = lc()
    perm = tuple(reversed(range(len(shape))))
    src_l, dst_l = L(shape, row_major(shape)), L(shape, permuted(shape, perm))
    for w in (1, 4, 16):
        assert run_case(src_l, dst_l, w, n_tiles=5, kernel="warp_permute", seed=w) == "warp_permute"
        plan, info = M.warp_unit_plan(src_l, dst_l, w)
        scos, dcos = info["src_cosize"], info["dst_cosize"]
        if max(scos, dcos) * w > 8192:
            continue
        n = 7
        g = torch.Generator().manual_seed(w)
        src_h = torch.randint(0, 256, (n * scos * w,), generator=g, dtype=torch.uint8)
        want = np.full(n * dcos * w, workloads.SENTINEL, np.uint8)
        oracle.copy(src_h.numpy(), dict(src_l, tile_stride=scos), want, dict(dst_l, tile_stride=dcos), w, n)
        dst_d = torch.from_numpy(np.full(n * dcos * w, workloads.SENTINEL, np.uint8)).cuda()
        M.warp_unit_run(src_h.cuda(), dst_d, plan, w, n, stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(dst_d.cpu().numpy(), want), (shape, w)


def test_warp_unit_run_refusals():
    M = lc()
    plan, _ = M.warp_unit_plan(L((4, 32), (32, 1)), L((4, 32), (1, 4)), 4)
    buf = torch.zeros(4 * 128 * 4 + 16, dtype=torch.uint8, device="cuda")
    out = torch.zeros(4 * 128 * 4 + 16, dtype=torch.uint8, device="cuda")
    lib, stream = M._lib.lib(), torch.cuda.current_stream().cuda_stream
    import ctypes
    run = lambda s, d, n, ip=0, p=plan: lib.lc_warp_unit_run(ctypes.c_void_p(s), ctypes.c_void_p(d),
                                                              ctypes.byref(p), 4, n, ip, ctypes.c_void_p(stream))
    assert run(buf.data_ptr(), out.data_ptr(), 4) == 0
    assert run(buf.data_ptr() + 4, out.data_ptr(), 4) == M.STATUS["LC_ERR_ALIGN"]
    assert run(buf.data_ptr(), buf.data_ptr() + 16, 2) == M.STATUS["LC_ERR_OVERLAP"]
    bad = M._lib.CWarpUnit.from_buffer_copy(plan)
    bad.P = 5  # extents no longer hold 32 * P words
    assert run(buf.data_ptr(), out.data_ptr(), 1, p=bad) == M.STATUS["LC_ERR_SHAPE"]
    bad = M._lib.CWarpUnit.from_buffer_copy(plan)
    bad.mask, bad.k = 7, 3  # the XOR would leave [0, P)
    assert run(buf.data_ptr(), out.data_ptr(), 1, p=bad) == M.STATUS["LC_ERR_SHAPE"]
    torch.cuda.synchronize()
    st, detail = M.last_device_error()
    assert st == 0, detail


def test_copies_capture_into_a_cuda_graph():
    """After one call per kernel class (which sets the kernel attributes and
    caches the plan), the copy launches nothing but its kernel on the given
    stream, so it can be captured into a CUDA graph and replayed."""
    M = lc()
    cases = [workloads.config(2, scale="small"), workloads.config(3, scale="small"),
             workloads.config(5, scale="small"), workloads.config(6, 2, scale="small"),
             workloads.config(8, scale="small")]  # the last through lc_layout_copy_loop
    for cfg in cases:
        src_h = workloads.make_src(cfg)
        want = workloads.make_dst(cfg).numpy().copy()
        oracle.copy(src_h.numpy(), cfg["src"], want, cfg["dst"], cfg["elem_bytes"], cfg["n_tiles"])
        src = src_h.cuda()
        dst = workloads.make_dst(cfg, device="cuda")
        side = torch.cuda.Stream()
        if "loop" in cfg:
            run = lambda: M.layout_copy_loop_ptr(src.data_ptr(), cfg["src"], dst.data_ptr(), cfg["dst"],
                                                 cfg["elem_bytes"], cfg["loop"], cfg["n_tiles"],
                                                 stream=side.cuda_stream)
        else:
            run = lambda: M.layout_copy_ptr(src.data_ptr(), cfg["src"], dst.data_ptr(), cfg["dst"],
                                            cfg["elem_bytes"], cfg["n_tiles"], stream=side.cuda_stream)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run()  # warm-up outside the capture
        torch.cuda.synchronize()
        dst.fill_(workloads.SENTINEL)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            run()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(dst.cpu().numpy(), want), cfg["name"]


# ---------------------------------------------------------------------------
# loop-layout override: the words against the definition, the partition (the
# trace of who moved what) against the oracle's (thread, slot) of each point
# ---------------------------------------------------------------------------

def _loop_trace_want(src_l, dst_l, loop, n_tiles):
    extents = [m[0] for m in oracle.paired_modes(src_l, dst_l)]
    T, L_ = oracle.index_maps.loop_layout_sizes(extents, loop)
    N = int(np.prod(extents))
    one = np.empty(N, np.int64)
    for flat in range(N):
        t, slot = oracle.index_maps.loop_layout_owner(flat, loop)
        one[flat] = t * L_ + slot
    return np.tile(one, n_tiles)


def run_loop_case(src_l, dst_l, w, loop, n_tiles=1, seed=0, src_shift=0, dst_shift=0):
    ns = _footprint(src_l, n_tiles) * w + src_shift
    nd = _footprint(dst_l, n_tiles) * w + dst_shift
    g = torch.Generator().manual_seed(seed)
    src_h = torch.randint(0, 256, (max(ns, 1),), generator=g, dtype=torch.uint8)
    dst_h = torch.full((max(nd, 1),), workloads.SENTINEL, dtype=torch.uint8)
    want = dst_h.numpy().copy()
    oracle.copy(src_h.numpy()[src_shift:].copy(), src_l, want[dst_shift:], dst_l, w, n_tiles)
    trace_want = _loop_trace_want(src_l, dst_l, loop, n_tiles)
    src_d, dst_d = src_h.cuda(), dst_h.cuda()
    trace_d = torch.full((max(trace_want.size, 1),), -1, dtype=torch.int64, device="cuda")
    lc().layout_copy_loop_ptr(src_d.data_ptr() + src_shift, src_l, dst_d.data_ptr() + dst_shift, dst_l, w,
                              loop, n_tiles, trace_d.data_ptr(), torch.cuda.current_stream().cuda_stream)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    got = dst_d.cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError("%d bytes differ, first at %d (got %d want %d)"
                             % (bad.size, bad[0], got[bad[0]], want[bad[0]]))
    got_trace = trace_d.cpu().numpy()[:trace_want.size]
    assert np.array_equal(got_trace, trace_want), "the partition differs from the override"


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_loop_layout_copies(w):
    dl = oracle.index_maps.default_loop_layout
    # the scale-factor transpose batch under the default plan (64 threads x 4)
    run_loop_case(L((2, 1, 4, 32), (128, 128, 32, 1)), L((2, 1, 4, 32), (128, 128, 1, 4)), w,
                  dl(256, 64, 4), n_tiles=37, seed=w)
    # one column per thread (no vectors)
    run_loop_case(L((8, 8), (8, 1)), L((8, 8), (1, 8)), w, [(8, 0, 1), (8, 1, 0)], n_tiles=3)
    # thread-major blocks of an identity copy (vectors of consecutive slots)
    run_loop_case(L((64, 128), (128, 1)), L((64, 128), (128, 1)), w,
                  [(16, 1, 0), (4, 0, 128), (128, 0, 1)], n_tiles=2)
    # ... the same with both bases moved off the vector grid
    run_loop_case(L((64, 128), (128, 1)), L((64, 128), (128, 1)), w,
                  [(16, 1, 0), (4, 0, 128), (128, 0, 1)], src_shift=w, dst_shift=3 * w)
    # ragged: 5 threads x 6 slots, offsets, padded tile strides
    run_loop_case(L((6, 5), (5, 1), 2, 40), L((6, 5), (1, 6), 1, 31), w, [(6, 0, 1), (5, 1, 0)], n_tiles=3)
    # 1024 threads of one slot, and one thread of 64 slots
    run_loop_case(L((32, 32), (32, 1)), L((32, 32), (1, 32)), w, [(32, 1, 0), (32, 32, 0)], n_tiles=2)
    run_loop_case(L((8, 8), (8, 1)), L((8, 8), (1, 8)), w, [(8, 0, 8), (8, 0, 1)])
    # radices that do not nest (suffix products 1, 6, 12 against 1, 4, 12):
    # the general path, every vector's offsets decoded from its flat index
    run_loop_case(L((3, 4), (4, 1)), L((3, 4), (1, 3)), w, [(2, 1, 0), (6, 0, 1)], n_tiles=2)
    run_loop_case(L((9, 10), (10, 1), 1), L((9, 10), (1, 9)), w, [(3, 0, 6), (5, 1, 0), (6, 0, 1)], n_tiles=2)
    # gapped and broadcast source strides
    run_loop_case(L((16, 16), (40, 2)), L((16, 16), (1, 16)), w, [(16, 0, 1), (16, 1, 0)])
    run_loop_case(L((12, 10), (0, 1)), L((12, 10), (10, 1)), w, dl(120, 12, 2), n_tiles=2)


def test_loop_layout_small_workload_and_random_partitions():
    c = workloads.config(8, scale="small")
    assert c["loop"] == oracle.index_maps.default_loop_layout(8 * 16 * 32, 128, 8)
    run_loop_case(c["src"], c["dst"], c["elem_bytes"], c["loop"], c["n_tiles"], seed=8)
    rng = random.Random(88)
    ran = 0
    for i in range(30):
        src, dst, w, n_tiles = _random_layout_pair(rng)
        extents = [m[0] for m in oracle.paired_modes(src, dst)]
        N = int(np.prod(extents))
        if N == 0 or N > 1 << 14:
            continue
        # an exact partition: factor N into digits, each a thread or a slot digit
        digits, rest = [], N
        for p in (2, 3, 5, 7, 11, 13):
            while rest % p == 0:
                digits.append(p)
                rest //= p
        if rest > 1:
            digits.append(rest)
        digits = digits or [1]  # a one-point nest: one unit mode
        rng.shuffle(digits)
        while len(digits) > 6:  # merge digits: at most 8 modes
            last = digits.pop()
            digits[rng.randrange(len(digits))] *= last
        loop, ts, ss = [None] * len(digits), 1, 1
        for k in rng.sample(range(len(digits)), len(digits)):
            if rng.random() < 0.5 and ts * digits[k] <= 1024:
                loop[k], ts = (digits[k], ts, 0), ts * digits[k]
            else:
                loop[k], ss = (digits[k], 0, ss), ss * digits[k]
        run_loop_case(src, dst, w, loop, n_tiles, seed=i)
        ran += 1
    assert ran >= 15


def test_loop_layout_empty_and_refused():
    run_loop_case(L((0, 4), (4, 1)), L((0, 4), (1, 4)), 4, [(0, 1, 0), (4, 0, 1)])
    run_loop_case(L((4, 4), (4, 1)), L((4, 4), (1, 4)), 4, [(4, 1, 0), (4, 0, 1)], n_tiles=0)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    for loop, status in [([(4, 2, 0), (4, 0, 1)], "LC_ERR_LOOP_LAYOUT"),
                         ([(2048, 1, 0)], "LC_ERR_SHAPE"),
                         ([(4, 0, 1), (4, 1, 1)], "LC_ERR_BAD_STRIDE")]:
        with pytest.raises(lc().LayoutCopyError) as e:
            lc().layout_copy_loop_ptr(p, L((4, 4), (4, 1)), p + 4096, L((4, 4), (1, 4)), 4, loop)
        assert e.value.status == lc().STATUS[status]
    with pytest.raises(lc().LayoutCopyError) as e:
        lc().layout_copy_loop_ptr(p, L((4, 4), (4, 1)), p + 32, L((4, 4), (1, 4)), 4, [(4, 1, 0), (4, 0, 1)])
    assert e.value.status == lc().STATUS["LC_ERR_OVERLAP"]
    assert (buf == 0).all()


def test_loop_layout_full_workload():
    c = workloads.config(8)
    assert c["loop"] == oracle.index_maps.default_loop_layout(32 * 128 * 128, 1024, 8)
    src_h = workloads.make_src(c)
    src_d = src_h.cuda()
    dst_d = workloads.make_dst(c, device="cuda")
    N = 32 * 128 * 128
    trace = torch.full((c["n_tiles"] * N,), -1, dtype=torch.int64, device="cuda")
    lc().layout_copy_loop(src_d, c["src"], dst_d, c["dst"], c["loop"], n_tiles=c["n_tiles"],
                          elem_bytes=2, trace=trace)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    _assert_same_bytes(dst_d.cpu().numpy(), _oracle_full(c, src_h.numpy()), c["name"])
    rng = np.random.default_rng(8)
    pts = rng.integers(0, c["n_tiles"] * N, size=1 << 18, dtype=np.int64)
    pts[:2] = [0, c["n_tiles"] * N - 1]
    so, do = oracle.offsets_of(c["src"], c["dst"], c["n_tiles"], pts)
    sv, dv = src_d.view(torch.int16), dst_d.view(torch.int16)
    assert torch.equal(sv[torch.from_numpy(so).cuda()], dv[torch.from_numpy(do).cuda()])
    T, L_ = 1024, N // 1024
    want = np.empty(pts.size, np.int64)
    for i, f in enumerate(pts[:4096]):
        t, slot = oracle.index_maps.loop_layout_owner(int(f % N), c["loop"])
        want[i] = t * L_ + slot
    got = trace[torch.from_numpy(pts[:4096]).cuda()].cpu().numpy()
    assert np.array_equal(got, want[:4096])
    # every point moved exactly once per tile: the trace is a permutation of 0..N-1
    assert torch.equal(torch.sort(trace[:N]).values, torch.arange(N, device="cuda"))
    assert torch.equal(torch.sort(trace[-N:]).values, torch.arange(N, device="cuda"))


# ---------------------------------------------------------------------------
# maximum sizes: indices past 32 bits (the 64-bit index paths) and the split
# path's 2^31-byte cut-off; inputs drawn on the device from a seeded
# generator, offsets of sampled points from the oracle, and whole-buffer
# equality of the slices the definition pairs
# ---------------------------------------------------------------------------

def _device_bytes(n, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8, device="cuda")


def _sampled_points_agree(src_d, dst_d, src_l, dst_l, n_tiles, n_points, seed, edges=()):
    rng = np.random.default_rng(seed)
    pts = np.concatenate([np.asarray(edges, np.int64), rng.integers(0, n_points, 1 << 16, dtype=np.int64)])
    so, do = oracle.offsets_of(src_l, dst_l, n_tiles, pts)
    assert torch.equal(src_d[torch.from_numpy(so).cuda()], dst_d[torch.from_numpy(do).cuda()])


def test_vector_copy_past_32_bit_indices():
    n = (1 << 32) + 5  # one-byte words gathered at stride 2: 2^32 + 5 vectors
    src_d = _device_bytes(2 * n, 321)
    dst_d = torch.full((n,), workloads.SENTINEL, dtype=torch.uint8, device="cuda")
    src_l, dst_l = L((n,), (2,)), L((n,), (1,))
    assert lc().plan(src_l, dst_l, 1)["kernel_name"] == "vec_copy"
    lc().layout_copy(src_d, src_l, dst_d, dst_l, elem_bytes=1)
    assert lc().last_device_error()[0] == 0
    _sampled_points_agree(src_d, dst_d, src_l, dst_l, 1, n, 3, edges=[0, (1 << 32) - 1, 1 << 32, n - 1])
    assert torch.equal(dst_d, src_d[::2])
    del src_d, dst_d
    torch.cuda.empty_cache()


def test_warp_shuffle_offsets_past_32_bits():
    # (4, 32) fp32 blocks of tiles spaced 1 GiB apart on the source: the
    # source span passes 4 GiB, so the kernel forms 64-bit offsets; the
    # compact destination is checked whole, point by point
    n_tiles = 5
    src_l = L((4, 32), (32, 1), 0, 1 << 28)
    dst_l = L((4, 32), (1, 4))
    assert lc().plan(src_l, dst_l, 4, n_tiles, "warp_shuffle")["kernel_name"] == "warp_shuffle"
    src_d = _device_bytes(_footprint(src_l, n_tiles) * 4, 911)
    dst_d = torch.full((_footprint(dst_l, n_tiles) * 4,), workloads.SENTINEL, dtype=torch.uint8, device="cuda")
    lc().layout_copy(src_d, src_l, dst_d, dst_l, n_tiles=n_tiles, elem_bytes=4, kernel="warp_shuffle")
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    n = n_tiles * 128
    so, do = oracle.offsets_of(src_l, dst_l, n_tiles, np.arange(n, dtype=np.int64))
    sv, dv = src_d.view(-1, 4), dst_d.view(-1, 4)
    assert torch.equal(sv[torch.from_numpy(so).cuda()], dv[torch.from_numpy(do).cuda()])
    assert sorted(do.tolist()) == list(range(dst_d.numel() // 4))  # every destination word written


def test_loop_copy_past_32_bit_indices():
    m = (1 << 31) + (1 << 13)  # two rows of m one-byte words: 2^32 + 2^14 points in one tile
    n = 2 * m
    gap = 64
    src_d = _device_bytes(n + gap, 322)
    dst_d = torch.full((n,), workloads.SENTINEL, dtype=torch.uint8, device="cuda")
    src_l, dst_l = L((2, m), (m + gap, 1)), L((2, m), (m, 1))
    loop = [((n >> 14), 0, 16), (1024, 1, 0), (16, 0, 1)]
    assert lc().loop_layout_info(loop, n) == (1024, n // 1024)
    lc().layout_copy_loop(src_d, src_l, dst_d, dst_l, loop, elem_bytes=1)
    assert lc().last_device_error()[0] == 0
    _sampled_points_agree(src_d, dst_d, src_l, dst_l, 1, n, 4, edges=[0, m - 1, m, (1 << 32) - 1, 1 << 32, n - 1])
    assert torch.equal(dst_d[:m], src_d[:m]) and torch.equal(dst_d[m:], src_d[m + gap:])
    del src_d, dst_d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [(1 << 31) - (1 << 14), (1 << 31) + (1 << 20)])
def test_loop_copy_around_the_split_cut_off(n):
    """Tiles just under and just over 2^31 bytes: the first takes the split
    path (31-bit byte offsets), the second the general path."""
    src_d = _device_bytes(2 * n, 323)
    dst_d = torch.full((2 * n,), workloads.SENTINEL, dtype=torch.uint8, device="cuda")
    src_l, dst_l = L((n,), (1,)), L((n,), (1,))
    loop = [(n >> 14, 0, 16), (1024, 1, 0), (16, 0, 1)]
    lc().layout_copy_loop(src_d, src_l, dst_d, dst_l, loop, n_tiles=2, elem_bytes=1)
    assert lc().last_device_error()[0] == 0
    assert torch.equal(dst_d, src_d)
    del src_d, dst_d
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# "copy -> gmem_smem" staged through shared memory: the device primitive
# (lc_device::gmem_smem_copy) driven by the staged-tile kernel, against the
# oracle's words and the oracle's replay of both partitions (guard included)
# ---------------------------------------------------------------------------

def _row_major(shape):
    st, acc = [], 1
    for e in reversed(shape):
        st.insert(0, acc)
        acc *= max(1, e)
    return tuple(st)


def _staged_case(src_l, dst_l, w, n_tiles, threads, swizzle, seed, check_trace=True, src_shift=0):
    ns = _footprint(src_l, n_tiles) * w + src_shift
    nd = _footprint(dst_l, n_tiles) * w
    g = torch.Generator().manual_seed(seed)
    src_h = torch.randint(0, 256, (max(ns, 1),), generator=g, dtype=torch.uint8)
    dst_h = torch.full((max(nd, 1),), workloads.SENTINEL, dtype=torch.uint8)
    want = dst_h.numpy().copy()
    oracle.copy(src_h.numpy()[src_shift:].copy(), src_l, want, dst_l, w, n_tiles)
    N = int(np.prod(src_l["shape"]))
    tin = torch.full((n_tiles * N,), -1, dtype=torch.int64, device="cuda")
    tout = torch.full((n_tiles * N,), -1, dtype=torch.int64, device="cuda")
    src_d, dst_d = src_h.cuda(), dst_h.cuda()
    view = src_d[src_shift:] if src_shift else src_d
    lc().layout_copy_staged(view, src_l, dst_d, dst_l, n_tiles=n_tiles, elem_bytes=w, threads=threads,
                            swizzle=swizzle, trace_in=tin, trace_out=tout)
    st, detail = lc().last_device_error()
    assert st == 0, "device error word %#x" % detail
    got = dst_d.cpu().numpy()
    assert np.array_equal(got, want), (src_l, dst_l, w, n_tiles, threads, swizzle)
    if not check_trace:
        return
    sh = _row_major(src_l["shape"])
    chunk = None if swizzle is None or swizzle[0] == 0 else 1 << swizzle[1]
    for tr, lay in ((tin, src_l), (tout, dst_l)):
        part = oracle.index_maps.gmem_smem_partition_guarded(lay["shape"], lay["stride"], sh, w, threads,
                                                             lay["offset"], 0, chunk)
        one = np.full(N, -1, np.int64)
        for f, tid, _g, _s, elems in oracle.index_maps.gmem_smem_replay(part, threads, lay["offset"], 0):
            for _gg, s in elems:
                one[s] = f * threads + tid
        assert np.array_equal(tr.cpu().numpy(), np.tile(one, n_tiles)), (lay, part["vec"], part["outer"])


def test_staged_copy_guarded_partitions():
    # the guard: 64 words, 128 threads -> 16 (4-byte) or 32 (8-byte) busy threads
    _staged_case(L((64,), (1,)), L((64,), (1,)), 4, 3, 128, None, 1)
    _staged_case(L((64,), (1,)), L((64,), (1,)), 8, 3, 128, None, 2)
    _staged_case(L((100,), (1,)), L((100,), (1,)), 4, 2, 32, None, 3)
    # a transposed copy with a thread count that divides nothing
    sh = (4, 8, 16)
    _staged_case(L(sh, _row_major(sh)), L(sh, permuted(sh, (0, 2, 1))), 2, 5, 96, (3, 4, 7), 4)


def test_staged_copy_page_tile_and_swizzles():
    # the page's 32 x 32 fp32 tile, transposed: a 4-byte-chunk swizzle makes the
    # column reads of copy 2 conflict-free and caps copy 1 at one word per access
    src_l, dst_l = L((32, 32), (32, 1)), L((32, 32), (1, 32))
    for swz in [(0, 0, 0), (5, 2, 7), (3, 4, 7)]:
        _staged_case(src_l, dst_l, 4, 1, 256, swz, 5)
    _staged_case(src_l, dst_l, 4, 3, 1024, (5, 2, 7), 6)
    sf = (2, 1, 4, 32)
    _staged_case(L(sf, (128, 128, 32, 1)), L(sf, (128, 128, 1, 4)), 4, 7, 64, (2, 4, 6), 7)


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_staged_copy_widths_and_library_swizzle(w):
    for i, (shape, perm) in enumerate([((16, 24), (1, 0)), ((3, 5, 33), (2, 0, 1)), ((8, 4, 2, 16), (0, 2, 1, 3))]):
        src_l = L(shape, _row_major(shape))
        dst_l = L(shape, permuted(shape, perm))
        _staged_case(src_l, dst_l, w, 4, 128, None, 10 * w + i, check_trace=False)
        run_case(src_l, dst_l, w, 4, kernel="smem_staged", seed=20 * w + i)
    # a source base off the vector grid: the copy narrows to single words
    _staged_case(L((16, 24), (24, 1)), L((16, 24), (1, 16)), w, 2, 64, None, 99, check_trace=False, src_shift=w)


def test_staged_copy_refusals():
    src = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(lc().LayoutCopyError) as e:
        lc().layout_copy_staged(src, L((64,), (1,)), dst, L((64,), (1,)), elem_bytes=4, threads=48)
    assert e.value.status == lc().STATUS["LC_ERR_SHAPE"]
    with pytest.raises(lc().LayoutCopyError) as e:  # a tile over LC_STAGED_MAX_BYTES
        lc().layout_copy_staged(src, L((256, 128), (128, 1)), dst, L((256, 128), (1, 256)), elem_bytes=4)
    assert e.value.status == lc().STATUS["LC_ERR_SHAPE"]
    with pytest.raises(lc().LayoutCopyError) as e:  # source and destination overlap
        lc().layout_copy_staged(src, L((64,), (1,)), src[64:], L((64,), (1,)), elem_bytes=4)
    assert e.value.status == lc().STATUS["LC_ERR_OVERLAP"]
    with pytest.raises(lc().LayoutCopyError) as e:  # a swizzle whose span is past the tile budget
        lc().layout_copy_staged(src, L((64,), (1,)), dst, L((64,), (1,)), elem_bytes=4, swizzle=(8, 10, 18))
    assert e.value.status == lc().STATUS["LC_ERR_SHAPE"]
