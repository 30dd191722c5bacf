"""The pages' index maps, restated step by step on the CPU.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* ``flatten`` / ``unflatten`` / ``plan``: the TileLang tutorial "loop_mapping.py"
  (Chapter 08, section 6, module docstring): the nest is flattened row-major,
  ``access_idx = flat // vector_size``, ``thread = access_idx % num_thread``,
  ``local_idx = (access_idx // num_thread) * vector_size + flat % vector_size``.
* ``gmem_smem_partition`` / ``gmem_smem_replay``: Apache TVM docs
  "copy -> gmem_smem", section "Algorithm" steps 1-3 and section "How inputs
  change the algorithm" (the ``[outer, threads, vec]`` split, the widest-first
  vector width, the serial loop of vector copies).
* ``loop_layout_owner`` / ``loop_layout_plan`` / ``loop_layout_sizes`` /
  ``default_loop_layout`` / ``loop_layout_replay``: the same tutorial's
  ``loop_layout=`` override of the default plan (module docstring), under the
  reading stated at them.
* ``permute_align`` / ``permute_replay``: Apache TVM docs "permute_layout",
  section "Algorithm" steps 1 and 3 (the aligned ``extent``/``src_str``/
  ``dst_str``, ``P = prod(extent) / 32``, and the two register-staged phases
  with ``j = r ^ ((lane >> shift) & mask)``).

Pure-Python loops: these are meant for the small cases the pages show.
"""
from __future__ import annotations

from .definition import as_layout, paired_modes, tile_strides

WARP = 32


# ---------------------------------------------------------------------------
# TileLang loop partition ("loop_mapping.py")
# ---------------------------------------------------------------------------

def flatten(index, extents) -> int:
    """Row-major position of ``index`` in a nest with ``extents`` (last fastest)."""
    flat = 0
    for k in range(len(extents)):
        flat = flat * extents[k] + index[k]
    return flat


def unflatten(flat: int, extents) -> tuple:
    """Inverse of ``flatten``: peel the last (fastest) coordinate first."""
    coords = []
    for e in reversed(extents):
        flat, c = divmod(flat, e)
        coords.append(c)
    return tuple(reversed(coords))


def plan(extents, num_thread: int, vector_size: int) -> dict:
    """{iteration point: (thread, per-thread slot)} of the default loop partition.

    Levels, fastest first: the ``vector_size`` innermost iterations share one
    thread's consecutive slots, consecutive groups rotate over the threads,
    and the remainder becomes a per-thread serial loop.
    """
    total = 1
    for e in extents:
        total *= e
    out = {}
    for flat in range(total):
        group, lane_in_vec = divmod(flat, vector_size)
        rnd, thread = divmod(group, num_thread)
        out[unflatten(flat, extents)] = (thread, rnd * vector_size + lane_in_vec)
    return out


# ---------------------------------------------------------------------------
# loop_layout= override of the default partition ("loop_mapping.py")
# ---------------------------------------------------------------------------
#
# The page says only that a ``loop_layout=`` annotation on ``T.Parallel``
# replaces the default plan above.  Reading: an override is again a map from
# each iteration point to (thread, slot), given as modes
# (extent, thread_stride, slot_stride), outermost first.  The point's
# row-major flat index is read as mixed-radix digits over the modes' extents
# (the last mode fastest); thread = sum(digit * thread_stride) and
# slot = sum(digit * slot_stride).  An override must be an exact partition:
# each non-unit mode feeds only the thread or only the slot, every point gets
# its own (thread, slot), and the pairs fill [0, T) x [0, L).


def _product(values) -> int:
    n = 1
    for v in values:
        n *= v
    return n


def loop_layout_owner(flat: int, loop) -> tuple:
    """(thread, slot) of the point with row-major flat index ``flat``."""
    digits = unflatten(flat, [m[0] for m in loop])
    thread = sum(c * m[1] for c, m in zip(digits, loop))
    slot = sum(c * m[2] for c, m in zip(digits, loop))
    return thread, slot


def loop_layout_plan(extents, loop) -> dict:
    """{iteration point: (thread, slot)} under the override ``loop``."""
    total = _product(extents)
    if _product(m[0] for m in loop) != total:
        raise Decline("the loop layout covers %d points, the nest %d"
                      % (_product(m[0] for m in loop), total))
    return {unflatten(flat, extents): loop_layout_owner(flat, loop) for flat in range(total)}


def loop_layout_sizes(extents, loop):
    """(threads T, slots per thread L) of an exact partition; Decline otherwise."""
    for e, ts, ss in loop:
        if e < 0 or ts < 0 or ss < 0:
            raise Decline("negative extent or stride in %r" % (loop,))
        if e > 1 and (ts > 0) == (ss > 0):
            raise Decline("mode %r must feed exactly one of thread and slot" % ((e, ts, ss),))
    pm = loop_layout_plan(extents, loop)
    if not pm:
        return 0, 0
    T = 1 + max(t for t, _ in pm.values())
    L = 1 + max(s for _, s in pm.values())
    if len(set(pm.values())) != len(pm) or T * L != len(pm):
        raise Decline("%r is not an exact partition of %d points" % (loop, len(pm)))
    return T, L


def default_loop_layout(total: int, num_thread: int, vector_size: int):
    """The default plan restated as an override.

    Its three levels are digits of the flat index: the serial round
    (total / (T * V), slot stride V), the thread (T, thread stride 1) and the
    lane in the vector (V, slot stride 1).  Declines when T * V does not
    divide the total: that is the page's guarded case, which no exact
    partition expresses.
    """
    if total % (num_thread * vector_size):
        raise Decline("%d points are not whole rounds of %d threads x %d"
                      % (total, num_thread, vector_size))
    return [(total // (num_thread * vector_size), 0, vector_size),
            (num_thread, 1, 0), (vector_size, 0, 1)]


def loop_layout_replay(src_words, dst_words, src_layout, dst_layout, loop,
                       n_tiles: int = 1):
    """Tile by tile, thread t moves its slots 0..L-1 in order: slot s of
    thread t is the point the override maps to (t, s), and that point moves
    one word from its source to its destination offset.

    Python lists of words, for small cases.  Returns the trace
    {(tile, flat index of the point): t * L + s}.
    """
    src_layout, dst_layout = as_layout(src_layout), as_layout(dst_layout)
    modes = paired_modes(src_layout, dst_layout)
    extents = [m[0] for m in modes]
    T, L = loop_layout_sizes(extents, loop)
    owner = {ts: idx for idx, ts in loop_layout_plan(extents, loop).items()}
    sts, dts = tile_strides(src_layout, dst_layout)
    trace = {}
    for tile in range(n_tiles):
        for t in range(T):
            for s in range(L):
                idx = owner[(t, s)]
                so = src_layout.offset + tile * sts + project(idx, [m[1] for m in modes])
                do = dst_layout.offset + tile * dts + project(idx, [m[2] for m in modes])
                dst_words[do] = src_words[so]
                trace[(tile, flatten(idx, extents))] = t * L + s
    return trace


# ---------------------------------------------------------------------------
# copy -> gmem_smem: [outer, threads, vec]
# ---------------------------------------------------------------------------

class Decline(Exception):
    """The variant does not accept this input (the page's "declines")."""


def _coalesce(modes):
    """Merge neighbours (outer, inner) that are row-major contiguous on both sides."""
    out = []
    for m in modes:
        if out:
            e0, *s0 = out[-1]
            e1, *s1 = m
            if all(a == b * e1 for a, b in zip(s0, s1)):
                out[-1] = (e0 * e1, *s1)
                continue
        out.append(tuple(m))
    return out


def gmem_smem_partition(shape, g_stride, s_stride, elem_bytes: int,
                        num_threads: int, g_offset: int = 0, s_offset: int = 0):
    """The synthesized partition of one global<->shared copy.

    Step 1: the region's modes (unit modes dropped) are put in the GLOBAL
    side's canonical order, stride descending, and neighbours contiguous on
    both sides are merged; the innermost mode is the contiguous tail.
    Step 2: vector widths of 128, 64, 32, 16, 8 bits are tried widest first;
    ``vec`` elements are accepted when the tail is contiguous on both sides
    and its extent is a multiple of ``vec``, and every other stride on both
    sides and both base offsets are multiples of ``vec`` (so each per-thread,
    per-round vector pointer is aligned).  Reading of the page: the split must
    also be exact, ``threads * vec`` dividing the element count.
    The variant declines when the element count is not a multiple of the
    thread count ("What it accepts", row "divisibility").

    Returns dict(modes=[(extent, g_stride, s_stride)], vec, outer, total).
    """
    modes = [(e, g, s) for e, g, s in zip(shape, g_stride, s_stride) if e != 1]
    modes.sort(key=lambda m: -m[1])  # stable: ties keep their logical order
    modes = _coalesce(modes)
    total = 1
    for e, _, _ in modes:
        total *= e
    if total % num_threads:
        raise Decline("element count %d not divisible by %d threads" % (total, num_threads))
    bits_per_elem = 8 * elem_bytes
    for bits in (128, 64, 32, 16, 8):
        if bits < bits_per_elem or bits % bits_per_elem:
            continue
        vec = bits // bits_per_elem
        if vec > 1:
            if not modes:
                continue
            te, tg, ts = modes[-1]
            if tg != 1 or ts != 1 or te % vec:
                continue
            others = [x for e, g, s in modes[:-1] for x in (g, s)]
            if any(x % vec for x in others) or g_offset % vec or s_offset % vec:
                continue
        if total % (num_threads * vec):
            continue
        return dict(modes=modes, vec=vec, outer=total // (num_threads * vec),
                    total=total)
    raise Decline("no vector width")


def gmem_smem_partition_guarded(shape, g_stride, s_stride, elem_bytes: int,
                                num_threads: int, g_offset: int = 0, s_offset: int = 0,
                                chunk_bytes: int | None = None):
    """The same partition with a guard instead of the page's "declines".

    Steps 1 and 2 as in ``gmem_smem_partition`` (global side drives the
    canonical order; widest vector whose per-thread pointers stay aligned),
    with two changes from other passages:
      * the element count need not be a multiple of ``threads * vec``: the
        rounds are ``outer = ceil(total / (threads * vec))`` and a vector whose
        first element lies past the end is not moved (TileLang tutorial
        "loop_mapping.py", closing note of ``compare_shapes``: when the count
        is below the thread count some threads get no work and the generated
        code adds a guard);
      * with a swizzled shared layout (``chunk_bytes`` = its swizzle chunk), a
        vector spans no more than one chunk ("copy -> gmem_smem", section
        "How inputs change the algorithm", last paragraph).
    Returns dict(modes, vec, outer, total, guarded).
    """
    if chunk_bytes is not None and chunk_bytes < elem_bytes:
        raise Decline("a swizzle chunk of %d bytes would split a %d-byte element" % (chunk_bytes, elem_bytes))
    modes = [(e, g, s) for e, g, s in zip(shape, g_stride, s_stride) if e != 1]
    modes.sort(key=lambda m: -m[1])
    modes = _coalesce(modes)
    total = 1
    for e, _, _ in modes:
        total *= e
    bits_per_elem = 8 * elem_bytes
    for bits in (128, 64, 32, 16, 8):
        if bits < bits_per_elem or bits % bits_per_elem:
            continue
        if chunk_bytes is not None and bits // 8 > chunk_bytes:
            continue
        vec = bits // bits_per_elem
        if vec > 1:
            if not modes:
                continue
            te, tg, ts = modes[-1]
            if tg != 1 or ts != 1 or te % vec:
                continue
            others = [x for e, g, s in modes[:-1] for x in (g, s)]
            if any(x % vec for x in others) or g_offset % vec or s_offset % vec:
                continue
        per_round = num_threads * vec
        return dict(modes=modes, vec=vec, outer=-(-total // per_round), total=total,
                    guarded=total % per_round != 0)
    raise Decline("no vector width")


def xor_swizzle(byte_offset: int, bits: int, chunk_log2: int, row_log2: int) -> int:
    """Where a shared byte offset is stored under the XOR swizzle: the
    ``bits``-bit field above ``row_log2`` is XORed into the chunk index
    (bits ``chunk_log2 .. chunk_log2 + bits``).  Reading of "copy ->
    gmem_smem" (whose swizzle formula is not given): the per-row XOR of the
    "permute_layout" page applied to 2^chunk_log2-byte chunks of a shared
    row; bytes inside a chunk keep their order.  ``bits = 0`` is no swizzle."""
    return byte_offset ^ (((byte_offset >> row_log2) & ((1 << bits) - 1)) << chunk_log2)


def gmem_smem_replay(part, num_threads: int, g_offset: int = 0, s_offset: int = 0):
    """The emitted serial loop: round f, thread tid moves elements
    ``[(f * threads + tid) * vec, +vec)`` of the canonical order; with a
    guarded partition, a vector starting at or past the element count is not
    moved (no thread's vector straddles the end: the tail is a multiple of
    vec).

    Yields (f, tid, g_lin, s_lin, [(g_off, s_off) per vector element]); g_lin
    and s_lin are the offsets of the vector's first element, the quantities
    the page's generated IR names.
    """
    extents = [m[0] for m in part["modes"]]
    vec = part["vec"]
    for f in range(part["outer"]):
        for tid in range(num_threads):
            if (f * num_threads + tid) * vec >= part["total"]:
                continue  # the guard
            elems = []
            for v in range(vec):
                idx = unflatten((f * num_threads + tid) * vec + v, extents)
                g = g_offset + sum(i * m[1] for i, m in zip(idx, part["modes"]))
                s = s_offset + sum(i * m[2] for i, m in zip(idx, part["modes"]))
                elems.append((g, s))
            yield f, tid, elems[0][0], elems[0][1], elems


def gmem_smem_copy(src_words, dst_words, part, num_threads, g_is_src: bool,
                   g_offset: int = 0, s_offset: int = 0):
    """Run the replayed loop on two Python lists of words (global, shared)."""
    for _f, _tid, _g, _s, elems in gmem_smem_replay(part, num_threads, g_offset, s_offset):
        for g, s in elems:
            if g_is_src:
                dst_words[s] = src_words[g]
            else:
                dst_words[g] = src_words[s]


# ---------------------------------------------------------------------------
# permute_layout: warp register-staged XOR swizzle
# ---------------------------------------------------------------------------

def permute_align(src_layout, dst_layout):
    """Step 1: sliced and canonicalized shards, source regrouped to the
    destination's shape.

    Reading of the page: unit modes are dropped, the non-unit modes are paired
    in logical order, and neighbours are merged only where BOTH sides are
    row-major contiguous; a linear source therefore collapses as far as the
    destination allows and ends up with the destination's shape.  Returns
    (extent, src_str, dst_str, P) with P = prod(extent) / 32; raises Decline
    when the element count is not a whole number of warp lanes.
    """
    modes = _coalesce(paired_modes(as_layout(src_layout), as_layout(dst_layout)))
    extent = tuple(m[0] for m in modes)
    total = 1
    for e in extent:
        total *= e
    if total % WARP:
        raise Decline("%d elements are not a multiple of the warp size" % total)
    return extent, tuple(m[1] for m in modes), tuple(m[2] for m in modes), total // WARP


def swizzled_iteration(lane: int, r: int, k: int, shift: int) -> int:
    """j = r ^ ((lane >> shift) & mask) with mask = 2**k - 1."""
    return r ^ ((lane >> shift) & ((1 << k) - 1))


def project(idx, strides) -> int:
    return sum(i * s for i, s in zip(idx, strides))


def permute_replay(src_words, dst_words, extent, src_str, dst_str, P: int,
                   k: int, shift: int, src_base: int = 0, dst_base: int = 0):
    """Step 3: phase 1 stages each lane's P words in registers through the
    source layout, a warp barrier follows, phase 2 writes them through the
    destination layout.  Because every read finishes before any write, the
    result is right even when the two buffers are the same list.

    Returns the access record [(lane, r, j, src_off, dst_off)].
    """
    regs = [[None] * P for _ in range(WARP)]
    record = []
    for lane in range(WARP):
        for r in range(P):
            j = swizzled_iteration(lane, r, k, shift)
            idx = unflatten(lane + j * WARP, extent)
            so = src_base + project(idx, src_str)
            regs[lane][r] = src_words[so]
            record.append((lane, r, j, so, dst_base + project(idx, dst_str)))
    # ---- warp barrier: every read above completes before any write below ----
    for lane, r, _j, _so, do in record:
        dst_words[do] = regs[lane][r]
    return record
