"""The copy's plain definition: every logical index moves one word.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A TileLayout ``S[shape : stride]`` maps a logical index ``i`` to the element
offset ``offset + sum_k i_k * stride_k`` (Apache TVM docs, "permute_layout",
section "Algorithm", step 3: ``project(idx, strides)``; "copy -> gmem_smem",
section "Demonstration program": ``TileLayout(S[shape])`` is row-major).  Both
operands of a copy carry the same non-unit extents ("copy -> gmem_smem",
section "What it accepts", row "dtype / shape"; "permute_layout", section
"What it accepts", row "operands"), so the k-th non-unit mode of the source is
paired with the k-th non-unit mode of the destination and both are indexed by
the same logical index.

Tiles are this library's batching convention (the pages only show a
``for s in T.serial(0, pipe)`` loop around one warp op): tile ``t`` adds
``t * tile_stride`` to each side, and a ``tile_stride`` of 0 means the
layout's cosize, ``1 + sum_k (shape_k - 1) * stride_k``, i.e. tiles packed
back to back.

The word loop itself lives in ``copy_oracle.c`` (a plain C loop, built by
``oracle/build.py``); this module pairs the modes, computes tile strides and
hands plain arrays to it.  ``offsets_of`` gives the two element offsets of any
chosen logical points, for sampled checks at sizes where a full replay would be
slow.
"""
from __future__ import annotations

import ctypes
from collections import namedtuple

import numpy as np

from . import build as _build

Layout = namedtuple("Layout", "shape stride offset tile_stride", defaults=(0, 0))


def as_layout(obj) -> Layout:
    """Accept an oracle Layout, a mapping, or any object with the four fields."""
    if isinstance(obj, Layout):
        return obj
    if isinstance(obj, dict):
        return Layout(tuple(obj["shape"]), tuple(obj["stride"]),
                      int(obj.get("offset", 0)), int(obj.get("tile_stride", 0)))
    return Layout(tuple(obj.shape), tuple(obj.stride), int(obj.offset),
                  int(obj.tile_stride))


def cosize(layout: Layout) -> int:
    """One past the largest offset a single tile reaches (base offset excluded)."""
    layout = as_layout(layout)
    if any(e == 0 for e in layout.shape):
        return 0
    return 1 + sum((e - 1) * s for e, s in zip(layout.shape, layout.stride))


def paired_modes(src: Layout, dst: Layout):
    """Pair the non-unit modes of the two layouts: [(extent, src_stride, dst_stride)].

    Raises ValueError when the non-unit extents differ, which both pages
    reject ("extent mismatch").
    """
    src, dst = as_layout(src), as_layout(dst)
    s_modes = [(e, s) for e, s in zip(src.shape, src.stride) if e != 1]
    d_modes = [(e, s) for e, s in zip(dst.shape, dst.stride) if e != 1]
    if [e for e, _ in s_modes] != [e for e, _ in d_modes]:
        raise ValueError("extent mismatch: %r vs %r" % (src.shape, dst.shape))
    return [(e, ss, ds) for (e, ss), (_, ds) in zip(s_modes, d_modes)]


def tile_strides(src: Layout, dst: Layout):
    src, dst = as_layout(src), as_layout(dst)
    sts = src.tile_stride if src.tile_stride else cosize(src)
    dts = dst.tile_stride if dst.tile_stride else cosize(dst)
    return sts, dts


_I64P = ctypes.POINTER(ctypes.c_int64)


def _lib():
    lib = _build.load()
    fn = lib.oracle_copy
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                   _I64P, _I64P, _I64P, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    return fn


def copy(src_bytes: np.ndarray, src_layout, dst_bytes: np.ndarray, dst_layout,
         elem_bytes: int, n_tiles: int = 1, tile_range=None) -> None:
    """dst[dst_off(t, i)] = src[src_off(t, i)] for every tile t and logical index i.

    ``src_bytes`` / ``dst_bytes`` are flat uint8 arrays addressed in elements of
    ``elem_bytes`` bytes; ``dst_bytes`` is written in place and bytes outside
    the destination image are left as they were.  ``tile_range=(b, e)``
    restricts the walk to tiles b..e-1 (used to split the work across threads).
    """
    src_layout, dst_layout = as_layout(src_layout), as_layout(dst_layout)
    modes = paired_modes(src_layout, dst_layout)
    sts, dts = tile_strides(src_layout, dst_layout)
    assert src_bytes.dtype == np.uint8 and dst_bytes.dtype == np.uint8
    assert src_bytes.flags.c_contiguous and dst_bytes.flags.c_contiguous
    if n_tiles <= 0 or any(e == 0 for e, _, _ in modes):
        return
    _check_bounds(src_bytes.size, src_layout.offset, sts, modes, 1, elem_bytes, n_tiles)
    _check_bounds(dst_bytes.size, dst_layout.offset, dts, modes, 2, elem_bytes, n_tiles)
    ext = np.array([m[0] for m in modes] or [1], dtype=np.int64)
    ss = np.array([m[1] for m in modes] or [0], dtype=np.int64)
    ds = np.array([m[2] for m in modes] or [0], dtype=np.int64)
    b, e = tile_range if tile_range is not None else (0, n_tiles)
    rc = _lib()(src_bytes.ctypes.data, dst_bytes.ctypes.data, int(elem_bytes),
                len(modes), ext.ctypes.data_as(_I64P), ss.ctypes.data_as(_I64P),
                ds.ctypes.data_as(_I64P), src_layout.offset, dst_layout.offset,
                sts, dts, int(b), int(e))
    if rc != 0:
        raise RuntimeError("oracle_copy failed (%d)" % rc)


def _check_bounds(nbytes, base, ts, modes, side, w, n_tiles):
    """Refuse to let the C loop touch bytes outside the given buffer."""
    hi = base + (n_tiles - 1) * ts
    for m in modes:
        hi += (m[0] - 1) * m[side]
    if base < 0 or (hi + 1) * w > nbytes:
        raise ValueError("layout reaches byte %d of a %d-byte buffer" % ((hi + 1) * w, nbytes))


def offsets_of(src_layout, dst_layout, n_tiles: int, points: np.ndarray):
    """Element offsets (src, dst) of chosen points of the tiles x logical box.

    ``points`` are flat indices into the row-major walk of (tile, i_0, ...,
    i_{r-1}), the same order ``copy`` walks.  Returns two int64 arrays.
    """
    src_layout, dst_layout = as_layout(src_layout), as_layout(dst_layout)
    modes = paired_modes(src_layout, dst_layout)
    sts, dts = tile_strides(src_layout, dst_layout)
    extents = [n_tiles] + [m[0] for m in modes]
    s_str = [sts] + [m[1] for m in modes]
    d_str = [dts] + [m[2] for m in modes]
    rest = np.asarray(points, dtype=np.int64).copy()
    so = np.full(rest.shape, src_layout.offset, dtype=np.int64)
    do = np.full(rest.shape, dst_layout.offset, dtype=np.int64)
    for e, s, d in reversed(list(zip(extents, s_str, d_str))):
        i = rest % e
        rest //= e
        so += i * s
        do += i * d
    return so, do


def logical_size(src_layout, dst_layout, n_tiles: int = 1) -> int:
    n = n_tiles
    for e, _, _ in paired_modes(src_layout, dst_layout):
        n *= e
    return n
