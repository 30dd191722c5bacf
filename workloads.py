"""Seeded synthetic workloads for the layout copy: shapes, layouts and bytes.

This module only DESCRIBES inputs and draws their bytes; it holds none of the
copy's arithmetic, so both the oracle side and the GPU side can take their
inputs from it.  Every buffer is generated on the host from a CPU
``torch.Generator`` with a fixed seed, so the oracle and the GPU see the same
bytes.

The five workloads are those the library is measured on:
  1  one 32x32 fp32 tile, row-major (32,1) -> transposed (1,32), one warp
  2  2^20 tiles of (pipe=2, high=1, 4, 32) fp32, strides (128,128,32,1) ->
     (128,128,1,4), tiles packed back to back (the scale-factor transpose of
     the Apache TVM "permute_layout" page, batched)
  3  16384x16384 bf16, row-major -> column-major
  4  8192x8192 transpose for element widths 1, 2, 4, 8 and 16 bytes
  5  (256,32,128,128) bf16 axis permute (0,2,1,3)
  6  8191 x 8193 transpose with row strides off the 16-byte grid (the layouts
     the TMA path cannot take), 4-byte words by default
  7  window sum b[i] = a[i] + a[i+1] + a[i+2] over 2^28 float32 outputs (the
     "Window Sum Example" of MLC Ep7, scaled up)
  8  workload 5's permute as 256 tiles of (32,128,128), one per batch entry,
     moved under an explicit loop layout (the "loop_layout=" override of the
     TileLang "loop_mapping.py" page): (64: slot stride 8), (1024: thread
     stride 1), (8: slot stride 1), which restates the default partition with
     1024 threads and vectors of 8 words
Layouts are plain dicts: shape, stride, offset, tile_stride (elements).
"""
from __future__ import annotations

import torch

HBM_L2_BYTES = 129 * 1024 * 1024  # GB300 L2; inputs larger than this defeat it


def _layout(shape, stride, offset=0, tile_stride=0):
    return dict(shape=tuple(shape), stride=tuple(stride), offset=int(offset),
                tile_stride=int(tile_stride))


def config(cfg: int, elem_bytes: int | None = None, scale: str = "full") -> dict:
    """One workload: dict(name, src, dst, elem_bytes, n_tiles, kind, seed).

    ``scale="small"`` gives a reduced case of the same structure (several
    tiles plus a ragged tail) that the CPU oracle finishes in well under a
    second; ``"full"`` gives the measured size.
    """
    small = scale == "small"
    if cfg == 1:
        return dict(name="tile32x32_f32_transpose", cfg=1,
                    src=_layout((32, 32), (32, 1)), dst=_layout((32, 32), (1, 32)),
                    elem_bytes=4, n_tiles=1, kind="uniform_f32", seed=1)
    if cfg == 2:
        shape = (2, 1, 4, 32)
        return dict(name="sf_transpose_batch_f32", cfg=2,
                    src=_layout(shape, (128, 128, 32, 1)),
                    dst=_layout(shape, (128, 128, 1, 4)),
                    elem_bytes=4, n_tiles=(1 << 12) + 3 if small else 1 << 20,
                    kind="uniform_f32", seed=2)
    if cfg == 3:
        r, c = (1000, 1104) if small else (16384, 16384)
        return dict(name="transpose2d_bf16", cfg=3,
                    src=_layout((r, c), (c, 1)), dst=_layout((r, c), (1, r)),
                    elem_bytes=2, n_tiles=1, kind="normal_bf16", seed=3)
    if cfg == 4:
        w = 4 if elem_bytes is None else int(elem_bytes)
        r, c = (528, 704) if small else (8192, 8192)
        return dict(name="transpose2d_w%d" % w, cfg=4,
                    src=_layout((r, c), (c, 1)), dst=_layout((r, c), (1, r)),
                    elem_bytes=w, n_tiles=1, kind="bytes", seed=40 + w)
    if cfg == 5:
        b, h, s, d = (3, 32, 128, 128) if small else (256, 32, 128, 128)
        return dict(name="permute0213_bf16", cfg=5,
                    src=_layout((b, h, s, d), (h * s * d, s * d, d, 1)),
                    dst=_layout((b, h, s, d), (h * s * d, d, h * d, 1)),
                    elem_bytes=2, n_tiles=1, kind="normal_bf16", seed=5)
    if cfg == 6:
        w = 4 if elem_bytes is None else int(elem_bytes)
        r, c = (301, 517) if small else (8191, 8193)
        return dict(name="transpose2d_unaligned_w%d" % w, cfg=6,
                    src=_layout((r, c), (c, 1)), dst=_layout((r, c), (1, r)),
                    elem_bytes=w, n_tiles=1, kind="bytes", seed=60 + w)
    if cfg == 7:
        n = (1 << 16) + 3 if small else 1 << 28
        return dict(name="window_sum3_f32", cfg=7, n_out=n, window=3, elem_bytes=4,
                    kind="uniform_f32", seed=7)
    if cfg == 8:
        b, (h, s, d) = (5, (8, 16, 32)) if small else (256, (32, 128, 128))
        loop = [(4, 0, 8), (128, 1, 0), (8, 0, 1)] if small else [(64, 0, 8), (1024, 1, 0), (8, 0, 1)]
        return dict(name="permute0213_loop_bf16", cfg=8,
                    src=_layout((h, s, d), (s * d, d, 1), 0, h * s * d),
                    dst=_layout((h, s, d), (d, h * d, 1), 0, h * s * d),
                    elem_bytes=2, n_tiles=b, kind="normal_bf16", seed=8, loop=loop)
    raise ValueError("unknown workload %r" % cfg)


def footprint_elems(layout: dict, n_tiles: int) -> int:
    """Elements a buffer must hold for ``n_tiles`` tiles of ``layout``.

    Only sizes the buffer: the largest reachable offset plus one.
    """
    shape, stride = layout["shape"], layout["stride"]
    if n_tiles <= 0 or any(e == 0 for e in shape):
        return layout["offset"]
    span = 1 + sum((e - 1) * s for e, s in zip(shape, stride))
    ts = layout["tile_stride"] or span
    return layout["offset"] + (n_tiles - 1) * ts + span


def logical_elems(cfg: dict) -> int:
    n = cfg["n_tiles"]
    for e in cfg["src"]["shape"]:
        n *= e
    return n


def make_bytes(n_elems: int, elem_bytes: int, kind: str, seed: int) -> torch.Tensor:
    """Seeded host bytes (uint8, contiguous) for ``n_elems`` words."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    if kind == "uniform_f32" and elem_bytes == 4:
        vals = torch.rand(n_elems, generator=g, dtype=torch.float32) * 2.0 - 1.0
        return vals.view(torch.uint8)
    if kind == "normal_bf16" and elem_bytes == 2:
        vals = torch.randn(n_elems, generator=g, dtype=torch.float32).to(torch.bfloat16)
        return vals.view(torch.uint8)
    return torch.randint(0, 256, (n_elems * elem_bytes,), generator=g, dtype=torch.uint8)


def make_src(cfg: dict) -> torch.Tensor:
    n = footprint_elems(cfg["src"], cfg["n_tiles"])
    return make_bytes(n, cfg["elem_bytes"], cfg["kind"], cfg["seed"])


SENTINEL = 0xA5


def make_dst(cfg: dict, device="cpu") -> torch.Tensor:
    """Destination bytes prefilled with the sentinel 0xA5."""
    n = footprint_elems(cfg["dst"], cfg["n_tiles"]) * cfg["elem_bytes"]
    return torch.full((n,), SENTINEL, dtype=torch.uint8, device=device)
