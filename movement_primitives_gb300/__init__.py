"""GB300-native strided tile layout copy / permute.

A TileLayout ``S[shape : stride]`` maps a logical index to the element offset
``offset + sum_k i_k * stride_k``; ``layout_copy`` moves every logical index's
word from the source layout to the destination layout on the GPU (Apache TVM
docs "copy -> gmem_smem" and "permute_layout").  Everything runs in the C-ABI
library ``liblayoutcopy.so`` (``include/layout_copy.h``); this module only
marshals arguments.  PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import Sequence

from . import _lib
from ._lib import KERNELS, STATUS, STATUS_NAMES

__all__ = ["TileLayout", "LayoutCopyError", "layout_copy", "layout_copy_ptr", "layout_copy_host",
           "host_staging_bytes", "layout_copy_host_static", "window_sum", "plan",
           "choose_swizzle", "swizzle_conflicts", "gmem_smem_partition",
           "last_device_error", "debug_wait_timeout", "warp_unit_plan", "warp_unit_run",
           "loop_layout_default", "loop_layout_info", "loop_plan", "layout_copy_loop", "layout_copy_loop_ptr",
           "KERNELS", "STATUS"]


@dataclass(frozen=True)
class TileLayout:
    """shape : stride (elements), base offset of tile 0, elements between tiles
    (0 = the layout's cosize, tiles packed back to back)."""
    shape: Sequence[int]
    stride: Sequence[int] = field(default=None)
    offset: int = 0
    tile_stride: int = 0

    def __post_init__(self):
        shape = tuple(int(e) for e in self.shape)
        object.__setattr__(self, "shape", shape)
        if self.stride is None:  # S[shape] alone: the library's row-major strides
            n = len(shape)
            sh, st = (ctypes.c_int64 * max(n, 1))(*shape), (ctypes.c_int64 * max(n, 1))()
            _check(_lib.lib().lc_row_major_strides(n, sh, st), "row-major strides of %r" % (shape,))
            object.__setattr__(self, "stride", tuple(st[:n]))
        else:
            object.__setattr__(self, "stride", tuple(int(s) for s in self.stride))

    @classmethod
    def of(cls, obj) -> "TileLayout":
        if isinstance(obj, TileLayout):
            return obj
        if isinstance(obj, dict):
            return cls(obj["shape"], obj.get("stride"), obj.get("offset", 0), obj.get("tile_stride", 0))
        return cls(*obj)

    def to_c(self) -> _lib.CTileLayout:
        if len(self.shape) != len(self.stride):
            raise ValueError("shape and stride lengths differ")
        c = _lib.CTileLayout()
        c.rank = len(self.shape)
        for k, (e, s) in enumerate(zip(self.shape[:_lib.MAX_RANK], self.stride[:_lib.MAX_RANK])):
            c.shape[k] = e
            c.stride[k] = s
        c.offset = self.offset
        c.tile_stride = self.tile_stride
        return c

    def footprint(self, n_tiles: int) -> int:
        """Elements a buffer needs to hold n_tiles tiles (the library's count;
        bounds check only)."""
        c = self.to_c()
        n = int(_lib.lib().lc_layout_footprint(ctypes.byref(c), int(n_tiles)))
        if n < 0:
            raise ValueError("invalid layout or tile count: %r, %d tiles" % (self, n_tiles))
        return n


_LAYOUT_CACHE = {}  # layout value -> (TileLayout, its C struct); the library only reads the struct
_LAYOUT_CACHE_MAX = 1024


def _layout_pair(obj):
    """(TileLayout, CTileLayout) of a layout given as a TileLayout, a dict or a
    sequence, converted once per distinct value (the conversion costs more
    than the library's own cached planning of a small copy)."""
    if isinstance(obj, TileLayout):
        key = (obj.shape, obj.stride, obj.offset, obj.tile_stride)
    elif isinstance(obj, dict):
        st = obj.get("stride")
        key = (tuple(obj["shape"]), None if st is None else tuple(st), obj.get("offset", 0),
               obj.get("tile_stride", 0))
    else:
        key = None
    pair = _LAYOUT_CACHE.get(key) if key is not None else None
    if pair is None:
        lay = TileLayout.of(obj)
        pair = (lay, lay.to_c())
        if key is not None:
            if len(_LAYOUT_CACHE) >= _LAYOUT_CACHE_MAX:
                _LAYOUT_CACHE.clear()
            _LAYOUT_CACHE[key] = pair
    return pair


def _c_layout(obj) -> _lib.CTileLayout:
    return _layout_pair(obj)[1]


class LayoutCopyError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib.lib().lc_status_string(status).decode()
        super().__init__("%s (%s)%s" % (STATUS_NAMES.get(status, status), msg,
                                        ": " + what if what else ""))


def _check(status: int, what: str = "") -> None:
    if status != 0:
        raise LayoutCopyError(status, what)


def _kernel_id(kernel) -> int:
    return KERNELS[kernel] if isinstance(kernel, str) else int(kernel)


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def layout_copy_ptr(src_ptr: int, src_layout, dst_ptr: int, dst_layout, elem_bytes: int,
                    n_tiles: int = 1, kernel="auto", stream=0) -> None:
    """Raw-pointer form: device addresses, layouts in elements, stream handle."""
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    st = _lib.lib().lc_layout_copy_ex(ctypes.c_void_p(src_ptr), ctypes.byref(sl),
                                      ctypes.c_void_p(dst_ptr), ctypes.byref(dl),
                                      int(elem_bytes), int(n_tiles), _kernel_id(kernel),
                                      ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "layout_copy")


def layout_copy(src, src_layout, dst, dst_layout, n_tiles: int = 1, elem_bytes: int | None = None,
                kernel="auto", stream=None) -> None:
    """Copy between two CUDA tensors viewed through TileLayouts.

    Layout strides and offsets count elements of ``elem_bytes`` bytes (default:
    the tensors' element size) from each tensor's first byte.  Launches on
    ``stream`` (default: the current torch stream) and returns at once.
    """
    if not (src.is_cuda and dst.is_cuda):
        raise ValueError("layout_copy needs CUDA tensors (there is no CPU path)")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("pass contiguous tensors; express strides through the layouts")
    w = int(elem_bytes) if elem_bytes is not None else src.element_size()
    if elem_bytes is None and dst.element_size() != w:
        raise ValueError("source and destination element sizes differ; pass elem_bytes")
    sl, dl = _layout_pair(src_layout)[0], _layout_pair(dst_layout)[0]
    for name, t, l in (("source", src, sl), ("destination", dst, dl)):
        need = l.footprint(n_tiles) * w
        have = t.numel() * t.element_size()
        if need > have:
            raise ValueError("%s layout reaches %d bytes; the tensor holds %d" % (name, need, have))
    layout_copy_ptr(src.data_ptr(), sl, dst.data_ptr(), dl, w, n_tiles, kernel, _stream_handle(stream))


def host_staging_bytes(src_layout, dst_layout, elem_bytes: int, n_tiles: int = 1) -> int:
    """Device staging bytes layout_copy_host needs for full pipelining."""
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    return int(_lib.lib().lc_host_staging_bytes(ctypes.byref(sl), ctypes.byref(dl), int(elem_bytes),
                                                int(n_tiles)))


def layout_copy_host(src, src_layout, dst, dst_layout, n_tiles: int = 1, elem_bytes: int | None = None,
                     staging=None, stream=None) -> None:
    """Copy between two HOST tensors (ideally pinned) through the GPU.

    Transfers and permutes are pipelined over chunks of tiles by the library
    (lc_layout_copy_host).  ``staging`` is a CUDA uint8 tensor of at least
    host_staging_bytes(...) bytes; when omitted one is allocated by torch for
    this call.  Returns once queued on ``stream``; synchronise it to finish.
    """
    import torch
    if src.is_cuda or dst.is_cuda:
        raise ValueError("layout_copy_host takes host tensors")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("pass contiguous tensors; express strides through the layouts")
    w = int(elem_bytes) if elem_bytes is not None else src.element_size()
    sl, dl = _layout_pair(src_layout)[0], _layout_pair(dst_layout)[0]
    for name, t, l in (("source", src, sl), ("destination", dst, dl)):
        need = l.footprint(n_tiles) * w
        if need > t.numel() * t.element_size():
            raise ValueError("%s layout reaches %d bytes; the tensor holds %d"
                             % (name, need, t.numel() * t.element_size()))
    if staging is None:
        staging = torch.empty(max(256, host_staging_bytes(sl, dl, w, n_tiles)), dtype=torch.uint8,
                              device="cuda")
    cs, cd = sl.to_c(), dl.to_c()
    st = _lib.lib().lc_layout_copy_host(ctypes.c_void_p(src.data_ptr()), ctypes.byref(cs),
                                        ctypes.c_void_p(dst.data_ptr()), ctypes.byref(cd), w,
                                        int(n_tiles), ctypes.c_void_p(staging.data_ptr()),
                                        staging.numel() * staging.element_size(),
                                        ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "layout_copy_host")


def layout_copy_mapped(src, src_layout, dst, dst_layout, n_tiles: int = 1, elem_bytes: int | None = None,
                       stream=None) -> None:
    """Copy between two PINNED host tensors, the kernels reading and writing
    them directly over the CPU-GPU link (lc_layout_copy_mapped): no staging
    buffer.  Returns once queued on ``stream``; synchronise it to finish.
    """
    if src.is_cuda or dst.is_cuda:
        raise ValueError("layout_copy_mapped takes host tensors")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("pass contiguous tensors; express strides through the layouts")
    w = int(elem_bytes) if elem_bytes is not None else src.element_size()
    sl, dl = _layout_pair(src_layout)[0], _layout_pair(dst_layout)[0]
    for name, t, l in (("source", src, sl), ("destination", dst, dl)):
        if l.footprint(n_tiles) * w > t.numel() * t.element_size():
            raise ValueError("%s layout reaches past the tensor" % name)
    cs, cd = sl.to_c(), dl.to_c()
    st = _lib.lib().lc_layout_copy_mapped(ctypes.c_void_p(src.data_ptr()), ctypes.byref(cs),
                                          ctypes.c_void_p(dst.data_ptr()), ctypes.byref(cd), w, int(n_tiles),
                                          ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "layout_copy_mapped")


def layout_copy_host_static(src, src_layout, dst, dst_layout, n_tiles: int = 1,
                            elem_bytes: int | None = None, stream=None) -> None:
    """layout_copy_host for callers that cannot allocate device memory.

    Stages through a fixed 32 MiB array inside the library instead of a
    caller-provided buffer (see lc_layout_copy_host_static); allocates
    nothing.  Calls share that array: do not let two calls overlap on the GPU.
    """
    if src.is_cuda or dst.is_cuda:
        raise ValueError("layout_copy_host_static takes host tensors")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("pass contiguous tensors; express strides through the layouts")
    w = int(elem_bytes) if elem_bytes is not None else src.element_size()
    sl, dl = _layout_pair(src_layout)[0], _layout_pair(dst_layout)[0]
    for name, t, l in (("source", src, sl), ("destination", dst, dl)):
        if l.footprint(n_tiles) * w > t.numel() * t.element_size():
            raise ValueError("%s layout reaches past the tensor" % name)
    cs, cd = sl.to_c(), dl.to_c()
    st = _lib.lib().lc_layout_copy_host_static(ctypes.c_void_p(src.data_ptr()), ctypes.byref(cs),
                                               ctypes.c_void_p(dst.data_ptr()), ctypes.byref(cd), w,
                                               int(n_tiles), ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "layout_copy_host_static")


def window_sum(a, b, window: int = 3, stream=None) -> None:
    """b[i] = a[i] + ... + a[i + window - 1] (float32 CUDA tensors, left to right)."""
    import torch
    if a.dtype != torch.float32 or b.dtype != torch.float32 or not (a.is_cuda and b.is_cuda):
        raise ValueError("window_sum takes float32 CUDA tensors")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("pass contiguous tensors")
    n = b.numel()
    if a.numel() < n + window - 1:
        raise ValueError("a holds %d floats, needs %d" % (a.numel(), n + window - 1))
    _check(_lib.lib().lc_window_sum_f32(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), n,
                                        int(window), ctypes.c_void_p(_stream_handle(stream))), "window_sum")


def plan(src_layout, dst_layout, elem_bytes: int, n_tiles: int = 1, kernel="auto") -> dict:
    """What the planner would launch (host only; pointers assumed aligned)."""
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    info = _lib.CPlanInfo()
    _check(_lib.lib().lc_plan(ctypes.byref(sl), ctypes.byref(dl), int(elem_bytes), int(n_tiles),
                              _kernel_id(kernel), ctypes.byref(info)), "plan")
    n = info.n_modes
    out = {f: getattr(info, f) for f, _ in _lib.CPlanInfo._fields_
           if f not in ("extent", "src_stride", "dst_stride")}
    out["kernel_name"] = _lib.lib().lc_kernel_name(info.kernel).decode()
    out["modes"] = [(info.extent[i], info.src_stride[i], info.dst_stride[i]) for i in range(n)]
    return out


def warp_unit_plan(src_layout, dst_layout, elem_bytes: int):
    """Plan of P4's warp-scope permute between two shared-memory buffers
    (lc_warp_unit_plan).  Returns (plan, info): `plan` is the C struct to pass
    to warp_unit_run or to device code, `info` a dict of its fields plus
    `conflict_free` (False when no XOR choice removes every bank conflict; the
    plan still runs correctly)."""
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    u = _lib.CWarpUnit()
    st = _lib.lib().lc_warp_unit_plan(ctypes.byref(sl), ctypes.byref(dl), int(elem_bytes), ctypes.byref(u))
    if st not in (0, STATUS["LC_ERR_NO_SWIZZLE"]):
        _check(st, "warp_unit_plan")
    n = u.n_modes
    info = {f: getattr(u, f) for f, _ in _lib.CWarpUnit._fields_
            if f not in ("extent", "src_stride", "dst_stride")}
    info["modes"] = [(u.extent[i], u.src_stride[i], u.dst_stride[i]) for i in range(n)]
    info["conflict_free"] = st == 0
    return u, info


def warp_unit_run(src, dst, plan, elem_bytes: int, n_units: int, in_place: bool = False, stream=None) -> None:
    """Runs the warp-scope permute on n_units units staged in shared memory
    (lc_warp_unit_run).  src / dst: CUDA uint8 tensors holding n_units source
    (destination) buffers back to back, src_cosize (dst_cosize) words each."""
    import torch
    for t in (src, dst):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
            raise ValueError("pass contiguous CUDA tensors")
    if src.numel() * src.element_size() < n_units * plan.src_cosize * elem_bytes:
        raise ValueError("src holds fewer than n_units source buffers")
    if dst.numel() * dst.element_size() < n_units * plan.dst_cosize * elem_bytes:
        raise ValueError("dst holds fewer than n_units destination buffers")
    _check(_lib.lib().lc_warp_unit_run(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()),
                                       ctypes.byref(plan), int(elem_bytes), int(n_units), int(bool(in_place)),
                                       ctypes.c_void_p(_stream_handle(stream))), "warp_unit_run")


def choose_swizzle(src_layout, dst_layout, elem_bytes: int) -> dict:
    """The warp permute's XOR swizzle for one warp shard (see lc_choose_swizzle)."""
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    v = [ctypes.c_int32() for _ in range(5)]
    st = _lib.lib().lc_choose_swizzle(ctypes.byref(sl), ctypes.byref(dl), int(elem_bytes),
                                      *[ctypes.byref(x) for x in v])
    if st not in (0, STATUS["LC_ERR_NO_SWIZZLE"]):
        _check(st, "choose_swizzle")
    k, shift, mask, cr, cw = (x.value for x in v)
    return dict(ok=st == 0, k=k, shift=shift, mask=mask, conflicts_read=cr, conflicts_write=cw)


def swizzle_conflicts(src_layout, dst_layout, elem_bytes: int, k: int, shift: int):
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    cr, cw = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.lib().lc_swizzle_conflicts(ctypes.byref(sl), ctypes.byref(dl), int(elem_bytes),
                                           int(k), int(shift), ctypes.byref(cr), ctypes.byref(cw)),
           "swizzle_conflicts")
    return cr.value, cw.value


def gmem_smem_partition(global_layout, shared_layout, elem_bytes: int, threads: int):
    """(vec, outer) of one global <-> shared copy by ``threads`` threads."""
    gl, sl = TileLayout.of(global_layout).to_c(), TileLayout.of(shared_layout).to_c()
    vec, outer = ctypes.c_int32(), ctypes.c_int64()
    _check(_lib.lib().lc_gmem_smem_partition(ctypes.byref(gl), ctypes.byref(sl), int(elem_bytes),
                                             int(threads), ctypes.byref(vec), ctypes.byref(outer)),
           "gmem_smem_partition")
    return vec.value, outer.value


def last_device_error(stream=None):
    """(status, raw word): synchronises the stream, reads and clears the error word."""
    detail = ctypes.c_uint64()
    st = _lib.lib().lc_last_device_error(ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(detail))
    return st, detail.value


def debug_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(_lib.lib().lc_debug_wait_timeout(int(timeout_ns), ctypes.c_void_p(_stream_handle(stream))),
           "debug_wait_timeout")


# ---------------------------------------------------------------------------
# loop-layout override: [(extent, thread_stride, slot_stride), ...], outermost
# first, over the row-major flat index of one tile's logical box
# ---------------------------------------------------------------------------

def _loop_to_c(loop) -> _lib.CLoopLayout:
    modes = [tuple(int(x) for x in m) for m in loop]
    if not 1 <= len(modes) <= _lib.MAX_RANK or any(len(m) != 3 for m in modes):
        raise ValueError("a loop layout is 1..%d modes (extent, thread_stride, slot_stride)" % _lib.MAX_RANK)
    c = _lib.CLoopLayout()
    c.rank = len(modes)
    for k, (e, ts, ss) in enumerate(modes):
        c.shape[k], c.thread_stride[k], c.slot_stride[k] = e, ts, ss
    return c


def loop_layout_default(n_elems: int, num_thread: int, vector_size: int):
    """The default partition of n_elems points as an override (three modes)."""
    c = _lib.CLoopLayout()
    _check(_lib.lib().lc_loop_layout_default(int(n_elems), int(num_thread), int(vector_size),
                                             ctypes.byref(c)), "loop_layout_default")
    return [(c.shape[k], c.thread_stride[k], c.slot_stride[k]) for k in range(c.rank)]


def loop_layout_info(loop, n_elems: int):
    """(threads, slots per thread) of an exact partition of n_elems points."""
    c = _loop_to_c(loop)
    T, L = ctypes.c_int32(), ctypes.c_int64()
    _check(_lib.lib().lc_loop_layout_info(ctypes.byref(c), int(n_elems), ctypes.byref(T), ctypes.byref(L)),
           "loop_layout_info")
    return T.value, L.value


def loop_plan(src_layout, dst_layout, elem_bytes: int, loop, n_tiles: int = 1) -> dict:
    """What layout_copy_loop would do (bases assumed aligned): threads,
    slots per thread, points per tile, vector width in words, split path."""
    info = _lib.CLoopPlanInfo()
    _check(_lib.lib().lc_loop_plan(ctypes.byref(_c_layout(src_layout)), ctypes.byref(_c_layout(dst_layout)),
                                   int(elem_bytes), int(n_tiles), ctypes.byref(_loop_to_c(loop)),
                                   ctypes.byref(info)), "loop_plan")
    return {f: getattr(info, f) for f, _ in _lib.CLoopPlanInfo._fields_}


def layout_copy_loop_ptr(src_ptr: int, src_layout, dst_ptr: int, dst_layout, elem_bytes: int, loop,
                         n_tiles: int = 1, trace_ptr: int = 0, stream=0) -> None:
    """Raw-pointer form of layout_copy_loop (trace_ptr 0: no trace)."""
    sl, dl = _c_layout(src_layout), _c_layout(dst_layout)
    c = _loop_to_c(loop)
    st = _lib.lib().lc_layout_copy_loop(ctypes.c_void_p(src_ptr), ctypes.byref(sl), ctypes.c_void_p(dst_ptr),
                                        ctypes.byref(dl), int(elem_bytes), int(n_tiles), ctypes.byref(c),
                                        ctypes.c_void_p(trace_ptr or None),
                                        ctypes.c_void_p(_stream_handle(stream)))
    _check(st, "layout_copy_loop")


def layout_copy_loop(src, src_layout, dst, dst_layout, loop, n_tiles: int = 1,
                     elem_bytes: int | None = None, trace=None, stream=None) -> None:
    """layout_copy with the partition given by the loop layout ``loop``: one
    CTA per tile, thread t moving the points the override maps to
    (t, 0), (t, 1), ... in order.  ``trace``: optional int64 CUDA tensor of at
    least n_tiles * (points per tile) entries; it receives, for each point,
    thread * slots_per_thread + slot."""
    if not (src.is_cuda and dst.is_cuda):
        raise ValueError("layout_copy_loop needs CUDA tensors (there is no CPU path)")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("pass contiguous tensors; express strides through the layouts")
    w = int(elem_bytes) if elem_bytes is not None else src.element_size()
    if elem_bytes is None and dst.element_size() != w:
        raise ValueError("source and destination element sizes differ; pass elem_bytes")
    sl, dl = _layout_pair(src_layout)[0], _layout_pair(dst_layout)[0]
    for name, t, l in (("source", src, sl), ("destination", dst, dl)):
        need = l.footprint(n_tiles) * w
        have = t.numel() * t.element_size()
        if need > have:
            raise ValueError("%s layout reaches %d bytes; the tensor holds %d" % (name, need, have))
    trace_ptr = 0
    if trace is not None:
        points = 1
        for e in sl.shape:
            points *= int(e)
        if not trace.is_cuda or not trace.is_contiguous() or trace.element_size() != 8 \
                or trace.numel() < n_tiles * points:
            raise ValueError("trace must be a contiguous 8-byte CUDA tensor of >= %d entries"
                             % (n_tiles * points))
        trace_ptr = trace.data_ptr()
    layout_copy_loop_ptr(src.data_ptr(), sl, dst.data_ptr(), dl, w, loop, n_tiles, trace_ptr,
                         _stream_handle(stream))


# ---------------------------------------------------------------------------
# "copy -> gmem_smem": the global <-> shared partition and the staged copy
# ---------------------------------------------------------------------------

def _swizzle_to_c(swizzle):
    if swizzle is None:
        return None
    bits, chunk_log2, row_log2 = (int(x) for x in swizzle)
    return _lib.CSmemSwizzle(bits, chunk_log2, row_log2)


def gmem_smem_plan(global_layout, shared_layout, elem_bytes: int, threads: int, swizzle=None) -> dict:
    """The library's partition of one global <-> shared copy by ``threads``
    threads (host only).  ``swizzle``: (bits, chunk_log2, row_log2) or None."""
    gl, sl = _c_layout(global_layout), _c_layout(shared_layout)
    z = _swizzle_to_c(swizzle)
    out = _lib.CGmemSmem()
    _check(_lib.lib().lc_gmem_smem_plan(ctypes.byref(gl), ctypes.byref(sl), int(elem_bytes), int(threads),
                                        ctypes.byref(z) if z is not None else None, ctypes.byref(out)),
           "gmem_smem_plan")
    n = out.n_modes
    return dict(modes=[(out.extent[i], out.g_stride[i], out.s_stride[i]) for i in range(n)],
                vec=out.vec, outer=out.outer, total=out.total, guarded=bool(out.guarded), threads=out.threads,
                swizzle=(out.swizzle.bits, out.swizzle.chunk_log2, out.swizzle.row_log2))


def layout_copy_staged(src, src_layout, dst, dst_layout, n_tiles: int = 1, elem_bytes: int | None = None,
                       threads: int = 256, swizzle=None, trace_in=None, trace_out=None, stream=None) -> None:
    """layout_copy with each tile staged through shared memory by one CTA of
    ``threads`` threads (the two copies of "copy -> gmem_smem").  ``swizzle``:
    (bits, chunk_log2, row_log2) of the shared tile, or None for the library's
    choice.  ``trace_in`` / ``trace_out``: optional int64 CUDA tensors of
    n_tiles * (elements per tile) entries receiving round * threads + thread
    of the copy that moved each element, indexed by its row-major position."""
    if not (src.is_cuda and dst.is_cuda):
        raise ValueError("layout_copy_staged needs CUDA tensors (there is no CPU path)")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("pass contiguous tensors; express strides through the layouts")
    w = int(elem_bytes) if elem_bytes is not None else src.element_size()
    sl, dl = _layout_pair(src_layout)[0], _layout_pair(dst_layout)[0]
    for name, t, l in (("source", src, sl), ("destination", dst, dl)):
        need = l.footprint(n_tiles) * w
        if need > t.numel() * t.element_size():
            raise ValueError("%s layout reaches %d bytes; the tensor holds %d"
                             % (name, need, t.numel() * t.element_size()))
    points = 1
    for e in sl.shape:
        points *= int(e)
    ptrs = []
    for tr in (trace_in, trace_out):
        if tr is None:
            ptrs.append(None)
            continue
        if not tr.is_cuda or not tr.is_contiguous() or tr.element_size() != 8 or tr.numel() < n_tiles * points:
            raise ValueError("a trace must be a contiguous 8-byte CUDA tensor of >= %d entries" % (n_tiles * points))
        ptrs.append(ctypes.c_void_p(tr.data_ptr()))
    z = _swizzle_to_c(swizzle)
    cs, cd = sl.to_c(), dl.to_c()
    _check(_lib.lib().lc_layout_copy_staged(ctypes.c_void_p(src.data_ptr()), ctypes.byref(cs),
                                            ctypes.c_void_p(dst.data_ptr()), ctypes.byref(cd), w, int(n_tiles),
                                            int(threads), ctypes.byref(z) if z is not None else None,
                                            ptrs[0], ptrs[1], ctypes.c_void_p(_stream_handle(stream))),
           "layout_copy_staged")
