"""The allocation-free host-buffer copy (lc_layout_copy_host_static).

Callers that cannot allocate device memory -- a plugin whose host
application's allocator owns all device memory, or code that must not call
cudaMalloc because it can synchronise the whole device -- cannot hand
lc_layout_copy_host a staging buffer.  This entry point stages through a
fixed array inside the library instead.  Here it is called through the C ABI
and must give exactly what lc_layout_copy_host gives, on two calls in a row
(the array keeps the previous call's bytes), and both must equal the oracle,
so that a fault shared by the two library paths (the planner, the kernels)
would show too.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import movement_primitives_gb300
    return movement_primitives_gb300


def L(shape, stride, offset=0, tile_stride=0):
    return dict(shape=tuple(shape), stride=tuple(stride), offset=offset, tile_stride=tile_stride)


def _static_call(M, src_h, src_l, dst_h, dst_l, w, n_tiles):
    """lc_layout_copy_host_static straight through ctypes."""
    sl, dl = M.TileLayout.of(src_l).to_c(), M.TileLayout.of(dst_l).to_c()
    stream = torch.cuda.current_stream()
    return M._lib.lib().lc_layout_copy_host_static(
        ctypes.c_void_p(src_h.data_ptr()), ctypes.byref(sl), ctypes.c_void_p(dst_h.data_ptr()),
        ctypes.byref(dl), int(w), int(n_tiles), ctypes.c_void_p(stream.cuda_stream))


def _compare(M, src_l, dst_l, w, n_tiles, seed):
    ns = workloads.footprint_elems(src_l, n_tiles) * w
    nd = workloads.footprint_elems(dst_l, n_tiles) * w
    g = torch.Generator().manual_seed(seed)
    for call in range(2):  # two calls in a row, fresh source bytes each time
        src_h = torch.randint(0, 256, (ns,), generator=g, dtype=torch.uint8).pin_memory()
        fill = torch.randint(0, 256, (nd,), generator=g, dtype=torch.uint8)
        want = fill.clone().pin_memory()
        got = fill.clone().pin_memory()
        M.layout_copy_host(src_h, src_l, want, dst_l, n_tiles=n_tiles, elem_bytes=w)
        torch.cuda.current_stream().synchronize()
        assert _static_call(M, src_h, src_l, got, dst_l, w, n_tiles) == 0
        torch.cuda.current_stream().synchronize()
        assert np.array_equal(got.numpy(), want.numpy()), "call %d differs" % call
        expect = fill.numpy().copy()
        oracle.copy(src_h.numpy(), src_l, expect, dst_l, w, n_tiles)
        assert np.array_equal(got.numpy(), expect), "call %d differs from the oracle" % call


def test_static_staging_matches_pipelined_host_copy(M):
    sh = (2, 1, 4, 32)
    sf_src, sf_dst = L(sh, (128, 128, 32, 1)), L(sh, (128, 128, 1, 4))
    _compare(M, sf_src, sf_dst, 4, 4099, seed=1)             # one chunk
    _compare(M, sf_src, sf_dst, 4, (1 << 16) + 5, seed=2)    # 64 MiB a side: several chunks
    _compare(M, L((4, 32), (32, 1)), L((4, 32), (1, 4), 8, 200), 2, 301, seed=3)  # holes
    c = workloads.config(3, scale="small")                   # one tile, a transpose
    _compare(M, c["src"], c["dst"], 2, 1, seed=4)


def test_static_staging_warp_shuffle_and_transposes(M):
    c = workloads.config(4, 1, scale="small")                # one-byte transpose
    _compare(M, c["src"], c["dst"], 1, 1, seed=5)
    V = 4                                                      # the shuffle's blocks, mirrored
    _compare(M, L((64, V), (V, 1)), L((64, V), (1, 64)), 4, 1001, seed=6)


def test_static_staging_refuses_oversized_tiles(M):
    # one 8192 x 8192 one-byte tile needs 64 MiB a side, beyond the 32 MiB array
    src_h = torch.zeros(8192 * 8192, dtype=torch.uint8)
    dst_h = torch.zeros(8192 * 8192, dtype=torch.uint8)
    st = _static_call(M, src_h, L((8192, 8192), (8192, 1)), dst_h, L((8192, 8192), (1, 8192)), 1, 1)
    assert st == M.STATUS["LC_ERR_STAGING"]
    assert M._lib.STATIC_STAGING_BYTES == 32 * 1024 * 1024
