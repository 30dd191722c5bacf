"""bench.py's host-side pieces, without a GPU.

The full-size parity tests and the benchmark's reference leg run the oracle
split over the host's cores (tiles, or slabs of the outermost mode, each its
own oracle copy).  The split must give exactly the bytes one serial oracle
call gives, on every workload's structure.
"""
import numpy as np
import pytest

import bench
import oracle
import workloads


@pytest.mark.parametrize("cfg,w", [(1, None), (2, None), (3, None), (4, 1), (4, 2), (4, 16), (5, None),
                                   (6, 1), (6, 8), (8, None)])
@pytest.mark.parametrize("cores", [1, 3, 8])
def test_split_oracle_equals_one_call(cfg, w, cores):
    c = workloads.config(cfg, w, scale="small")
    src = workloads.make_src(c).numpy()
    one = workloads.make_dst(c).numpy()
    split = one.copy()
    oracle.copy(src, c["src"], one, c["dst"], c["elem_bytes"], c["n_tiles"])
    bench.run_oracle(c, src, split, cores)
    assert np.array_equal(one, split)


def test_per_config_list_parsing():
    assert bench.parse_per_config(None) == bench.PER_CONFIG
    assert bench.parse_per_config("3,4:1,5") == [(3, None), (4, 1), (5, None)]
    for c_id, c_w in bench.PER_CONFIG:
        workloads.config(c_id, c_w)  # every listed workload exists at full size
