"""Oracle for the strided tile layout copy / permute.

TEST INFRASTRUCTURE.  A plain, slow, obviously correct CPU statement of what
the GPU library computes, written from the pages and checked against what the
pages and the mathematics fix (``tests/test_oracle_pins.py``).  Only the test
suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
leg may import or run it; the product library (``movement_primitives_gb300``)
never does, and the two share no code.

Contents
  definition   the copy's definition (every logical index moves one raw word),
               with the word loop in plain C (copy_oracle.c)
  index_maps   flatten / unflatten / default loop partition (TileLang tutorial
               "loop_mapping.py") and its ``loop_layout=`` override, with the
               override's serial replay; the [outer, threads, vec] partition and its
               serial loop (Apache TVM "copy -> gmem_smem"); the aligned warp
               permute and its two register-staged phases (Apache TVM
               "permute_layout")
  banks        the shared-memory bank simulator and the XOR-bit choice
               (Apache TVM "permute_layout", "Algorithm" step 2)
  stencil      the window sum of MLC "Ep7", "Window Sum Example"

Every function is pinned by at least one test; nothing here is "parity
unpinned".
"""
from . import banks, build, definition, index_maps, stencil  # noqa: F401
from .definition import Layout, copy, offsets_of, paired_modes, cosize  # noqa: F401
