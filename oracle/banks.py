"""Shared-memory bank simulator and the XOR-bit choice of the warp permute.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Apache TVM docs "permute_layout", section "Algorithm" step 2: the simulator
tries k = 0, 1, ..., log2(P) and keeps the smallest k whose shift and mask
(mask = 2**k - 1) make BOTH the read phase and the write phase free of bank
conflicts; section "What it accepts" (row "bank-freedom"): if no k works the
variant fails.

Readings (the page leaves these open):
* shift is searched upward from 0 to 5 - k for each k, first conflict-free
  pair wins (smallest k, then smallest shift); k = 0 needs no shift.
* P must be a power of two for k > 0, so the XOR keeps j below P.
* bank model "hardware": 32 banks of 4-byte words, bank = (byte address / 4)
  mod 32; a warp access is served in wavefronts of 128 bytes (32 lanes for
  accesses of up to 4 bytes, 16 lanes for 8 bytes, 8 lanes for 16 bytes);
  the degree of a wavefront is the largest number of DISTINCT 4-byte words
  any one bank must deliver (lanes reading the same word share it).
* bank model "strict": as above, but distinct ELEMENTS in one bank count
  separately, so several sub-4-byte elements packed in one word conflict.
  This is the reading under which the page's remark holds that stride-1
  reads of words under 4 bytes put several lanes in one bank and can make the choice
  fail; for 4-byte and wider elements the two models agree.
Byte addresses are element offsets times the element size, relative to a
128-byte-aligned base.
"""
from __future__ import annotations

from .index_maps import WARP, swizzled_iteration, unflatten, project

BANKS = 32
WORD = 4


def wavefront_lanes(elem_bytes: int) -> int:
    return WARP if elem_bytes <= WORD else 128 // elem_bytes


def access_degree(byte_addrs, elem_bytes: int, model: str = "hardware") -> int:
    """Worst bank degree of one warp-wide access (one address per lane)."""
    per = wavefront_lanes(elem_bytes)
    worst = 0
    for start in range(0, len(byte_addrs), per):
        banks = {}
        for a in byte_addrs[start:start + per]:
            first, last = a // WORD, (a + elem_bytes - 1) // WORD
            for word in range(first, last + 1):
                key = word if (model == "hardware" or elem_bytes >= WORD) else a
                banks.setdefault(word % BANKS, set()).add(key)
        worst = max([worst] + [len(v) for v in banks.values()])
    return worst


def phase_degrees(extent, src_str, dst_str, elem_bytes, k, shift, model="hardware"):
    """(read degree, write degree), each the worst over the P unrolled steps."""
    total = 1
    for e in extent:
        total *= e
    P = total // WARP
    rd = wd = 0
    for r in range(P):
        reads, writes = [], []
        for lane in range(WARP):
            idx = unflatten(lane + WARP * swizzled_iteration(lane, r, k, shift), extent)
            reads.append(project(idx, src_str) * elem_bytes)
            writes.append(project(idx, dst_str) * elem_bytes)
        rd = max(rd, access_degree(reads, elem_bytes, model))
        wd = max(wd, access_degree(writes, elem_bytes, model))
    return rd, wd


def choose_xor_k(extent, src_str, dst_str, elem_bytes, model="hardware"):
    """Smallest (k, shift) conflict-free in both phases.

    Returns (k, shift, mask, read_degree, write_degree), or None when no k in
    [0, log2 P] works (the page's "fail").
    """
    total = 1
    for e in extent:
        total *= e
    P = total // WARP
    kmax = P.bit_length() - 1 if P > 0 and (P & (P - 1)) == 0 else 0
    for k in range(kmax + 1):
        for shift in (range(0, 5 - k + 1) if k else (0,)):
            rd, wd = phase_degrees(extent, src_str, dst_str, elem_bytes, k, shift, model)
            if rd <= 1 and wd <= 1:
                return k, shift, (1 << k) - 1, rd, wd
    return None
