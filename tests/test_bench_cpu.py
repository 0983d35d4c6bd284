"""Host-side helpers of bench.py on the CPU: the oracle timings count the
bytes of the rows they ran and stop on their time budget."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _packed(orc, n):
    out = []
    for i in range(n):
        gv = synth.Gemv(f"t{i}", 128, 512, 2 - (i % 2), 128, "normal", 0.02, 900 + i, 950 + i)
        out.append((gv, orc.pack(gv.weight(), gv.n_keep, gv.group), gv.x(1)))
    return out


def test_oracle_time_counts_rows_and_bytes(orc):
    packed = _packed(orc, 2)
    b, t, rows = bench.oracle_time(packed, 0.05)
    assert t > 0 and rows > 0
    # every row block is 2 rows (128 // 64) of one of the two matrices
    per_row = [gv.packed_bytes() / gv.rows for gv, _, _ in packed]
    assert min(per_row) * rows <= b <= (max(per_row) + 2 + 2 * 512) * rows


def test_oracle_time_threads_whole_passes(orc):
    packed = _packed(orc, 2)
    b, t, rows = bench.oracle_time_threads(packed, 0.05, 4)
    total_rows = sum(gv.rows for gv, _, _ in packed)
    assert rows > 0 and rows % 2 == 0
    assert t >= 0.05
    # at least one whole pass over both matrices, counted once per row block
    assert rows >= total_rows
    nr = 128 // 64
    full_pass = sum(gv.packed_bytes() + (gv.rows // nr) * (2 * gv.cols + 2 * nr)
                    for gv, _, _ in packed)
    assert b >= 0.99 * full_pass * (rows // total_rows)
