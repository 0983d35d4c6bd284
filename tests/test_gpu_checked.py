"""The checked build (libsgemv_checked.so, -DSGEMV_CHECKED): the product
kernels validate every 2:4 position nibble they decode (a < b) and every
group and chunk index they form, and record a device error instead of
reading out of range.  On valid packed weights -- every case below -- the
checked kernels must agree with the oracle and leave the error word clean.

The library is loaded in a child process, so that this process keeps the
product library it has loaded.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = r'''
import sys
sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
import numpy as np, torch
import oracle, synth
import sparse_weight_only_gb300 as swo
from _check import check_y
swo.load(LIB)
oracle.build()
shapes = [(300, 1024, 2, 64), (257, 2304, 2, 256), (96, 4160, 1, 64), (129, 512, 1, 256),
          (1100, 4096, 2, 128), (24, 16384, 1, 128)]
for rows, cols, n, g in shapes:
    W = synth.weight_outliers(rows + cols, rows, cols)
    p = oracle.pack(W, n, g)
    h = swo.SparseGemv(rows, cols, n, g, max_m=64)
    h.pack(W)                                   # the packer too runs checked code
    norms = np.abs(oracle.dequant(p)).sum(axis=1)
    for m in (1, 4, 16, 24, 32, 40, 48, 64):
        x = synth.activations(m + rows, m, cols)
        xd = torch.from_numpy(x).cuda()
        y = torch.empty((m, rows), dtype=torch.float16, device="cuda")
        h.run(xd, y)
        torch.cuda.synchronize()
        assert h.status() == 0, (rows, cols, n, g, m, swo.load().sgemv_last_error())
        check_y(oracle, y.cpu().numpy(), oracle.matvec(p, x), norms, f"checked {rows}x{cols} m={m}")
# grouped, both N in one launch
mats = []
for i, (rows, n, g) in enumerate([(300, 1, 256), (129, 2, 128), (64, 1, 128), (200, 2, 64)]):
    W = synth.weight_outliers(400 + i, rows, 1536)
    p = oracle.pack(W, n, g)
    h = swo.SparseGemv(rows, 1536, n, g)
    h.import_canonical(p.vals, p.idx, p.scale, p.zero)
    mats.append((h, p))
x = torch.from_numpy(synth.activations(7, 1, 1536)).cuda()
ys = [torch.empty((1, h.rows), dtype=torch.float16, device="cuda") for h, _ in mats]
swo.run_group([h for h, _ in mats], x, ys)
torch.cuda.synchronize()
for (h, p), y in zip(mats, ys):
    assert h.status() == 0
    check_y(oracle, y.cpu().numpy(), oracle.matvec(p, x.cpu().numpy()),
            np.abs(oracle.dequant(p)).sum(axis=1), "checked group")
print("checked build clean")
'''


def test_checked_build_runs_clean():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from sparse_weight_only_gb300.build import build
    lib = build(variant="checked")
    code = f"import os\nROOT = {ROOT!r}\nLIB = {lib!r}\n" + CASES
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked build clean" in r.stdout
