"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: bit-exact pack for every matrix, and y checked against
the oracle on sampled rows (the oracle computes them one by one)."""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N_SAMPLE = 192


def _sample_rows(rows, seed):
    g = synth.rng(seed)
    pick = g.choice(rows, size=min(rows, N_SAMPLE - 2), replace=False)
    return np.unique(np.concatenate([pick, [0, rows - 1]])).astype(np.int64)


def _check_gemv(native, orc, gv, m):
    W = gv.weight()
    p = orc.pack(W, gv.n_keep, gv.group)
    h = native.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, max_m=max(m, 1))
    h.pack(W)
    vals, idx, scale, zero = h.export_canonical()
    assert np.array_equal(vals, p.vals) and np.array_equal(idx, p.idx)
    assert np.array_equal(scale, p.scale) and np.array_equal(zero, p.zero)
    del W
    x = gv.x(m)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty((m, gv.rows), dtype=torch.float16, device="cuda")
    h.run(xd, y)
    torch.cuda.synchronize()
    assert h.status() == 0
    rows = _sample_rows(gv.rows, gv.w_seed)
    ref = orc.matvec(p, x, rows)
    norms = np.array([np.abs(orc.dequant(p, int(r), 1)).sum() for r in rows])
    return check_y(orc, y.cpu().numpy()[:, rows], ref, norms,
                   f"{gv.name} m={m}")


@pytest.mark.parametrize("cfg", ["1", "2", "3", "5"])
def test_config_m1(native, orc, cfg):
    for gv in synth.CONFIGS[cfg]():
        _check_gemv(native, orc, gv, 1)


@pytest.mark.parametrize("m", synth.CONFIG4_M)
def test_config4_batch(native, orc, m):
    gvs = synth.config4()
    # one square and one rectangular matrix per M keeps the suite short;
    # all seven at M = 64, the largest batch
    pick = gvs if m == 64 else [gvs[0], gvs[6]]
    for gv in pick:
        _check_gemv(native, orc, gv, m)


@pytest.mark.parametrize("m", [4, 16, 24, 40, 64])
def test_layerset_batch_mixed(native, orc, m):
    """The config-3 layer set (2:4 and 1:4, groups 64..256) with M activation
    rows: the 1:4 matrices take the 2:4 sparse MMAs with zero partners."""
    gvs = synth.config3()
    pick = gvs if m == 16 else [g for g in gvs if g.n_keep == 1]
    for gv in pick:
        _check_gemv(native, orc, gv, m)
