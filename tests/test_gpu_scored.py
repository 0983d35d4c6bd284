"""Eq. 3 importance pruning on the GPU (sgemv_pack_scored through the C ABI)
against the oracle: the exported canonical bytes are identical, and the
product of the packed weight matches the oracle's fp64 product.

Method: Dong et al., "Efficient LLM ad generation via model compression and
parallel verification" (arXiv 2605.11582), section 3.2 (Sparsification,
Eq. 3): score = |W_ij| * ||X_j||_2 + |W_ij| * |dE/dW_ij|.
"""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _inputs(seed, rows, cols):
    rng = np.random.default_rng(seed)
    W = synth.weight_outliers(seed, rows, cols)
    xnorm = rng.uniform(0.0, 3.0, cols).astype(np.float32)
    xnorm[rng.integers(0, cols, 8)] = 0.0          # silent input channels
    grad = rng.normal(0.0, 0.05, (rows, cols)).astype(np.float32)
    return W, xnorm, grad


def _same_bytes(h, p):
    vals, idx, scale, zero = h.export_canonical()
    assert np.array_equal(vals, p.vals), "vals differ"
    assert np.array_equal(idx, p.idx), "idx differ"
    assert np.array_equal(scale, p.scale), "scale differs"
    assert np.array_equal(zero, p.zero), "zero differs"


SHAPES = [  # rows, cols, n_keep, group
    (33, 256, 2, 128),
    (64, 192, 1, 64),       # 1:4, cols % 128 == 64
    (100, 1024, 1, 256),
    (257, 2304, 2, 64),
]


@pytest.mark.parametrize("rows,cols,n_keep,group", SHAPES)
@pytest.mark.parametrize("with_grad", [True, False])
def test_pack_scored_bytes_match_oracle(native, orc, rows, cols, n_keep, group, with_grad):
    W, xnorm, grad = _inputs(rows + cols, rows, cols)
    g = grad if with_grad else None
    p = orc.pack_scored(W, xnorm, g, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group)
    h.pack_scored(W, xnorm, g)
    _same_bytes(h, p)
    # the scores changed the selection (not a disguised magnitude pack)
    assert not np.array_equal(p.idx, orc.pack(W, n_keep, group).idx)


def test_pack_scored_power_of_two_norms_is_magnitude(native, orc):
    W = synth.weight_normal(9, 40, 512, 0.02)
    for n_keep, group in ((2, 128), (1, 64)):
        h = native.SparseGemv(40, 512, n_keep, group)
        h.pack_scored(W, np.full(512, 4.0, np.float32), None)
        _same_bytes(h, orc.pack(W, n_keep, group))


@pytest.mark.parametrize("m", [1, 4])
def test_run_after_scored_pack(native, orc, m):
    rows, cols, n_keep, group = 300, 4096, 2, 64
    W, xnorm, grad = _inputs(77, rows, cols)
    p = orc.pack_scored(W, xnorm, grad, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=4)
    h.pack_scored(W, xnorm, grad)
    x = synth.activations(5 + m, m, cols)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty((m, rows), dtype=torch.float16, device="cuda")
    h.run(xd, y)
    torch.cuda.synchronize()
    assert h.status() == 0
    ref = orc.matvec(p, x)
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    check_y(orc, y.cpu().numpy(), ref, norms, "scored pack")


def test_pack_scored_rejects_bad_inputs(native):
    from sparse_weight_only_gb300 import SgemvError
    W = np.ones((16, 256), np.float32)
    h = native.SparseGemv(16, 256, 2, 64)
    xn = np.ones(256, np.float32)
    for bad, code in ((-1.0, native.SGEMV_ERR_ARG), (np.nan, native.SGEMV_ERR_NONFINITE),
                      (np.inf, native.SGEMV_ERR_NONFINITE)):
        x2 = xn.copy()
        x2[17] = bad
        with pytest.raises(SgemvError) as e:
            h.pack_scored(W, x2)
        assert e.value.code == code
    g = np.zeros_like(W)
    g[3, 200] = np.nan
    with pytest.raises(SgemvError) as e:
        h.pack_scored(W, xn, g)
    assert e.value.code == native.SGEMV_ERR_NONFINITE
    # the handle is left unpacked
    x = torch.zeros((1, 256), dtype=torch.float16, device="cuda")
    y = torch.empty((1, 16), dtype=torch.float16, device="cuda")
    with pytest.raises(SgemvError) as e:
        h.run(x, y)
    assert e.value.code == native.SGEMV_ERR_STATE


def test_pack_scored_with_row_groups(native, orc):
    """Eq. 3 pruning on a handle with a group size per row: the oracle's
    scored pruning, then its per-row quantisation and encoding."""
    rows, cols = 90, 1024
    W, xnorm, grad = _inputs(12, rows, cols)
    rg = np.random.default_rng(13).choice([64, 128, 256], rows).astype(np.int32)
    for n_keep in (1, 2):
        pos = orc.prune_scored(W, xnorm, grad, n_keep)
        q, sc, z = orc.quantize_rowg(W, pos, n_keep, rg)
        vals, idx = orc.encode(pos, q, rows, cols, n_keep)
        h = native.SparseGemv(rows, cols, n_keep, None, row_group=rg)
        h.pack_scored(W, xnorm, grad)
        ev, ei, es, ez = h.export_canonical()
        assert np.array_equal(ev, vals) and np.array_equal(ei, idx)
        assert np.array_equal(es, sc) and np.array_equal(ez, z)
