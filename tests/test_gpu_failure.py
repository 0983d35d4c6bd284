"""Failure detection on the GPU without a GPU fault.

Every wait of the batch kernels on their own copies and MMAs is bounded
(2 <= m <= 8: the pushed split-K sums; 33 <= m <= 64: the tcgen05 kernel's
copies and MMAs; 9 <= m <= 32 waits on cluster barriers only).  The test hook
sgemv_debug_withhold makes the kernel withhold its x
loads (nothing is in flight that it would have to wait for) and shortens the
limit: the wait runs out, the kernel records SGEMV_ERR_TIMEOUT in the
handle's error word, lets the copies it did issue land, frees its tensor
memory and returns, and the device stays usable -- the next calls are
correct, including tiles whose split-K counters the aborted launch left.
"""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _setup(native, orc, rows, cols, n_keep, group, max_m):
    W = synth.weight_outliers(rows + cols, rows, cols)
    p = orc.pack(W, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=max_m)
    h.import_canonical(p.vals, p.idx, p.scale, p.zero)
    return h, p


def _run(h, x):
    xd = torch.from_numpy(x).cuda()
    y = torch.empty((x.shape[0], h.rows), dtype=torch.float16, device="cuda")
    h.run(xd, y)
    return y


@pytest.mark.parametrize("m", [2, 4, 8, 33, 48, 64])
def test_bounded_wait_runs_out_and_recovers(native, orc, m):
    rows, cols = 256, 4096          # two row tiles: clusters of several ranks
    h, p = _setup(native, orc, rows, cols, 2, 128, max_m=64)
    x = synth.activations(40 + m, m, cols)
    norms = np.abs(orc.dequant(p)).sum(axis=1)

    h.debug_withhold(1)
    _run(h, x)
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_ERR_TIMEOUT
    assert "gave up" in native.load().sgemv_last_error().decode()
    assert h.status() == native.SGEMV_OK      # the word was cleared

    for _ in range(2):                         # later calls run normally
        y = _run(h, x)
        torch.cuda.synchronize()
        assert h.status() == native.SGEMV_OK
        check_y(orc, y.cpu().numpy(), orc.matvec(p, x), norms, f"after timeout m={m}")


def test_withhold_leaves_m1_alone(native, orc):
    """m = 1 has no such wait: the hook is not consumed by it and its result
    stays exact; the pending hook fires on the next batch call."""
    rows, cols = 256, 4096
    h, p = _setup(native, orc, rows, cols, 2, 128, max_m=64)
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    h.debug_withhold(1)
    x = synth.activations(71, 1, cols)
    y = _run(h, x)
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_OK
    check_y(orc, y.cpu().numpy(), orc.matvec(p, x), norms, "m=1")
    _run(h, synth.activations(5, 4, cols))
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_ERR_TIMEOUT
    h.debug_withhold(0)


@pytest.mark.parametrize("m", [9, 16, 17, 24, 25, 32])
def test_withhold_leaves_pulled_sums_alone(native, orc, m):
    """9 <= m <= 32 pulls the split-K sums between cluster barriers and
    waits on no copy: the hook is not consumed and the result stays exact;
    the pending hook fires on the next call with a bounded wait."""
    rows, cols = 256, 4096
    h, p = _setup(native, orc, rows, cols, 2, 128, max_m=64)
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    h.debug_withhold(1)
    x = synth.activations(72 + m, m, cols)
    y = _run(h, x)
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_OK
    check_y(orc, y.cpu().numpy(), orc.matvec(p, x), norms, f"m={m}")
    _run(h, synth.activations(6, 8, cols))
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_ERR_TIMEOUT
    h.debug_withhold(0)


def test_timeout_in_a_1of4_multi_tile_matrix_recovers(native, orc):
    """A larger 1:4 matrix, many CTAs sharing tiles: after the aborted launch
    every tile's split-K counter is back at zero, so the next results are
    exact."""
    rows, cols = 1100, 4096
    h, p = _setup(native, orc, rows, cols, 1, 64, max_m=8)
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    x = synth.activations(90, 8, cols)
    h.debug_withhold(1)
    _run(h, x)
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_ERR_TIMEOUT
    for _ in range(2):
        y = _run(h, x)
        torch.cuda.synchronize()
        assert h.status() == native.SGEMV_OK
        check_y(orc, y.cpu().numpy(), orc.matvec(p, x), norms, "1:4 after timeout")


def test_withhold_rejects_negative(native):
    h = native.SparseGemv(8, 64, 2, 64)
    with pytest.raises(native.SgemvError) as e:
        h.debug_withhold(-1)
    assert e.value.code == native.SGEMV_ERR_ARG
