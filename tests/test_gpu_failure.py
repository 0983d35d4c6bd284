"""Failure detection on the GPU without a GPU fault.

The small-batch kernel's split-K reduction is the library's one device-side
wait on other CTAs, and it is bounded.  The test hook sgemv_debug_withhold
makes every cluster rank withhold its partial sums (nothing is sent, so no
remote store is in flight) and shortens the limit: the wait runs out, the
kernel records SGEMV_ERR_TIMEOUT in the handle's error word and returns, and
the device stays usable -- the next call is correct.
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


@pytest.mark.parametrize("m", [2, 4, 16])
def test_bounded_wait_runs_out_and_recovers(native, orc, m):
    rows, cols = 256, 4096          # two row tiles: clusters of several ranks
    h, p = _setup(native, orc, rows, cols, 2, 128, max_m=16)
    x = synth.activations(40 + m, m, cols)
    norms = np.abs(orc.dequant(p)).sum(axis=1)

    h.debug_withhold(1)
    _run(h, x)
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_ERR_TIMEOUT
    assert "split-K" in native.load().sgemv_last_error().decode()
    assert h.status() == native.SGEMV_OK      # the word was cleared

    for _ in range(2):                         # later calls run normally
        y = _run(h, x)
        torch.cuda.synchronize()
        assert h.status() == native.SGEMV_OK
        check_y(orc, y.cpu().numpy(), orc.matvec(p, x), norms, f"after timeout m={m}")


def test_withhold_leaves_other_kernels_alone(native, orc):
    """m = 1 and the pulled reduction (m > 16) have no such wait: the hook
    is not consumed by them and their results stay exact."""
    rows, cols = 256, 4096
    h, p = _setup(native, orc, rows, cols, 2, 128, max_m=64)
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    h.debug_withhold(1)
    for m in (1, 33):
        x = synth.activations(70 + m, m, cols)
        y = _run(h, x)
        torch.cuda.synchronize()
        assert h.status() == native.SGEMV_OK
        check_y(orc, y.cpu().numpy(), orc.matvec(p, x), norms, f"m={m}")
    # the pending hook still fires on the next eligible call
    _run(h, synth.activations(5, 4, cols))
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_ERR_TIMEOUT
    h.debug_withhold(0)


def test_withhold_rejects_negative(native):
    h = native.SparseGemv(8, 64, 2, 64)
    with pytest.raises(native.SgemvError) as e:
        h.debug_withhold(-1)
    assert e.value.code == native.SGEMV_ERR_ARG
