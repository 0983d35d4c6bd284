"""sgemv_run_noalloc: the batch product for callers that cannot allocate
device memory when they run it (an allocator that owns all device memory, a
plug-in handed buffers but no right to allocate).  The entry point runs the
batch kernel on a split-K workspace that is a fixed array inside the library
instead of the handle's own; its result must match sgemv_run's within the
tolerance the other parity tests use, on two calls in a row (the second
finds the array as the first left it).  This file is collected last, so that
a run stopping at the first failure has run every other test already.
"""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _handle(native, orc, rows, cols, n_keep, group, max_m, seed):
    W = synth.weight_outliers(seed, rows, cols)
    p = orc.pack(W, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=max_m)
    h.import_canonical(p.vals, p.idx, p.scale, p.zero)
    return h, p


@pytest.mark.parametrize("rows,cols,n_keep,group,m", [
    (4096, 4096, 2, 128, 16),     # many CTAs share every row tile
    (1100, 4096, 1, 64, 33),      # 1:4, ragged last tile
    (300, 1024, 2, 256, 64),      # the widest batch
])
def test_noalloc_matches_run(native, orc, rows, cols, n_keep, group, m):
    h, p = _handle(native, orc, rows, cols, n_keep, group, 64, rows + m)
    x = torch.from_numpy(synth.activations(m + 3, m, cols)).cuda()
    y_run = torch.empty((m, rows), dtype=torch.float16, device="cuda")
    h.run(x, y_run)
    torch.cuda.synchronize()
    assert h.status() == native.SGEMV_OK
    ref = y_run.cpu().numpy()
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    y_ref64 = orc.matvec(p, x.cpu().numpy())
    for call in range(2):                       # two calls in a row
        y = torch.full((m, rows), 7.0, dtype=torch.float16, device="cuda")
        h.run_noalloc(x, y)
        torch.cuda.synchronize()
        assert h.status() == native.SGEMV_OK
        got = y.cpu().numpy()
        # against the existing entry point's output, within the parity tolerance
        check_y(orc, got, ref.astype(np.float64), norms, f"noalloc vs run, call {call}")
        # and against the oracle, like every other product
        check_y(orc, got, y_ref64, norms, f"noalloc vs oracle, call {call}")


def test_noalloc_on_a_handle_after_another(native, orc):
    """The shared array keeps the previous call's contents: a different
    matrix right after still gets its counters from zero."""
    a, pa = _handle(native, orc, 2048, 4096, 2, 64, 16, 11)
    b, pb = _handle(native, orc, 640, 2048, 1, 128, 16, 12)
    for h, p in ((a, pa), (b, pb), (a, pa)):
        x = torch.from_numpy(synth.activations(5, 16, h.cols)).cuda()
        y = torch.empty((16, h.rows), dtype=torch.float16, device="cuda")
        h.run_noalloc(x, y)
        torch.cuda.synchronize()
        assert h.status() == native.SGEMV_OK
        check_y(orc, y.cpu().numpy(), orc.matvec(p, x.cpu().numpy()),
                np.abs(orc.dequant(p)).sum(axis=1), "alternating handles")


def test_noalloc_rejects_out_of_range(native, orc):
    h, _ = _handle(native, orc, 64, 256, 2, 64, 8, 3)
    x = torch.zeros((1, 256), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(native.SgemvError) as e:
        h.run_noalloc(x, y)                     # m = 1: no workspace needed
    assert e.value.code == native.SGEMV_ERR_ARG
    x9 = torch.zeros((9, 256), dtype=torch.float16, device="cuda")
    y9 = torch.zeros((9, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(native.SgemvError) as e:
        h.run_noalloc(x9, y9)                   # m > max_m
    assert e.value.code == native.SGEMV_ERR_ARG
    # more row tiles than the fixed counters hold
    big = native.SparseGemv(16384 * 128 + 1, 64, 2, 64, max_m=2)
    big.import_canonical(*_zero_canonical(big))
    xb = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
    yb = torch.zeros((2, big.rows), dtype=torch.float16, device="cuda")
    with pytest.raises(native.SgemvError) as e:
        big.run_noalloc(xb, yb)
    assert e.value.code == native.SGEMV_ERR_UNSUPPORTED
    assert "2,097,152" in str(e.value)


def _zero_canonical(h):
    s = h.sizes()
    return (np.zeros(s["vals"], np.uint8),
            np.full(s["idx"], 0x44, np.uint8),   # positions (0, 1) in every quad
            np.full(s["groups"], 0x3C00, np.uint16), np.zeros(s["groups"], np.uint16))
