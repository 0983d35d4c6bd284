"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Pack parity is bit-exact: the library's sgemv_pack followed by
sgemv_export must reproduce the oracle's canonical bytes.  Kernel parity
isolates the product kernels: the oracle's bytes are imported, run on the
GPU, and y is compared with the oracle's fp64 y under the tolerance in
tests/_check.py.
"""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev():
    return torch.device("cuda:0")


def _lib_pack(native, W, n_keep, group, max_m=1):
    rows, cols = W.shape
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=max_m)
    h.pack(W)
    return h


def _assert_same_bytes(h, p):
    vals, idx, scale, zero = h.export_canonical()
    assert np.array_equal(vals, p.vals), "vals differ"
    assert np.array_equal(idx, p.idx), "idx differ"
    assert np.array_equal(scale, p.scale), "scale differs"
    assert np.array_equal(zero, p.zero), "zero differs"


def _run(h, x_np):
    x = torch.from_numpy(np.ascontiguousarray(x_np)).to(_dev())
    y = torch.empty((x.shape[0], h.rows), dtype=torch.float16, device=_dev())
    h.run(x, y)
    torch.cuda.synchronize()
    assert h.status() == 0
    return y.cpu().numpy()


def _rownorm(orc, p, rows):
    return np.array([np.abs(orc.dequant(p, int(r), 1)).sum() for r in rows])


SMALL = [  # rows, cols, n_keep, group, dist
    (1, 64, 2, 64, "normal"),
    (7, 128, 1, 64, "outliers"),      # ragged: 1:4 chunk half full
    (33, 256, 2, 128, "outliers"),
    (64, 192, 1, 64, "normal"),       # 1:4, cols % 128 == 64
    (129, 512, 1, 256, "outliers"),
    (300, 1024, 2, 64, "outliers"),
    (257, 2304, 2, 256, "normal"),
    (96, 4160, 1, 64, "outliers"),    # 1:4 ragged tail, K not a multiple of 128
    (50, 8192, 1, 128, "normal"),     # longer rows: several chunks per lane
    (40, 8192, 1, 256, "outliers"),
    (24, 16384, 2, 128, "outliers"),  # rows longer than one K slice
    (24, 16384, 1, 64, "normal"),
    (70, 4160, 2, 64, "outliers"),    # M=1: three items per row, the last one lane wide
    (33, 6144, 2, 128, "normal"),     # three full items per row
    (20, 10240, 2, 256, "outliers"),  # K slices of three and two items per row
    (17, 11008, 1, 128, "normal"),    # 1:4 K slices of two items and one ragged item
]


def _weight(seed, rows, cols, dist):
    if dist == "normal":
        return synth.weight_normal(seed, rows, cols, 0.02)
    return synth.weight_outliers(seed, rows, cols)


@pytest.mark.parametrize("rows,cols,n_keep,group,dist", SMALL)
def test_pack_parity_small(native, orc, rows, cols, n_keep, group, dist):
    W = _weight(rows * 7 + cols, rows, cols, dist)
    p = orc.pack(W, n_keep, group)
    h = _lib_pack(native, W, n_keep, group)
    _assert_same_bytes(h, p)


def test_pack_parity_tie_alphabet(native, orc):
    """Every quad of a tie-heavy alphabet (signed zeros, equal magnitudes)."""
    import itertools
    alphabet = [0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0]
    quads = np.array(list(itertools.product(alphabet, repeat=4)), np.float32)
    quads = np.concatenate([quads, np.zeros((2560 - len(quads), 4), np.float32)])
    W = quads.reshape(40, 256)
    for n_keep in (1, 2):
        for group in (64, 128, 256):
            _assert_same_bytes(_lib_pack(native, W, n_keep, group),
                               orc.pack(W, n_keep, group))


def test_pack_parity_special_groups(native, orc):
    W = np.zeros((6, 256), np.float32)
    W[1] = 1e-12                      # scale underflows -> 2^-24
    W[2] = np.abs(synth.weight_normal(3, 1, 256, 0.02))      # z = 0
    W[3] = -np.abs(synth.weight_normal(4, 1, 256, 0.02))     # z = 15
    W[4, ::7] = 1.0                   # sparse spikes
    W[5] = np.float32(2.0 ** -6) * np.arange(256) % np.float32(0.2)
    for n_keep in (1, 2):
        _assert_same_bytes(_lib_pack(native, W, n_keep, 64),
                           orc.pack(W, n_keep, 64))


def test_pack_parity_ties_to_even(native, orc):
    """Halfway quantiser cases (tests/_ties.py): the GPU packer's codes equal
    the hand-derived ties-to-even table, and the oracle's bytes."""
    import _ties
    for n_keep in (1, 2):
        for group in (64, 128):
            W, _ = _ties.weight(n_keep, group)
            h = _lib_pack(native, W, n_keep, group)
            vals, idx, scale, zero = h.export_canonical()
            ev, ei, es, ez = _ties.expected_bytes(n_keep, group)
            assert np.array_equal(vals, ev) and np.array_equal(idx, ei)
            assert np.array_equal(scale, es) and np.array_equal(zero, ez)
            _assert_same_bytes(h, orc.pack(W, n_keep, group))


@pytest.mark.parametrize("rows,cols,n_keep,group,dist", SMALL)
@pytest.mark.parametrize("m", [1, 3, 8])
def test_run_parity_small(native, orc, rows, cols, n_keep, group, dist, m):
    W = _weight(rows * 11 + cols, rows, cols, dist)
    p = orc.pack(W, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=8)
    h.import_canonical(p.vals, p.idx, p.scale, p.zero)
    _assert_same_bytes(h, p)          # import/export round trip
    x = synth.activations(rows + m, m, cols)
    y = _run(h, x)
    ref = orc.matvec(p, x)
    check_y(orc, y, ref, _rownorm(orc, p, range(rows)),
            f"{rows}x{cols} N={n_keep} g={group} m={m}")


@pytest.mark.parametrize("m", [1, 2, 4, 9, 16, 17, 24, 25, 32, 33, 40, 41, 48, 64])
def test_run_parity_all_m(native, orc, m):
    rows, cols = 200, 1536
    for n_keep, group in ((2, 128), (1, 64)):
        W = _weight(5 + m, rows, cols, "outliers")
        p = orc.pack(W, n_keep, group)
        h = native.SparseGemv(rows, cols, n_keep, group, max_m=64)
        h.import_canonical(p.vals, p.idx, p.scale, p.zero)
        x = synth.activations(77 + m, m, cols)
        check_y(orc, _run(h, x), orc.matvec(p, x), _rownorm(orc, p, range(rows)),
                f"m={m} N={n_keep}")


@pytest.mark.parametrize("n_keep,m", [(2, 33), (1, 41)])
def test_run_parity_more_tiles_than_ctas(native, orc, n_keep, m):
    """The tcgen05 batch kernel's split-K with more 128-row tiles than CTAs: a CTA
    may cover a whole tile (written to y directly) before a shared one, so
    its partial of the shared tile sits in its first workspace slot.  At
    20000 x 1024 five tiles are completed through such a CTA."""
    rows, cols, group = 20000, 1024, 128
    W = synth.weight_outliers(rows + n_keep, rows, cols)
    p = orc.pack(W, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=m)
    h.import_canonical(p.vals, p.idx, p.scale, p.zero)
    x = synth.activations(m + 5, m, cols)
    y = _run(h, x)
    check_y(orc, y, orc.matvec(p, x), np.abs(orc.dequant(p)).sum(axis=1),
            f"{rows}x{cols} {n_keep}:4 m={m}")


@pytest.mark.parametrize("n_keep,m", [(2, 4), (2, 20), (1, 12)])
def test_mma_unsplit_tiles(native, orc, n_keep, m):
    """The mma.sp batch kernel when the row tiles alone fill the GPU: 20000
    rows are 157 tiles of 128, more than one wave of two CTAs per SM can
    split, so every cluster is a single CTA that walks the whole of K and
    reduces with itself (pushed sums at one n-tile, pulled at two or
    three)."""
    rows, cols, group = 20000, 1024, 64
    W = synth.weight_outliers(rows + 7 * m + n_keep, rows, cols)
    p = orc.pack(W, n_keep, group)
    h = native.SparseGemv(rows, cols, n_keep, group, max_m=m)
    h.import_canonical(p.vals, p.idx, p.scale, p.zero)
    x = synth.activations(m + 11, m, cols)
    y = _run(h, x)
    check_y(orc, y, orc.matvec(p, x), np.abs(orc.dequant(p)).sum(axis=1),
            f"{rows}x{cols} {n_keep}:4 m={m}")


def test_run_host_matches_device(native, orc):
    rows, cols, n_keep, group = 130, 1024, 2, 64
    W = _weight(99, rows, cols, "outliers")
    h = _lib_pack(native, W, n_keep, group, max_m=4)
    x = synth.activations(3, 4, cols)
    y_dev = _run(h, x)
    y_host = np.zeros((4, rows), np.float16)
    s = torch.cuda.current_stream()
    h.run_host(x, y_host, s)
    s.synchronize()
    assert np.array_equal(y_host.view(np.uint16), y_dev.view(np.uint16))


def test_empty_and_degenerate(native, orc):
    # rows = 0: nothing to do
    h0 = native.SparseGemv(0, 256, 2, 64)
    h0.pack(np.zeros((0, 256), np.float32))
    x = torch.zeros((1, 256), dtype=torch.float16, device=_dev())
    y = torch.empty((1, 0), dtype=torch.float16, device=_dev())
    h0.run(x, y)
    # cols = 0: y is the empty sum, +0
    hk = native.SparseGemv(5, 0, 1, 64)
    hk.pack(np.zeros((5, 0), np.float32))
    yk = torch.full((1, 5), 7.0, dtype=torch.float16, device=_dev())
    hk.run(torch.zeros((1, 0), dtype=torch.float16, device=_dev()), yk)
    torch.cuda.synchronize()
    assert (yk.cpu().numpy().view(np.uint16) == 0).all()
    # m = 0: no work, y untouched
    h = _lib_pack(native, _weight(1, 8, 64, "normal"), 2, 64)
    y1 = torch.full((1, 8), 3.0, dtype=torch.float16, device=_dev())
    h.run(torch.zeros((0, 64), dtype=torch.float16, device=_dev()), y1)
    torch.cuda.synchronize()
    assert (y1.cpu().numpy() == 3.0).all()
    # all-zero weight gives exact zeros
    hz = _lib_pack(native, np.zeros((16, 256), np.float32), 1, 256)
    yz = _run(hz, synth.activations(1, 1, 256))
    assert (yz.view(np.uint16) == 0).all()


def test_error_paths(native, orc):
    from sparse_weight_only_gb300 import SgemvError
    h = native.SparseGemv(8, 128, 2, 64, max_m=2)
    x = torch.zeros((1, 128), dtype=torch.float16, device=_dev())
    y = torch.zeros((1, 8), dtype=torch.float16, device=_dev())
    with pytest.raises(SgemvError) as e:
        h.run(x, y)
    assert e.value.code == native.SGEMV_ERR_STATE
    W = _weight(2, 8, 128, "normal")
    W[3, 17] = np.nan
    with pytest.raises(SgemvError) as e:
        h.pack(W)
    assert e.value.code == native.SGEMV_ERR_NONFINITE
    W[3, 17] = np.inf
    with pytest.raises(SgemvError) as e:
        h.pack(W)
    assert e.value.code == native.SGEMV_ERR_NONFINITE
    with pytest.raises(SgemvError) as e:
        h.pack(np.full((8, 128), 3e6, np.float32))
    assert e.value.code == native.SGEMV_ERR_RANGE
    h.pack(_weight(3, 8, 128, "normal"))
    x3 = torch.zeros((3, 128), dtype=torch.float16, device=_dev())
    y3 = torch.zeros((3, 8), dtype=torch.float16, device=_dev())
    with pytest.raises(SgemvError) as e:
        h.run(x3, y3)                 # m > max_m
    assert e.value.code == native.SGEMV_ERR_ARG
    buf = torch.zeros(200, dtype=torch.float16, device=_dev())
    lib = native.load()
    rc = lib.sgemv_run(h.handle, buf.data_ptr() + 2, y.data_ptr(), 1,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == native.SGEMV_ERR_ARG      # misaligned x
    rc = lib.sgemv_run(h.handle, buf.data_ptr(), buf.data_ptr() + 16, 1,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == native.SGEMV_ERR_ARG      # x and y overlap
    # canonical 2:4 bytes whose two positions do not ascend are rejected
    p = orc.pack(_weight(4, 8, 128, "normal"), 2, 64)
    bad = p.idx.copy()
    bad[0, 0] = 0b0101                # quad 0 positions (1, 1)
    with pytest.raises(SgemvError) as e:
        h.import_canonical(p.vals, bad, p.scale, p.zero)
    assert e.value.code == native.SGEMV_ERR_ARG
    assert h.status() == 0
