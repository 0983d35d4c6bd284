"""Group size per row (sgemv_create_rowgroups) through the C ABI against the
oracle: bit-exact pack and canonical round trip, products within the
tolerance of tests/_check.py, grouped launches, and the uniform case.

Method: Dong et al., "Efficient LLM ad generation via model compression and
parallel verification" (arXiv 2605.11582), section 3.2 "Adaptive group
quantization": sensitive channels get more (finer) groups inside a layer.
"""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _rg(seed, rows, choices=(64, 128, 256)):
    return np.random.default_rng(seed).choice(choices, rows).astype(np.int32)


def _same(h, p):
    vals, idx, scale, zero = h.export_canonical()
    assert np.array_equal(vals, p.vals), "vals differ"
    assert np.array_equal(idx, p.idx), "idx differ"
    assert np.array_equal(scale, p.scale), "scale differs"
    assert np.array_equal(zero, p.zero), "zero differs"


def _y(h, x):
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    y = torch.empty((x.shape[0], h.rows), dtype=torch.float16, device="cuda")
    h.run(xd, y)
    torch.cuda.synchronize()
    assert h.status() == 0
    return y.cpu().numpy()


CASES = [  # rows, cols, n_keep, group choices
    (40, 512, 2, (64, 128, 256)),
    (64, 768, 1, (64, 128, 256)),
    (33, 4160, 1, (64,)),              # ragged 1:4 tail, one size allowed
    (300, 4096, 2, (64, 256)),
    (130, 1536, 1, (128, 256)),
]


@pytest.mark.parametrize("rows,cols,n_keep,choices", CASES)
def test_rowgroups_pack_and_run_match_oracle(native, orc, rows, cols, n_keep, choices):
    W = synth.weight_outliers(rows + cols, rows, cols)
    rg = _rg(rows, rows, choices)
    p = orc.pack_rowg(W, n_keep, rg)
    h = native.SparseGemv(rows, cols, n_keep, None, max_m=8, row_group=rg)
    assert h.sizes()["groups"] == p.scale.size
    kept = rows * (cols // 4 * n_keep)
    assert h.packed_bytes() == kept // 2 + kept // 4 + 4 * p.scale.size
    h.pack(W)
    _same(h, p)
    norms = np.abs(orc.dequant(p)).sum(axis=1)
    for m in (1, 5):
        x = synth.activations(3 + m, m, cols)
        check_y(orc, _y(h, x), orc.matvec(p, x), norms, f"rowgroups {rows}x{cols} m={m}")


def test_rowgroups_import_export_roundtrip(native, orc):
    rows, cols = 77, 1024
    W = synth.weight_normal(4, rows, cols, 0.02)
    rg = _rg(9, rows)
    for n_keep in (1, 2):
        p = orc.pack_rowg(W, n_keep, rg)
        h = native.SparseGemv(rows, cols, n_keep, None, row_group=rg)
        h.import_canonical(p.vals, p.idx, p.scale, p.zero)
        _same(h, p)
        x = synth.activations(8, 1, cols)
        check_y(orc, _y(h, x), orc.matvec(p, x), np.abs(orc.dequant(p)).sum(axis=1),
                f"imported rowgroups N={n_keep}")


def test_rowgroups_uniform_is_the_matrix_group(native):
    rows, cols = 96, 2048
    W = synth.weight_outliers(6, rows, cols)
    for n_keep, g in ((2, 128), (1, 64)):
        a = native.SparseGemv(rows, cols, n_keep, g, max_m=4)
        b = native.SparseGemv(rows, cols, n_keep, None, max_m=4,
                              row_group=np.full(rows, g, np.int32))
        a.pack(W)
        b.pack(W)
        ea, eb = a.export_canonical(), b.export_canonical()
        for u, v in zip(ea, eb):
            assert np.array_equal(np.ravel(u), np.ravel(v))
        for m in (1, 4):
            x = synth.activations(2 + m, m, cols)
            assert np.array_equal(_y(a, x), _y(b, x))


def test_rowgroups_in_a_grouped_launch(native, orc):
    cols = 4096
    W1 = synth.weight_outliers(31, 500, cols)
    W2 = synth.weight_outliers(32, 300, cols)
    rg = _rg(33, 500)
    p1 = orc.pack_rowg(W1, 2, rg)
    p2 = orc.pack(W2, 2, 128)
    h1 = native.SparseGemv(500, cols, 2, None, row_group=rg)
    h2 = native.SparseGemv(300, cols, 2, 128)
    h1.pack(W1)
    h2.pack(W2)
    x = torch.from_numpy(synth.activations(34, 1, cols)).cuda()
    ys = [torch.empty((1, 500), dtype=torch.float16, device="cuda"),
          torch.empty((1, 300), dtype=torch.float16, device="cuda")]
    native.run_group([h1, h2], x, ys)
    torch.cuda.synchronize()
    for h, p, y in ((h1, p1, ys[0]), (h2, p2, ys[1])):
        single = torch.empty_like(y)
        h.run(x, single)
        torch.cuda.synchronize()
        assert torch.equal(y, single)
        check_y(orc, y.cpu().numpy(), orc.matvec(p, x.cpu().numpy()),
                np.abs(orc.dequant(p)).sum(axis=1), "grouped rowgroups")


def test_rowgroups_full_size_sampled(native, orc):
    """An 11008 x 4096 2:4 layer with a group size per row, rows sampled."""
    rows, cols = 11008, 4096
    W = synth.weight_normal(41, rows, cols, 0.02)
    rg = _rg(42, rows)
    p = orc.pack_rowg(W, 2, rg)
    h = native.SparseGemv(rows, cols, 2, None, row_group=rg)
    h.pack(W)
    _same(h, p)
    x = synth.activations(43, 1, cols)
    y = _y(h, x)
    sel = np.arange(0, rows, 97, dtype=np.int64)
    norms = np.array([np.abs(orc.dequant(p, int(r), 1)).sum() for r in sel])
    check_y(orc, y[:, sel], orc.matvec(p, x, sel), norms, "rowgroups 11008x4096")


def test_rowgroups_rejects_bad_sizes(native):
    from sparse_weight_only_gb300 import SgemvError
    for rg, cols in (([64, 96], 512), ([64, 256], 320), ([512, 64], 1024)):
        with pytest.raises(SgemvError) as e:
            native.SparseGemv(2, cols, 2, None, row_group=np.array(rg, np.int32))
        assert e.value.code == native.SGEMV_ERR_ARG
