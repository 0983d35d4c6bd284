"""Grouped run (several matrices sharing x) through the C ABI.  Every output
matches the oracle; at m = 1 it also equals the per-matrix run bit for bit
(each row is computed the same way in either launch).  At m >= 2 the
matrices of one N (and, from m = 33, one group size) share a launch of a
batch kernel, whose split of K across CTAs depends on the launch's tile
count, so there the summation order -- not the tolerance -- may differ from
a single run."""
import numpy as np
import pytest

import synth
from _check import check_y

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _mats(native, orc, specs, cols, max_m=1):
    out = []
    for i, (rows, n_keep, group) in enumerate(specs):
        W = synth.weight_outliers(300 + i, rows, cols)
        p = orc.pack(W, n_keep, group)
        h = native.SparseGemv(rows, cols, n_keep, group, max_m=max_m)
        h.import_canonical(p.vals, p.idx, p.scale, p.zero)
        out.append((h, p))
    return out


def _ys(mats, m):
    return [torch.full((m, h.rows), 9.0, dtype=torch.float16, device="cuda")
            for h, _ in mats]


SPECS_MIXED = [(300, 1, 256), (129, 2, 128), (64, 1, 128), (1, 2, 64),
               (257, 1, 64), (33, 2, 64), (200, 2, 256), (96, 1, 128),
               (70, 2, 128), (5, 1, 64)]      # 5 of each N: one launch, two CTA ranges
SPECS_MANY = [(40 + 7 * i, 1, (64, 128, 256)[i % 3]) for i in range(9)] + \
             [(90, 2, 128), (17, 2, 64)]      # 9 > 8 of one N: a launch per N and per 8


@pytest.mark.parametrize("m,cols,specs", [(1, 1536, SPECS_MIXED), (5, 1536, SPECS_MIXED),
                                          (1, 8192, SPECS_MIXED), (1, 1024, SPECS_MANY),
                                          (1, 6144, SPECS_MIXED),
                                          (2, 1536, SPECS_MIXED), (16, 1536, SPECS_MIXED),
                                          (9, 1024, SPECS_MANY), (24, 1536, SPECS_MIXED),
                                          (64, 1536, SPECS_MIXED), (40, 1024, SPECS_MANY)])
def test_group_matches_single_and_oracle(native, orc, m, cols, specs):
    mats = _mats(native, orc, specs, cols, max_m=64)
    x = torch.from_numpy(synth.activations(41 + m, m, cols)).cuda()
    ys = _ys(mats, m)
    native.run_group([h for h, _ in mats], x, ys)
    torch.cuda.synchronize()
    for (h, p), y in zip(mats, ys):
        single = torch.empty_like(y)
        h.run(x, single)
        torch.cuda.synchronize()
        if m == 1:
            assert torch.equal(y, single)
        ref = orc.matvec(p, x.cpu().numpy())
        norms = np.abs(orc.dequant(p)).sum(axis=1)
        check_y(orc, y.cpu().numpy(), ref, norms, f"group member {h.rows}x{cols} m={m}")
        check_y(orc, single.cpu().numpy(), ref, norms, f"single {h.rows}x{cols} m={m}")
        assert h.status() == 0


@pytest.mark.parametrize("config,m", [("config3", 1), ("config4", 4), ("config4", 16),
                                      ("config3", 8), ("config4", 33), ("config4", 64),
                                      ("config3", 24)])
def test_group_qkv_shapes(native, orc, config, m):
    """The decoder layer's q/k/v (mixed N, g in the layer set; all 2:4 g128 in
    the verification-batch set) and gate/up groups at full size."""
    gvs = getattr(synth, config)()
    for names in (("q", "k", "v"), ("gate", "up")):
        sel = [g for g in gvs if g.name in names]
        mats = []
        for gv in sel:
            W = gv.weight()
            p = orc.pack(W, gv.n_keep, gv.group)
            h = native.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, max_m=m)
            h.pack(W)
            mats.append((h, p))
        x = torch.from_numpy(sel[0].x(m)).cuda()
        ys = _ys(mats, m)
        native.run_group([h for h, _ in mats], x, ys)
        torch.cuda.synchronize()
        for (h, p), y in zip(mats, ys):
            single = torch.empty_like(y)
            h.run(x, single)
            torch.cuda.synchronize()
            if m == 1:
                assert torch.equal(y, single)
            assert h.status() == 0
            rows = np.arange(0, h.rows, 37, dtype=np.int64)
            ref = orc.matvec(p, x.cpu().numpy(), rows)
            norms = np.array([np.abs(orc.dequant(p, int(r), 1)).sum() for r in rows])
            check_y(orc, y.cpu().numpy()[:, rows], ref, norms, f"{names} {h.rows}")


def test_group_edges(native, orc):
    from sparse_weight_only_gb300 import SgemvError
    cols = 512
    mats = _mats(native, orc, [(0, 2, 64), (40, 1, 128), (0, 1, 64)], cols)
    x = torch.from_numpy(synth.activations(7, 1, cols)).cuda()
    ys = _ys(mats, 1)
    native.run_group([h for h, _ in mats], x, ys)       # empty members skipped
    torch.cuda.synchronize()
    single = torch.empty_like(ys[1])
    mats[1][0].run(x, single)
    torch.cuda.synchronize()
    assert torch.equal(ys[1], single)
    native.run_group([], x, [])                          # count 0: no-op
    other = _mats(native, orc, [(8, 2, 64)], 256)
    with pytest.raises(SgemvError) as e:                 # cols differ
        native.run_group([mats[1][0], other[0][0]], x,
                         [ys[1], torch.empty((1, 8), dtype=torch.float16, device="cuda")])
    assert e.value.code == native.SGEMV_ERR_ARG
    with pytest.raises(SgemvError) as e:                 # m > max_m
        native.run_group([mats[1][0]], torch.zeros((2, cols), dtype=torch.float16,
                                                    device="cuda"),
                         [torch.empty((2, 40), dtype=torch.float16, device="cuda")])
    assert e.value.code == native.SGEMV_ERR_ARG


def test_group_outputs_complete_for_next_work(native, orc):
    """Work queued right after a grouped call on the same stream (no host
    synchronisation in between) sees every output of both launches (one per
    N) complete."""
    cols = 4096
    specs = [(4096, 1, 256), (4096, 2, 128), (4096, 1, 128)]   # q, k, v shapes
    mats = _mats(native, orc, specs, cols)
    x = torch.from_numpy(synth.activations(5, 1, cols)).cuda()
    singles = []
    for h, _ in mats:
        y = torch.empty((1, h.rows), dtype=torch.float16, device="cuda")
        h.run(x, y)
        singles.append(y)
    torch.cuda.synchronize()
    want = torch.cat(singles, dim=1)
    stream = torch.cuda.current_stream()
    for rep in range(20):
        ys = _ys(mats, 1)
        native.run_group([h for h, _ in mats], x, ys, stream.cuda_stream)
        got = torch.cat(ys, dim=1)          # queued on the same stream
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"repetition {rep}"


def test_group_rejects_overlapping_outputs(native, orc):
    cols = 256
    mats = _mats(native, orc, [(64, 2, 64), (64, 1, 64)], cols)
    x = torch.from_numpy(synth.activations(6, 1, cols)).cuda()
    buf = torch.empty((1, 96), dtype=torch.float16, device="cuda")
    with pytest.raises(native.SgemvError):
        native.run_group([h for h, _ in mats], x, [buf[:, :64], buf[:, 32:96]])


@pytest.mark.parametrize("m", [1, 4, 33])
def test_group_host_matches_device(native, orc, m):
    """sgemv_run_group_host: x in, outputs out through host buffers, the same
    products as sgemv_run_group on device buffers, bit for bit."""
    cols = 1536
    mats = _mats(native, orc, SPECS_MIXED[:6], cols, max_m=64)
    hs = [h for h, _ in mats]
    x = synth.activations(55 + m, m, cols)
    ys = _ys(mats, m)
    native.run_group(hs, torch.from_numpy(x).cuda(), ys)
    torch.cuda.synchronize()
    xh = torch.from_numpy(x).pin_memory()
    yh = [torch.zeros((m, h.rows), dtype=torch.float16).pin_memory() for h in hs]
    stream = torch.cuda.current_stream()
    native.run_group_host(hs, xh, yh, stream)
    stream.synchronize()
    for (h, p), y, yy in zip(mats, ys, yh):
        assert torch.equal(y.cpu(), yy), f"{h.rows} rows"
        assert h.status() == 0
    with pytest.raises(native.SgemvError) as e:          # a handle twice
        native.run_group_host([hs[0], hs[0]], xh, [yh[0], yh[0]])
    assert e.value.code == native.SGEMV_ERR_ARG
