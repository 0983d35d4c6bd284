"""Tolerance check of a GPU y against the oracle.

The stated y tolerance: max |dy| <= 1e-2 * ||row||_1 * 2^-10 and rel-L2 <= 1e-3.
Reading (the bound is silent on which norm and which reference): ||row||_1
is the L1 norm of the dequantised pruned row, and the binary16 y is
compared with binary16(y_ref), allowing the larger of that bound and one
binary16 ulp of binary16(y_ref) -- a binary16 output cannot be closer to an
fp64 value than half an ulp, so only rounding-boundary flips pass.  The
rel-L2 bound is checked against the fp64 y_ref itself.
"""
import numpy as np


def f16_ulp(bits: np.ndarray) -> np.ndarray:
    """Spacing of binary16 at each finite value (bit patterns)."""
    e = (bits.astype(np.int64) >> 10) & 0x1F
    return np.exp2(np.maximum(e, 1) - 25.0)


def check_y(orc, y_gpu, y_ref, rownorm1, label=""):
    """y_gpu: binary16 array (m x n); y_ref: fp64 (m x n); rownorm1: (n,)."""
    y_gpu = np.asarray(y_gpu)
    if y_gpu.dtype != np.float16:
        y_gpu = y_gpu.astype(np.float16)
    ref16_bits = orc.f64_to_f16_array(y_ref).astype(np.uint16)
    ref16 = ref16_bits.view(np.float16).astype(np.float64)
    got = y_gpu.astype(np.float64)
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    bound = np.maximum(1e-2 * np.asarray(rownorm1)[None, :] * 2.0 ** -10,
                       f16_ulp(ref16_bits))
    err = np.abs(got - ref16)
    bad = err > bound
    assert not bad.any(), (
        f"{label}: {int(bad.sum())} outputs out of tolerance; worst "
        f"{float((err - bound).max()):.3g} over the bound at "
        f"{np.unravel_index(np.argmax(err - bound), err.shape)}")
    nref = np.linalg.norm(y_ref)
    if nref > 0:
        rel = np.linalg.norm(got - y_ref) / nref
        assert rel <= 1e-3, f"{label}: rel-L2 {rel:.3g} > 1e-3"
    else:
        assert not got.any()
    return {"max_abs_vs_f64": float(np.abs(got - y_ref).max()) if got.size else 0.0,
            "flips": int((err > 0).sum())}
