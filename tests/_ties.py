"""Quantiser tie cases with hand-derived codes (rounding: nearest, ties to even).

The paper quantises each group's kept weights from FP16 to INT4 (section 1,
"Our core idea"; section 3.2, "Adaptive group quantization") but does not say
how halfway cases round.  The reading taken is IEEE round-to-nearest, ties to
even, for both the zero point z = rint(-lo / s) and the codes
q = rint(w / s) + z.  Every group below has s = 0.25 exactly, so w / s and
-lo / s are exact and land on halves: a quantiser that rounded halves away
from zero (roundf) would produce different z and q, and fail these cases.

Group layout: one row, 2:4 keeps positions 0 and 1 of every quad (positions 2
and 3 hold 0), 1:4 keeps position 0 (positions 1..3 hold 0).  The kept values
of a group are KEPT (padded with zeros); lo = -1.125 and hi = 2.625 give
(hi - lo) / 15 = 0.25 exactly.
"""
import numpy as np

# kept value, w / s, rint(w / s) (ties to even)
KEPT = [
    (2.625, 10.5, 10),    # hi; even k: 10.5 -> 10
    (-1.125, -4.5, -4),   # lo; even k: -4.5 -> -4
    (0.125, 0.5, 0),      # 0.5 -> 0
    (0.375, 1.5, 2),      # odd k: 1.5 -> 2
    (0.625, 2.5, 2),      # 2.5 -> 2
    (-0.125, -0.5, 0),    # -0.5 -> -0
    (-0.375, -1.5, -2),
    (-0.625, -2.5, -2),
    (1.125, 4.5, 4),
    (-0.875, -3.5, -4),
    (0.875, 3.5, 4),
    (1.875, 7.5, 8),
]
SCALE_BITS = 0x3400        # binary16 0.25
Z = 4                      # rint(1.125 / 0.25) = rint(4.5) = 4
ZERO_BITS = 0x4400         # binary16 4.0
CODE_OF_ZERO = Z           # a kept 0.0 quantises to q = z


def codes(values):
    """q = rint(w / s) + z for the listed values (hand table above)."""
    table = {w: k for w, _, k in KEPT}
    return [table[w] + Z if w != 0.0 else CODE_OF_ZERO for w in values]


def weight(n_keep: int, group: int, groups: int = 2) -> tuple[np.ndarray, list]:
    """One row of `groups` groups, each holding every KEPT value once (zeros
    after them); returns (W, kept values in kept order)."""
    kept_per_group = group // 4 * n_keep
    vals = [w for w, _, _ in KEPT]
    assert len(vals) <= kept_per_group
    kept = []
    for G in range(groups):
        # rotate so each group starts with a different value
        v = vals[G % len(vals):] + vals[:G % len(vals)]
        kept += v + [0.0] * (kept_per_group - len(v))
    W = np.zeros((1, group * groups), np.float32)
    for j, w in enumerate(kept):
        t = j // n_keep
        W[0, 4 * t + j % n_keep] = w
    return W, kept


def expected_bytes(n_keep: int, group: int, groups: int = 2):
    """Canonical vals and idx bytes, scale and zero bits, built by hand from
    the code table: nibble j at byte j / 2 (low first), position of kept j at
    bits 2 (j % 4) of byte j / 4."""
    _, kept = weight(n_keep, group, groups)
    q = codes(kept)
    vals = np.zeros((1, (len(q) + 1) // 2), np.uint8)
    idx = np.zeros((1, (len(q) + 3) // 4), np.uint8)
    for j, c in enumerate(q):
        vals[0, j // 2] |= c << (4 * (j % 2))
        idx[0, j // 4] |= (j % n_keep) << (2 * (j % 4))
    scale = np.full((1, groups), SCALE_BITS, np.uint16)
    zero = np.full((1, groups), ZERO_BITS, np.uint16)
    return vals, idx, scale, zero
