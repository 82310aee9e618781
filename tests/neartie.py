"""Near-tie rows for the 9..20-row decode sweep (test input construction).

A quarter of the rows (r mod 4 == 3) are edited so that the experts at ranks
16 and 17 have float64 logits within 1 FP32 ULP (alternate rows: within 2 ULP)
of each other.  This exercises the near-tie rule of "Kimi K3.1 recipe: route
9..20 decode rows through the pushed pair gather and standalone top-16",
commit message: a difference in the selected set may only be a one-for-one
exchange of two experts whose logits lie at most 2 FP32 ULP apart.

The pages give no construction; this one edits only hidden coordinates of the
row (weights are shared by every row):
  1. a coarse coordinate k1 with a large |W[k1, a] - W[k1, b]| cancels most of
     the gap between experts a (rank 16) and b (rank 17);
  2. two coordinates whose hidden values are the row's smallest are set to
     small BF16 values that move the remaining gap onto the target, each
     step working at a finer scale than the one before.
Gaps are measured with the oracle's float64 sums.  A row is accepted only if
a and b are still at ranks 16 and 17 afterwards.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from gates import ulp_f32


def _bf16(x: float) -> int:
    t = torch.tensor([x], dtype=torch.float32).to(torch.bfloat16)
    return int(t.view(torch.int16).numpy().view(np.uint16)[0])


def _exact(h_row_bits, wr_bits):
    return oracle.dot64(h_row_bits[None, :], wr_bits)[0]


def _rank(y):
    # rank order by value desc, id asc (float64 values are distinct here)
    return np.lexsort((np.arange(y.size), -y))


def inject_row(h_row_bits: np.ndarray, wr_bits: np.ndarray, target_ulps: float):
    """Return (edited row bits, a, b, gap in FP32 ULP) or None."""
    Wv = oracle.bf16_to_f64(wr_bits)
    y = _exact(h_row_bits, wr_bits)
    order = _rank(y)
    a, b = int(order[15]), int(order[16])
    D = Wv[:, a] - Wv[:, b]
    hv = oracle.bf16_to_f64(h_row_bits)
    small = np.argsort(np.abs(hv))  # smallest hidden values first
    for k1 in np.argsort(-np.abs(D))[:12]:
        h = h_row_bits.copy()
        gap = y[a] - y[b]
        h[k1] = _bf16(hv[k1] - gap / D[k1])
        fine = [k for k in small[:200] if k != k1 and abs(D[k]) > 0.25 * np.abs(D).max()][:4]
        target = None
        for k in fine[:3]:
            yy = _exact(h, wr_bits)
            ulp = float(ulp_f32(yy[a]))
            target = target_ulps * ulp
            need = target - (yy[a] - yy[b])
            cur = float(oracle.bf16_to_f64(np.array([h[k]], np.uint16))[0])
            h[k] = _bf16(cur + need / D[k])
        yy = _exact(h, wr_bits)
        new_order = _rank(yy)
        gap_ulps = (yy[a] - yy[b]) / float(ulp_f32(yy[a]))
        lo, hi = (0.0, 1.0) if target_ulps <= 1.0 else (1.0, 2.0)
        if int(new_order[15]) == a and int(new_order[16]) == b and lo < gap_ulps <= hi:
            return h, a, b, gap_ulps
    return None


def inject(hidden_bits: np.ndarray, wr_bits: np.ndarray, rows=None):
    """Edit rows r with r mod 4 == 3 (or the given rows); returns the edited
    hidden array and a list of (row, a, b, gap_ulps)."""
    h = hidden_bits.copy()
    if rows is None:
        rows = [r for r in range(h.shape[0]) if r % 4 == 3]
    done = []
    for i, r in enumerate(rows):
        res = inject_row(h[r], wr_bits, 0.5 if i % 2 == 0 else 1.5)
        if res is not None:
            h[r] = res[0]
            done.append((r, res[1], res[2], res[3]))
    return h, done
