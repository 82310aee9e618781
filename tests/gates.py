"""Acceptance gates comparing the CUDA path with the oracle.

G1  top-16 on the same FP32 logits: ids bit-exact (order included), routing
    weights within 5 FP32 ULP ("Kimi K3.1 recipe ...", commit message:
    "weights within 5 fp32 ULP").
G2  latent: relative RMS against float64 <= 2e-3 over the tensor, and per
    element within 1 BF16 ulp of the oracle's rounded value, or within
    ulp_bf16(y64) + 2^-20 * sum_k |h w| of the float64 value (the FP32
    accumulation allowance for values near zero).
G3  logits: |out - y64| <= 2^-20 * sum_k |h w| per element.
G4  end-to-end ids (GPU logits -> GPU top-16) against the oracle's ids: equal
    sets, or one id out and one in whose oracle logits lie within 2 FP32 ULP
    of each other (same page: "a 1-for-1 swap within 2 fp32 ULP"); within
    equal sets, two ids may trade places only if their float64 logits are
    closer than the sum of their G3 allowances.

Set ROUTE_PARITY_STATS=<file> to append each check's statistics (relative
RMS, ULP distances, swap counts) to a JSON-lines file.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

SLACK = 2.0 ** -20
REL_RMS_BAR = 2e-3


def record(case: str, **stats) -> None:
    path = os.environ.get("ROUTE_PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **stats}) + "\n")


def bf16_vals(bits) -> np.ndarray:
    return oracle.bf16_to_f64(np.asarray(bits).view(np.uint16))


def ulp_bf16(x) -> np.ndarray:
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(x)
    return np.where(x == 0, 2.0 ** -133, np.ldexp(1.0, e - 8))


def ulp_f32(x) -> np.ndarray:
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(x)
    return np.where(x == 0, 2.0 ** -149, np.ldexp(1.0, np.maximum(e - 24, -149)))


def abs_dot(h_bits, W_bits) -> np.ndarray:
    """sum_k |h[r,k]| |W[k,n]| in float64 (sign bits cleared)."""
    return oracle.dot64(np.asarray(h_bits, np.uint16) & 0x7FFF,
                        np.asarray(W_bits, np.uint16) & 0x7FFF)


def check_latent(out_bits, ref_bits, y64, absdot, rms_bar: bool = True) -> dict:
    out = bf16_vals(out_bits)
    ref = bf16_vals(ref_bits)
    assert np.isfinite(out).all(), "non-finite latent"
    rel = math.sqrt(float(((out - y64) ** 2).sum() / (y64 ** 2).sum()))
    strict = np.abs(out - ref) <= ulp_bf16(ref)
    slack = np.abs(out - y64) <= ulp_bf16(y64) + SLACK * absdot
    bad = ~(strict | slack)
    assert not bad.any(), (
        f"{int(bad.sum())} latent elements outside the gate; first at "
        f"{np.argwhere(bad)[0].tolist()}")
    if rms_bar:
        assert rel <= REL_RMS_BAR, f"latent relative RMS {rel:.3e} > {REL_RMS_BAR}"
    exact = np.asarray(out_bits).view(np.uint16) == np.asarray(ref_bits).view(np.uint16)
    return {"rel_rms": rel, "slack_only": int((~strict).sum()),
            "cr_miss_rate": float(1.0 - exact.mean())}


def check_logits(out, y64, absdot) -> dict:
    out = np.asarray(out, np.float64)
    err = np.abs(out - y64)
    bad = err > SLACK * absdot
    assert not bad.any(), f"{int(bad.sum())} logits outside 2^-20 sum|hw|"
    ulps = err / ulp_f32(y64)
    return {"max_ulp": float(ulps.max()), "median_ulp": float(np.median(ulps))}


def check_topk_exact(ids, w, ids_ref, w_ref, ulp_bound: int = 5) -> dict:
    assert np.array_equal(ids, ids_ref), (
        f"ids differ in {int((ids != ids_ref).any(axis=1).sum())} rows")
    both_nan = np.isnan(w) & np.isnan(w_ref)
    diff = np.abs(w.astype(np.float64) - w_ref.astype(np.float64))
    ulps = np.where(both_nan, 0.0, diff / ulp_f32(w_ref))
    assert np.all(np.isfinite(ulps)) and ulps.max() <= ulp_bound, f"weights {ulps.max()} ULP off"
    return {"max_weight_ulp": float(ulps.max())}


def check_ids_end_to_end(ids, ids_ref, logits_ref, y_log=None, abs_log=None) -> dict:
    """G4.  A set difference must be one id out, one in, within 2 FP32 ULP of
    each other.  Within equal sets, two ids may trade places only if their
    float64 logits are closer than the sum of the two logits' G3 error
    allowances (when y_log / abs_log are given), else within 2 ULP."""
    swaps = 0
    for r in range(ids.shape[0]):
        got, want = list(ids[r]), list(ids_ref[r])
        lg = logits_ref[r].astype(np.float64)
        gs, ws = set(got), set(want)
        if gs != ws:
            out_ = ws - gs
            in_ = gs - ws
            assert len(out_) == 1 and len(in_) == 1, f"row {r}: {len(out_)} ids differ"
            o, g = out_.pop(), in_.pop()
            win = 2 * ulp_f32(max(abs(lg[o]), abs(lg[g])))
            assert abs(lg[g] - lg[o]) <= win, (
                f"row {r}: swap {o}->{g} outside 2 ULP ({lg[o]!r} vs {lg[g]!r})")
            swaps += 1
            continue
        for a, b in zip(got, want):
            if a != b:
                if y_log is not None:
                    win = SLACK * (abs_log[r][a] + abs_log[r][b])
                    d = abs(y_log[r][a] - y_log[r][b])
                else:
                    win = 2 * ulp_f32(max(abs(lg[a]), abs(lg[b])))
                    d = abs(lg[a] - lg[b])
                assert d <= win, f"row {r}: ids {a},{b} trade places {d!r} apart (window {win!r})"
    return {"swap_rows": swaps, "rows": int(ids.shape[0])}
