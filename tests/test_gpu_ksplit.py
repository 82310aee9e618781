"""The general (K-split) path's latent arithmetic as a decode plan option
(route_set_latent_ksplit) against the oracle's K-split definition: eight
896-deep K-slice partials rounded to BF16, summed in FP32, rounded again."""

import numpy as np
import pytest

import latent_projection_top_gb300 as route
import oracle
from gates import bf16_vals, ulp_bf16
from gpu_util import bank, require_gpu, run_step, to_dev_bf16

pytestmark = pytest.mark.gpu

SLICES = 8


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rel_rms(out_bits, y64):
    d = bf16_vals(out_bits) - y64
    return float(np.sqrt((d * d).sum() / (y64 * y64).sum()))


@pytest.mark.parametrize("workload,rows", [("decode_r8", 8), ("prefill_r1024", 20)])
def test_ksplit_latent_matches_the_general_path(workload, rows):
    # prefill_r1024's first rows meet its cancel group: large slice partials
    # of alternating sign
    hid, wl, wr = bank(workload, 0)
    h_bits = np.ascontiguousarray(hid[:rows])
    h, dwl, dwr = to_dev_bf16(h_bits), to_dev_bf16(wl), to_dev_bf16(wr)
    with route.Plan(route.DECODE, rows) as plan:
        full = run_step(plan, h, dwl, dwr)
        route.route_set_latent_ksplit(plan, True)
        got = run_step(plan, h, dwl, dwr)
        again = run_step(plan, h, dwl, dwr)
        route.route_set_latent_ksplit(plan, False)
        back = run_step(plan, h, dwl, dwr)
    for name, a, b in zip(("logits", "ids", "weights"), got[1:], full[1:]):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), name
    assert np.array_equal(got[0], again[0]) and np.array_equal(back[0], full[0])

    ref = oracle.latent_ksplit(h_bits, wl, SLICES)
    K = h_bits.shape[1]
    sl = K // SLICES
    parts = np.stack([oracle.dot64(h_bits[:, s * sl:(s + 1) * sl], wl[s * sl:(s + 1) * sl])
                      for s in range(SLICES)])
    g, r = bf16_vals(got[0]), bf16_vals(ref)
    miss = g != r
    # A slice partial within a hair of a BF16 rounding boundary may round the
    # other way (its FP32 value comes from 64-deep tensor-core blocks); that
    # moves the FP32 sum by one BF16 ulp of that partial, and the last rounding
    # by at most one ulp of the result.
    bound = ulp_bf16(np.abs(parts)).max(axis=0) + ulp_bf16(np.abs(r))
    assert miss.mean() <= 2e-3, miss.mean()
    assert np.all(np.abs(g - r)[miss] <= bound[miss])
    # the two roundings cost accuracy against float64, as the pages report
    y64 = oracle.dot64(h_bits, wl)
    assert _rel_rms(got[0], y64) > _rel_rms(full[0], y64)


def _check_ksplit(got_bits, h_bits, wl):
    ref = oracle.latent_ksplit(h_bits, wl, SLICES)
    sl = h_bits.shape[1] // SLICES
    parts = np.stack([oracle.dot64(h_bits[:, s * sl:(s + 1) * sl], wl[s * sl:(s + 1) * sl])
                      for s in range(SLICES)])
    g, r = bf16_vals(got_bits), bf16_vals(ref)
    miss = g != r
    bound = ulp_bf16(np.abs(parts)).max(axis=0) + ulp_bf16(np.abs(r))
    assert miss.mean() <= 2e-3, miss.mean()
    assert np.all(np.abs(g - r)[miss] <= bound[miss])


@pytest.mark.parametrize("rows,sample", [(40, None), (1024, (0, 1, 2, 3, 17, 255, 256, 500, 777, 1023))])
def test_prefill_ksplit_latent_matches_the_general_path(rows, sample):
    hid, wl, wr = bank("prefill_r1024", 0)
    h_bits = np.ascontiguousarray(hid[:rows])
    h, dwl, dwr = to_dev_bf16(h_bits), to_dev_bf16(wl), to_dev_bf16(wr)
    with route.Plan(route.PREFILL, rows) as plan:
        full = run_step(plan, h, dwl, dwr)
        route.route_set_latent_ksplit(plan, True)
        got = run_step(plan, h, dwl, dwr)
        again = run_step(plan, h, dwl, dwr)
    for name, a, b in zip(("logits", "ids", "weights"), got[1:], full[1:]):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), name
    assert np.array_equal(got[0], again[0])
    idx = list(range(rows)) if sample is None else list(sample)
    _check_ksplit(got[0][idx], np.ascontiguousarray(h_bits[idx]), wl)
